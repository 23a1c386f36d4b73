"""Element-wise check of the device activations and derivatives through the C ABI.

One sequence of N queries and a single key, head dim 64: q_i = (z_i, 0, ...),
k = v = dO_i = (1, 0, ...), scale 1. Then the forward output is
out[i, 0] = bf16(act(z_i)) and the backward gives dq[i, 0] = bf16(act'(z_i)),
so every device evaluation (polynomial erf, Newton reciprocal, MUFU tanh) is
compared point by point with the float64 oracle's act / act' on a dense grid
of bf16-representable z. Allowed error: one bf16 ulp of the reference (the
kernel rounds P and dS to bf16 once more than the oracle) plus the stated
approximation bound of the device formula.
"""

import pytest
import torch

import oracle
from generalized_attention_recsys_gb300 import _lib
from gpu_util import ensure_built

pytestmark = pytest.mark.gpu

ELEMENTWISE = ["identity", "gelu", "gelu_tanh", "fast_gelu", "relu", "relu2", "leaky_relu", "silu", "hardswish",
               "fast_gelu_bf16", "fast_silu"]
# approximation bound of the device forward evaluation, as a multiple of max(1, |z|).
# fast_gelu_bf16 rounds s^2, the cubic, u, z/2, tanh(u) and the result to bf16:
# emulating that (tanh exact, then rounded) gives at most 1.8e-3 beyond the one
# bf16 ulp allowed below; 6e-3 leaves room for the hardware bf16 tanh.
FWD_BOUND = {"gelu": 2e-5, "fast_gelu": 6e-4, "gelu_tanh": 2e-5, "silu": 2e-5, "fast_gelu_bf16": 6e-3,
             "fast_silu": 6e-4}


def _grid(lo, hi, n):
    z = torch.linspace(lo, hi, n).to(torch.bfloat16)
    return torch.unique(torch.cat([z, torch.tensor([0.0, -3.0, 3.0, 1.0, -1.0], dtype=torch.bfloat16)]))


@pytest.mark.parametrize("act", ELEMENTWISE)
def test_device_activation_and_derivative_pointwise(act):
    ensure_built()
    z = _grid(-9.0, 9.0, 6000)
    n, d = z.numel(), 64
    q = torch.zeros(n, 1, d, dtype=torch.bfloat16)
    q[:, 0, 0] = z
    k = torch.zeros(1, 1, d, dtype=torch.bfloat16)
    k[0, 0, 0] = 1
    v = k.clone()
    do = torch.zeros(n, 1, d, dtype=torch.bfloat16)
    do[:, 0, 0] = 1
    cu_q = torch.tensor([0, n], dtype=torch.int32).cuda()
    cu_k = torch.tensor([0, 1], dtype=torch.int32).cuda()
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, _ = _lib.gdpa_fwd(qd, kd, vd, cu_q, cu_k, n, 1, act, 1.0, batch=1)
    dq, dk, dv = _lib.gdpa_bwd(qd, kd, vd, cu_q, cu_k, n, 1, act, 1.0, False, -1, None, None, dod, batch=1)
    assert _lib.gdpa_get_status() == 0
    zz = z.double()
    ref_f = oracle.act_fwd(act, zz)
    ref_g = oracle.act_grad(act, zz)
    got_f = out[:, 0, 0].double().cpu()
    got_g = dq[:, 0, 0].double().cpu()
    scale_z = torch.clamp(zz.abs(), min=1.0)
    bound_f = 2.0 ** -8 * ref_f.abs() + FWD_BOUND.get(act, 0.0) * scale_z + 1e-30
    bound_g = 2.0 ** -8 * ref_g.abs() + 2e-5 * scale_z + 1e-30
    bad_f = (got_f - ref_f).abs() > bound_f
    bad_g = (got_g - ref_g).abs() > bound_g
    assert not bad_f.any(), f"{act}: act mismatch at z={zz[bad_f][:5].tolist()} got {got_f[bad_f][:5].tolist()} " \
                            f"ref {ref_f[bad_f][:5].tolist()}"
    assert not bad_g.any(), f"{act}: act' mismatch at z={zz[bad_g][:5].tolist()} got {got_g[bad_g][:5].tolist()} " \
                            f"ref {ref_g[bad_g][:5].tolist()}"
