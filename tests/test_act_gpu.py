"""Element-wise check of the device activations and derivatives through the C ABI.

Forward: one sequence of N queries and 128 keys, head dim 128, scale 1, with
q_i = (z_i, 0, ...), every key k_j = (1, 0, ...) and v_j = e_j (the identity).
Then every score of query row i is z_i, and out[i, j] = bf16(P) as the kernel
evaluated it at tile column j, so every column position of the activation
warps (and every evaluation path a column can take) is compared point by
point with the float64 oracle on a dense grid of bf16-representable z.
Backward: one key, k = v = dO_i = (1, 0, ...), so dq[i, 0] = bf16(act'(z_i)).
Allowed error: the rounding of P or dS to bf16 (one bf16 ulp of the
reference; 2/3 of an ulp beyond the value for GELU, whose P is packed by
truncation of a biased value) plus the stated approximation bound of the
device formula.
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
# gelu mixes a fitted tanh form of Phi with MUFU tanh (|Phi error| <= 3.9e-4)
# and a degree-5 erf polynomial (<= 1.7e-4).
FWD_BOUND = {"gelu": 4e-4, "fast_gelu": 6e-4, "gelu_tanh": 2e-5, "silu": 2e-5, "fast_gelu_bf16": 6e-3,
             "fast_silu": 6e-4}
# relative rounding allowance of the forward value: one bf16 ulp (2^-8 of the
# value at worst) where P is rounded to nearest; gelu packs bf16 P by
# truncating the value times (1 + 1/384), within 2/3 of an ulp (2^-7 * 2/3).
FWD_REL = {"gelu": 2.0 ** -7 * (2.0 / 3.0) * 1.0001}


def _grid(lo, hi, n):
    z = torch.linspace(lo, hi, n).to(torch.bfloat16)
    return torch.unique(torch.cat([z, torch.tensor([0.0, -3.0, 3.0, 1.0, -1.0], dtype=torch.bfloat16)]))


@pytest.mark.parametrize("act", ELEMENTWISE)
def test_device_activation_and_derivative_pointwise(act):
    ensure_built()
    z = _grid(-9.0, 9.0, 6000)
    n, d, nk = z.numel(), 128, 128
    # forward: all 128 tile columns see the same score z_i
    q = torch.zeros(n, 1, d, dtype=torch.bfloat16)
    q[:, 0, 0] = z
    kf = torch.zeros(nk, 1, d, dtype=torch.bfloat16)
    kf[:, 0, 0] = 1
    vf = torch.eye(nk, d, dtype=torch.bfloat16).reshape(nk, 1, d)
    qd = q.cuda()
    cu_q = torch.tensor([0, n], dtype=torch.int32).cuda()
    cu_kf = torch.tensor([0, nk], dtype=torch.int32).cuda()
    out, _ = _lib.gdpa_fwd(qd, kf.cuda(), vf.cuda(), cu_q, cu_kf, n, nk, act, 1.0, batch=1)
    # backward: one key
    k = torch.zeros(1, 1, d, dtype=torch.bfloat16)
    k[0, 0, 0] = 1
    v = k.clone()
    do = torch.zeros(n, 1, d, dtype=torch.bfloat16)
    do[:, 0, 0] = 1
    cu_k = torch.tensor([0, 1], dtype=torch.int32).cuda()
    dq, dk, dv = _lib.gdpa_bwd(qd, k.cuda(), v.cuda(), cu_q, cu_k, n, 1, act, 1.0, False, -1, None, None, do.cuda(),
                               batch=1)
    assert _lib.gdpa_get_status() == 0
    zz = z.double()
    ref_f = oracle.act_fwd(act, zz)[:, None].expand(n, nk)
    ref_g = oracle.act_grad(act, zz)
    got_f = out[:, 0, :nk].double().cpu()
    got_g = dq[:, 0, 0].double().cpu()
    scale_z = torch.clamp(zz.abs(), min=1.0)
    bound_f = FWD_REL.get(act, 2.0 ** -8) * ref_f.abs() + FWD_BOUND.get(act, 0.0) * scale_z[:, None] + 1e-30
    bound_g = 2.0 ** -8 * ref_g.abs() + 2e-5 * scale_z + 1e-30
    bad_f = (got_f - ref_f).abs() > bound_f
    bad_g = (got_g - ref_g).abs() > bound_g
    if bad_f.any():
        rows, cols = torch.nonzero(bad_f, as_tuple=True)
        raise AssertionError(f"{act}: act mismatch at z={zz[rows[:5]].tolist()} columns {cols[:5].tolist()} "
                             f"got {got_f[rows[:5], cols[:5]].tolist()} ref {ref_f[rows[:5], cols[:5]].tolist()}")
    assert not bad_g.any(), f"{act}: act' mismatch at z={zz[bad_g][:5].tolist()} got {got_g[bad_g][:5].tolist()} " \
                            f"ref {ref_g[bad_g][:5].tolist()}"


# e4m3 forward: bound of the device evaluation before P is rounded to e4m3,
# as a multiple of max(1, |z|). gelu as for 16-bit P; fast_gelu and gelu_tanh
# mix the MUFU tanh form (about 2^-11 of tanh) with a fitted polynomial
# (|Phi error| <= 1.6e-4); silu takes fast_silu's MUFU tanh form.
FP8_BOUND = {"gelu": 4e-4, "gelu_tanh": 6e-4, "fast_gelu": 6e-4, "silu": 6e-4, "fast_silu": 6e-4,
             "fast_gelu_bf16": 6e-3}


@pytest.mark.parametrize("act", ELEMENTWISE)
def test_device_activation_pointwise_e4m3(act):
    # z = a + b / 32 with a, b e4m3 codes (exact in the fp32 accumulator);
    # every key is (1, 1/32, 0, ...) and v the identity, so out[i, j] is the
    # kernel's e4m3 P at tile column j, exactly representable in bf16.
    ensure_built()
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    a = codes[torch.isfinite(codes) & (codes.abs() <= 9)]
    b = torch.arange(-16.0, 17.0)
    z = (a[:, None] + b[None, :] / 32).reshape(-1)
    z, idx = torch.unique(z, return_inverse=True, sorted=True)
    aa = (a[:, None] + 0 * b[None, :]).reshape(-1)
    bb = (0 * a[:, None] + b[None, :]).reshape(-1)
    rep = torch.empty(z.numel(), dtype=torch.long).scatter_(0, idx, torch.arange(idx.numel()))  # one (a, b) per z
    n, d, nk = z.numel(), 128, 128
    q = torch.zeros(n, 1, d)
    q[:, 0, 0] = aa[rep]
    q[:, 0, 1] = bb[rep]
    kf = torch.zeros(nk, 1, d)
    kf[:, 0, 0] = 1
    kf[:, 0, 1] = 1.0 / 32
    vf = torch.eye(nk, d).reshape(nk, 1, d)
    f8 = torch.float8_e4m3fn
    assert torch.equal(q.to(f8).float(), q) and torch.equal(kf.to(f8).float(), kf)
    cu_q = torch.tensor([0, n], dtype=torch.int32).cuda()
    cu_k = torch.tensor([0, nk], dtype=torch.int32).cuda()
    desc = torch.ones(3, dtype=torch.float32).cuda()
    out, _ = _lib.gdpa_fwd(q.to(f8).cuda(), kf.to(f8).cuda(), vf.to(f8).cuda(), cu_q, cu_k, n, nk, act, 1.0,
                           descale_qkv=desc, batch=1)
    assert _lib.gdpa_get_status() == 0
    zz = z.double()
    assert torch.equal(q[:, 0, 0].double() + q[:, 0, 1].double() / 32, zz)
    ref = oracle.act_fwd(act, zz)[:, None].expand(n, nk)
    got = out[:, 0, :nk].double().cpu()
    # half an e4m3 ulp: 2^-4 of the value (normal), 2^-10 (subnormal step 2^-9)
    bound = 2.0 ** -4 * ref.abs() + 2.0 ** -10 + 1.07 * FP8_BOUND.get(act, 2e-5) * torch.clamp(zz.abs(), min=1.0)[:, None]
    bad = (got - ref).abs() > bound
    if bad.any():
        rows, cols = torch.nonzero(bad, as_tuple=True)
        raise AssertionError(f"{act}: e4m3 P mismatch at z={zz[rows[:5]].tolist()} columns {cols[:5].tolist()} "
                             f"got {got[rows[:5], cols[:5]].tolist()} ref {ref[rows[:5], cols[:5]].tolist()}")
