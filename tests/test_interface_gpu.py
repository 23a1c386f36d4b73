"""The PyTorch-facing API (flash_attn_varlen_func / flash_attn_func, the call
shapes of the gdpa/README.md page's "CUTE-DSL" block) as a
torch.autograd.Function: forward outputs and the gradients that .backward()
produces, against the float64 oracle, on jagged GQA inputs and on the
fixed-length [batch, seq, heads, dim] layout."""

import math

import pytest
import torch

import oracle
from generalized_attention_recsys_gb300 import inputs
from generalized_attention_recsys_gb300.interface import flash_attn_func, flash_attn_varlen_func
from gpu_util import FWD_TOL, GRAD_TOL, assert_close, ensure_built, ref_bwd, ref_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act,causal,window", [("gelu", False, -1), ("silu", True, -1), ("softmax", True, 50),
                                               ("relu2", False, 70)])
def test_varlen_autograd_matches_oracle(act, causal, window):
    ensure_built()
    lens_q, lens_k = [130, 1, 0, 257, 64], [200, 17, 5, 257, 1]
    inp = inputs.custom(5, 4, 2, 128, 128, lens_q, lens_k, act, causal=causal, window=window, seed=31)
    q, k, v = (t.cuda().requires_grad_(True) for t in (inp.q, inp.k, inp.v))
    out, lse = flash_attn_varlen_func(q, k, v, inp.cu_seqlens_q.cuda(), inp.cu_seqlens_k.cuda(), max(lens_q),
                                      max(lens_k), softmax_scale=inp.wl.softmax_scale, causal=causal,
                                      window=window, activation=act)
    ref_out, ref_lse = ref_fwd(inp)
    assert_close(out, ref_out, FWD_TOL, "out")
    if act == "softmax":
        finite = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse.cpu()), finite)
        assert_close(lse.cpu()[finite], ref_lse[finite], 1e-3, "lse")
    else:
        assert lse is None
    out.backward(inp.dout.cuda())
    rq, rk, rv = ref_bwd(inp)
    assert_close(q.grad, rq, GRAD_TOL, "dq")
    assert_close(k.grad, rk, GRAD_TOL, "dk")
    assert_close(v.grad, rv, GRAD_TOL, "dv")


def test_fixed_length_autograd_matches_oracle():
    ensure_built()
    b, n, h, d = 2, 200, 2, 64
    g = torch.Generator().manual_seed(32)
    q, k, v, do = (torch.randn(b, n, h, d, generator=g).to(torch.bfloat16) for _ in range(4))
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out, lse = flash_attn_func(qd, kd, vd, causal=True, activation="gelu_tanh")
    assert lse is None and out.shape == (b, n, h, d)
    out.backward(do.cuda())
    # the oracle on the packed view of the same memory
    pack = lambda t: t.double().reshape(b * n, h, d)
    scale = 1.0 / math.sqrt(d)
    ref_out, _ = oracle.gdpa_fwd(pack(q), pack(k), pack(v), None, None, b, n, n, "gelu_tanh", scale, True, -1)
    rq, rk, rv = oracle.gdpa_bwd(pack(q), pack(k), pack(v), pack(do), None, None, b, n, n, "gelu_tanh", scale,
                                 True, -1)
    assert_close(out.reshape(b * n, h, d), ref_out, FWD_TOL, "out")
    assert_close(qd.grad.reshape(b * n, h, d), rq, GRAD_TOL, "dq")
    assert_close(kd.grad.reshape(b * n, h, d), rk, GRAD_TOL, "dk")
    assert_close(vd.grad.reshape(b * n, h, d), rv, GRAD_TOL, "dv")
