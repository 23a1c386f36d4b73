"""Backward with one key block per sequence (max_seqlen_k <= 128): dQ has a
single producer per row and the kernel writes it in the output type, with no
fp32 accumulator. Checked against the float64 oracle on ragged query lengths
(empty, partial and multi-tile sequences), key lengths up to 128 (including
empty), causal and windowed masks that leave whole query tiles without keys,
GQA, softmax and fp16; dq is pre-filled with a sentinel so that every element
must be written. Also: a max_seqlen_k below a real key length is reported
through the device status instead of writing outside the workspace."""

import pytest
import torch

import oracle
from generalized_attention_recsys_gb300 import _lib, inputs
from gpu_util import GRAD_TOL, assert_close, ensure_built, ref_bwd, run_bwd, run_fwd, to_dev

pytestmark = pytest.mark.gpu

LQ = [300, 0, 1, 128, 129, 513, 77, 256]
LK = [50, 20, 0, 128, 1, 128, 127, 64]


def _bwd_into(inp, out, lse, deterministic, sentinel=7.0, max_k=None):
    wl = inp.wl
    d = to_dev(inp)
    mq = max(inp.max_q, 1)
    mk = max(inp.max_k, 1) if max_k is None else max_k
    dq = torch.full_like(d["q"], sentinel)
    dk = torch.full_like(d["k"], sentinel)
    dv = torch.full_like(d["v"], sentinel)
    _lib.gdpa_bwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], mq, mk, wl.act, wl.softmax_scale, wl.causal,
                  wl.window, out, lse, d["dout"], dq=dq, dk=dk, dv=dv, deterministic=deterministic, batch=wl.batch)
    return dq, dk, dv


@pytest.mark.parametrize(
    "h_q,h_kv,d,act,causal,window,dtype",
    [
        (4, 4, 128, "gelu", False, -1, "bf16"),
        (4, 2, 128, "relu2", True, -1, "bf16"),
        (4, 1, 64, "silu", True, 40, "bf16"),
        (2, 2, 96, "gelu_tanh", False, 30, "bf16"),
        (2, 2, 128, "softmax", True, -1, "bf16"),
        (2, 2, 128, "identity", False, -1, "fp16"),
        (4, 2, 192, "gelu", True, 50, "bf16"),
    ],
)
@pytest.mark.parametrize("deterministic", [False, True])
def test_direct_dq_matches_oracle_and_writes_every_row(h_q, h_kv, d, act, causal, window, dtype, deterministic):
    ensure_built()
    dv_ = 128 if d == 192 else d  # (192, 128): dQ written by two column-part items
    inp = inputs.custom(len(LQ), h_q, h_kv, d, dv_, LQ, LK, act, causal=causal, window=window, dtype=dtype, seed=21)
    out, lse = run_fwd(inp) if act == "softmax" else (None, None)
    dq, dk, dv = _bwd_into(inp, out, lse, deterministic)
    assert _lib.gdpa_get_status() == 0
    rq, rk, rv = ref_bwd(inp)
    assert_close(dq, rq, GRAD_TOL, "dq")
    assert_close(dk, rk, GRAD_TOL, "dk")
    assert_close(dv, rv, GRAD_TOL, "dv")
    # rows with no allowed key (whole query tiles among them) are exact zeros, not the sentinel
    keyless = torch.cat([~oracle.allowed_mask(lq, lk, causal, window).any(dim=1) for lq, lk in zip(LQ, LK)])
    assert keyless.any()
    assert torch.count_nonzero(dq.double().cpu()[keyless]) == 0
    # one producer per row: the same bits on every call
    dq2, dk2, dv2 = _bwd_into(inp, out, lse, deterministic, sentinel=-3.0)
    assert _lib.gdpa_get_status() == 0
    assert torch.equal(dq2, dq) and torch.equal(dk2, dk) and torch.equal(dv2, dv)


@pytest.mark.parametrize("max_k,deterministic", [(128, False), (256, False), (256, True)])
def test_understated_max_seqlen_k_is_reported(max_k, deterministic):
    # key lengths up to 400 but a smaller max_seqlen_k: the workspace (in the
    # deterministic mode, the number of dQ slices) and, at 128, the direct dQ
    # mode are sized for fewer key blocks. The kernel must write nothing for
    # the blocks beyond and report it.
    ensure_built()
    lq, lk = [200, 64, 300], [300, 128, 400]
    inp = inputs.custom(3, 2, 2, 128, 128, lq, lk, "gelu", seed=22)
    _bwd_into(inp, None, None, deterministic, max_k=max_k)
    assert _lib.gdpa_get_status() == _lib.GDPA_ERR_INVALID
    # the device stays usable: a correct call afterwards passes
    dq, dk, dv = run_bwd(inp, deterministic=deterministic)
    rq, rk, rv = ref_bwd(inp)
    assert_close(dq, rq, GRAD_TOL, "dq")
