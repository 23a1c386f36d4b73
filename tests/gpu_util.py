"""Helpers shared by the GPU parity tests: move seeded inputs to the GPU, run the
C-ABI through the binding, and compare with the float64 oracle."""

from __future__ import annotations

import torch

import oracle
from generalized_attention_recsys_gb300 import _lib, build

FWD_TOL = 2e-2      # bf16/fp16 forward: max|d| <= 2e-2 * max|ref| + 2e-3
FP8_TOL = 1e-1      # e4m3 forward
GRAD_TOL = 4e-2     # bf16/fp16 gradients, per tensor
ABS_TOL = 2e-3

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        _lib.load()
        _built = True


def to_dev(inp):
    d = {}
    for n in ("q", "k", "v", "dout"):
        t = getattr(inp, n)
        d[n] = None if t is None else t.cuda()
    fixed = inp.is_fixed_length()
    d["cu_q"] = None if fixed else inp.cu_seqlens_q.cuda()
    d["cu_k"] = None if fixed else inp.cu_seqlens_k.cuda()
    d["descale"] = None if inp.descale is None else torch.tensor(inp.descale, dtype=torch.float32).cuda()
    d["mx"] = None if inp.mx is None else tuple(t.cuda() for t in inp.mx)
    return d


def max_lens(inp):
    if inp.is_fixed_length():
        return inp.wl.max_q, inp.wl.max_k
    return max(inp.max_q, 1), max(inp.max_k, 1)


def run_fwd(inp, act=None):
    ensure_built()
    wl = inp.wl
    d = to_dev(inp)
    mq, mk = max_lens(inp)
    if d["mx"] is not None:
        out, lse = _lib.gdpa_fwd_mxfp8(d["q"], d["k"], d["v"], *d["mx"], d["cu_q"], d["cu_k"], mq, mk, act or wl.act,
                                       wl.softmax_scale, wl.causal, wl.window, batch=wl.batch)
    else:
        out, lse = _lib.gdpa_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], mq, mk, act or wl.act,
                                 wl.softmax_scale, wl.causal, wl.window, descale_qkv=d["descale"], batch=wl.batch)
    assert _lib.gdpa_get_status() == 0
    return out, lse


def run_bwd(inp, out=None, lse=None, deterministic=False):
    ensure_built()
    wl = inp.wl
    d = to_dev(inp)
    mq, mk = max_lens(inp)
    dq, dk, dv = _lib.gdpa_bwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], mq, mk, wl.act, wl.softmax_scale,
                               wl.causal, wl.window, out, lse, d["dout"], deterministic=deterministic,
                               batch=wl.batch)
    assert _lib.gdpa_get_status() == 0
    return dq, dk, dv


def ref_fwd(inp, units=None):
    wl = inp.wl
    cu_q = None if inp.is_fixed_length() else inp.cu_seqlens_q
    cu_k = None if inp.is_fixed_length() else inp.cu_seqlens_k
    return oracle.gdpa_fwd(inp.values("q"), inp.values("k"), inp.values("v"), cu_q, cu_k, wl.batch, wl.max_q,
                           wl.max_k, wl.act, wl.softmax_scale, wl.causal, wl.window, units=units)


def ref_bwd(inp, units=None):
    wl = inp.wl
    cu_q = None if inp.is_fixed_length() else inp.cu_seqlens_q
    cu_k = None if inp.is_fixed_length() else inp.cu_seqlens_k
    return oracle.gdpa_bwd(inp.values("q"), inp.values("k"), inp.values("v"), inp.dout.double(), cu_q, cu_k,
                           wl.batch, wl.max_q, wl.max_k, wl.act, wl.softmax_scale, wl.causal, wl.window,
                           units=units)


def assert_close(got, ref, rel, what=""):
    got = got.detach().double().cpu()
    ref = ref.detach().double().cpu()
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite values"
    err = (got - ref).abs().max().item() if ref.numel() else 0.0
    bound = rel * (ref.abs().max().item() if ref.numel() else 0.0) + ABS_TOL
    assert err <= bound, f"{what}: max|d|={err:.3e} > {bound:.3e} (max|ref|={ref.abs().max().item():.3e})"
    return err, bound
