"""PyTorch-facing GDPA API with autograd.

Mirrors the calls shown in the "CUTE-DSL" block of the gdpa/README.md page:
``flash_attn_varlen_func(q, k, v, cu_seqlens_q=..., cu_seqlens_k=...,
max_seqlen_q=..., max_seqlen_k=..., activation=...)`` on packed
``[tokens, heads, dim]`` tensors and ``flash_attn_func(q, k, v,
softmax_scale=..., causal=...)`` on ``[batch, seq, heads, dim]``. Both
return ``(out, lse)``; ``lse`` is None for elementwise activations (it has no
meaning without a softmax).
"""

from __future__ import annotations

import math

import torch

from . import _lib


class _GdpaFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_q, cu_k, max_q, max_k, act, scale, causal, window, batch, deterministic):
        out, lse = _lib.gdpa_fwd(q, k, v, cu_q, cu_k, max_q, max_k, act, scale, causal, window, batch=batch)
        ctx.save_for_backward(q, k, v, cu_q, cu_k, out, lse)
        ctx.cfg = (max_q, max_k, act, scale, causal, window, batch, deterministic)
        return out, lse

    @staticmethod
    def backward(ctx, dout, dlse):
        q, k, v, cu_q, cu_k, out, lse = ctx.saved_tensors
        max_q, max_k, act, scale, causal, window, batch, deterministic = ctx.cfg
        dq, dk, dv = _lib.gdpa_bwd(q, k, v, cu_q, cu_k, max_q, max_k, act, scale, causal, window, out, lse,
                                   dout, deterministic=deterministic, batch=batch)
        return dq, dk, dv, None, None, None, None, None, None, None, None, None, None


def flash_attn_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           softmax_scale=None, causal=False, window=-1, activation="fast_gelu",
                           deterministic=False):
    """GDPA on packed q [Tq, Hq, dqk], k [Tk, Hkv, dqk], v [Tk, Hkv, dv].
    deterministic=True makes the backward's dq bitwise reproducible."""
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(q.shape[-1])
    batch = cu_seqlens_q.numel() - 1
    cu_q = cu_seqlens_q.to(device=q.device, dtype=torch.int32)
    cu_k = cu_seqlens_k.to(device=q.device, dtype=torch.int32)
    return _GdpaFn.apply(q, k, v, cu_q, cu_k, int(max_seqlen_q), int(max_seqlen_k), activation, float(scale),
                         bool(causal), int(window), batch, bool(deterministic))


def flash_attn_func(q, k, v, softmax_scale=None, causal=False, window=-1, activation="fast_gelu",
                    deterministic=False):
    """GDPA on fixed-length q [B, Nq, Hq, dqk], k/v [B, Nk, Hkv, d]."""
    b, nq, hq, dqk = q.shape
    nk = k.shape[1]
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    qp, kp, vp = (t.reshape(-1, t.shape[2], t.shape[3]) for t in (q, k, v))
    out, lse = _GdpaFn.apply(qp.contiguous(), kp.contiguous(), vp.contiguous(), None, None, nq, nk, activation,
                             float(scale), bool(causal), int(window), b, bool(deterministic))
    out = out.view(b, nq, hq, v.shape[3])
    return out, (lse.view(hq, b, nq) if lse is not None else None)
