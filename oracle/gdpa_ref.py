"""Plain float64 CPU oracle for Generalized Dot Product Attention (GDPA).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The product path
(the CUDA library and its Python binding) never calls it, and this module
imports nothing from the product package.

What it computes follows the gdpa/README.md page of
facebookresearch/ads_model_kernel_library:

* intro paragraph: GDPA is dot-product attention whose softmax is replaced by
  an elementwise activation;
* "Features": activations (GELU, GELUApprox, FastGELU, ReLU, ReLU^2,
  LeakyReLU, SiLU, HardSwish, identity), causal / non-causal / sliding-window
  masks, MHA/GQA/MQA, jagged (variable-length) sequences;
* "CUTE-DSL" API block: ``flash_attn_varlen_func(q, k, v, cu_seqlens_q,
  cu_seqlens_k, max_seqlen_q, max_seqlen_k, activation=...)`` on packed
  ``[total_tokens, heads, head_dim]`` tensors.

The Dao-AILab/flash-attention overview page fixes the softmax cross-check
mode (online softmax with a log-sum-exp per row) and the packed varlen layout.

For each sequence b and query head h (kv head g = h // (Hq / Hkv)):

    S = Q_bh K_bg^T,   Z = scale * S,   P = where(M, act(Z), 0),   O = P V_bg

with M the allowed-position mask. There is no row normalisation. Backward
with upstream gradient dO:

    dV_bg += P^T dO,   dP = dO V_bg^T,   dZ = where(M, dP * act'(Z), 0),
    dS = scale * dZ,   dQ_bh = dS K_bg,   dK_bg += dS^T Q_bh

S, Z, P, dP and dS are materialised as full matrices; no blocking, fusion or
reordering is applied beyond the definition.

Readings taken where the pages are silent (each is also listed with the
design notes):

* activation formulas: the textbook definitions written below;
* ``fast_gelu`` is the same function as ``gelu_tanh`` (the page lists it as a
  faster evaluation, not a different function) -- parity unpinned by the
  pages;
* ``fast_gelu_bf16`` ("FastGELU (BF16)") is again ``gelu_tanh``, evaluated by
  the kernels in bf16 arithmetic, and ``fast_silu`` ("FastSiLU") is ``silu``
  evaluated through tanh; the oracle computes the exact functions -- parity
  unpinned by the pages;
* LeakyReLU slope 0.01 -- parity unpinned by the pages;
* derivatives at kinks follow PyTorch's conventions;
* causal with Lq != Lk is bottom-right aligned: allowed iff j <= i + Lk - Lq;
* window W > 0 with causal: allowed iff 0 <= (i + Lk - Lq) - j < W;
  W > 0 without causal: |i + Lk - Lq - j| < W; W <= 0: no window --
  parity unpinned by the pages;
* rows with no allowed key produce an all-zero output (softmax: lse = -inf).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

ACTIVATIONS = (
    "identity",
    "gelu",
    "gelu_tanh",
    "fast_gelu",
    "relu",
    "relu2",
    "leaky_relu",
    "silu",
    "hardswish",
    "softmax",
    "fast_gelu_bf16",
    "fast_silu",
)

LEAKY_SLOPE = 0.01
_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_TANH_CUBIC = 0.044715
_INV_SQRT_2 = 1.0 / math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


# --------------------------------------------------------------------------
# Activations and their derivatives ("Features": custom activations)
# --------------------------------------------------------------------------

def act_fwd(name: str, z: torch.Tensor) -> torch.Tensor:
    """Elementwise activation act(z) in float64, written out from its definition."""
    if name == "identity":
        return z.clone()
    if name == "gelu":
        return 0.5 * z * (1.0 + torch.erf(z * _INV_SQRT_2))
    if name in ("gelu_tanh", "fast_gelu", "fast_gelu_bf16"):
        u = _SQRT_2_OVER_PI * (z + _TANH_CUBIC * z * z * z)
        return 0.5 * z * (1.0 + torch.tanh(u))
    if name == "relu":
        return torch.where(z > 0, z, torch.zeros_like(z))
    if name == "relu2":
        r = torch.where(z > 0, z, torch.zeros_like(z))
        return r * r
    if name == "leaky_relu":
        return torch.where(z > 0, z, LEAKY_SLOPE * z)
    if name in ("silu", "fast_silu"):
        return z / (1.0 + torch.exp(-z))
    if name == "hardswish":
        return z * torch.clamp(z + 3.0, 0.0, 6.0) / 6.0
    raise ValueError(f"no elementwise activation named {name!r}")


def act_grad(name: str, z: torch.Tensor) -> torch.Tensor:
    """d act / d z in float64; kinks follow PyTorch's backward conventions."""
    one = torch.ones_like(z)
    zero = torch.zeros_like(z)
    if name == "identity":
        return one
    if name == "gelu":
        cdf = 0.5 * (1.0 + torch.erf(z * _INV_SQRT_2))
        pdf = _INV_SQRT_2PI * torch.exp(-0.5 * z * z)
        return cdf + z * pdf
    if name in ("gelu_tanh", "fast_gelu", "fast_gelu_bf16"):
        u = _SQRT_2_OVER_PI * (z + _TANH_CUBIC * z * z * z)
        t = torch.tanh(u)
        du = _SQRT_2_OVER_PI * (1.0 + 3.0 * _TANH_CUBIC * z * z)
        return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * du
    if name == "relu":
        return torch.where(z > 0, one, zero)
    if name == "relu2":
        return torch.where(z > 0, 2.0 * z, zero)
    if name == "leaky_relu":
        return torch.where(z > 0, one, LEAKY_SLOPE * one)
    if name in ("silu", "fast_silu"):
        sig = 1.0 / (1.0 + torch.exp(-z))
        return sig * (1.0 + z * (1.0 - sig))
    if name == "hardswish":
        # PyTorch's convention: the middle branch is the open interval (-3, 3)
        mid = z / 3.0 + 0.5
        return torch.where(z <= -3.0, zero, torch.where(z < 3.0, mid, one))
    raise ValueError(f"no elementwise activation named {name!r}")


# --------------------------------------------------------------------------
# Masks ("Features": causal, non-causal, sliding window)
# --------------------------------------------------------------------------

def allowed_mask(lq: int, lk: int, causal: bool, window: int) -> torch.Tensor:
    """Boolean [lq, lk]: True where query i may attend key j.

    The query row i is aligned to key position i + lk - lq (bottom-right
    alignment), so for lq == lk the diagonal is i == j.
    """
    i = torch.arange(lq, dtype=torch.int64).unsqueeze(1)
    j = torch.arange(lk, dtype=torch.int64).unsqueeze(0)
    diag = i + (lk - lq) - j  # >= 0 means key j is at or before the query's position
    m = torch.ones(lq, lk, dtype=torch.bool)
    if causal:
        m &= diag >= 0
        if window > 0:
            m &= diag < window
    elif window > 0:
        m &= diag.abs() < window
    return m


# --------------------------------------------------------------------------
# One (sequence, head) unit
# --------------------------------------------------------------------------

@dataclass
class UnitFwd:
    out: torch.Tensor          # [lq, dv]
    lse: torch.Tensor | None   # [lq] (softmax only)
    s: torch.Tensor            # [lq, lk] raw Q K^T
    p: torch.Tensor            # [lq, lk] masked activation (or softmax probabilities)
    mask: torch.Tensor         # [lq, lk]


def unit_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, act: str,
             scale: float, causal: bool, window: int) -> UnitFwd:
    """GDPA forward for one unit. q [lq,dqk], k [lk,dqk], v [lk,dv], float64."""
    lq, lk = q.shape[0], k.shape[0]
    m = allowed_mask(lq, lk, causal, window)
    s = q @ k.transpose(0, 1)
    z = scale * s
    if act == "softmax":
        neg_inf = torch.full_like(z, -math.inf)
        zm = torch.where(m, z, neg_inf)
        rowmax = zm.max(dim=1, keepdim=True).values if lk > 0 else torch.full((lq, 1), -math.inf, dtype=z.dtype)
        safe_max = torch.where(torch.isfinite(rowmax), rowmax, torch.zeros_like(rowmax))
        e = torch.where(m, torch.exp(z - safe_max), torch.zeros_like(z))
        denom = e.sum(dim=1, keepdim=True)
        has_key = denom > 0
        p = torch.where(has_key, e / torch.where(has_key, denom, torch.ones_like(denom)), torch.zeros_like(e))
        lse = torch.where(has_key, safe_max + torch.log(torch.where(has_key, denom, torch.ones_like(denom))),
                          torch.full_like(denom, -math.inf)).squeeze(1)
    else:
        p = torch.where(m, act_fwd(act, z), torch.zeros_like(z))
        lse = None
    out = p @ v
    return UnitFwd(out=out, lse=lse, s=s, p=p, mask=m)


@dataclass
class UnitBwd:
    dq: torch.Tensor   # [lq, dqk]
    dk: torch.Tensor   # [lk, dqk] (this query head's contribution)
    dv: torch.Tensor   # [lk, dv]  (this query head's contribution)
    dp: torch.Tensor   # [lq, lk]
    ds: torch.Tensor   # [lq, lk]


def unit_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor,
             act: str, scale: float, causal: bool, window: int) -> UnitBwd:
    """GDPA backward for one unit, every intermediate materialised."""
    f = unit_fwd(q, k, v, act, scale, causal, window)
    dv = f.p.transpose(0, 1) @ dout
    dp = dout @ v.transpose(0, 1)
    if act == "softmax":
        d_row = (dout * f.out).sum(dim=1, keepdim=True)
        dz = f.p * (dp - d_row)
    else:
        z = scale * f.s
        dz = torch.where(f.mask, dp * act_grad(act, z), torch.zeros_like(dp))
    ds = scale * dz
    dq = ds @ k
    dk = ds.transpose(0, 1) @ q
    return UnitBwd(dq=dq, dk=dk, dv=dv, dp=dp, ds=ds)


# --------------------------------------------------------------------------
# Packed (jagged) tensors: [total_tokens, heads, head_dim] + cu_seqlens
# --------------------------------------------------------------------------

def _bounds(cu: torch.Tensor | None, b: int, fixed_len: int) -> tuple[int, int]:
    if cu is None:
        return b * fixed_len, (b + 1) * fixed_len
    return int(cu[b]), int(cu[b + 1])


def _group(hq: int, hkv: int) -> int:
    if hq % hkv != 0:
        raise ValueError("query heads must be a multiple of kv heads")
    return hq // hkv


def gdpa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
             cu_seqlens_q: torch.Tensor | None, cu_seqlens_k: torch.Tensor | None,
             batch: int, max_seqlen_q: int, max_seqlen_k: int, act: str,
             scale: float, causal: bool = False, window: int = -1,
             units: list[tuple[int, int]] | None = None):
    """Packed GDPA forward in float64.

    q [Tq, Hq, dqk], k [Tk, Hkv, dqk], v [Tk, Hkv, dv]. ``cu_seqlens_*`` are
    int [batch+1] offsets, or None for fixed-length sequences of
    ``max_seqlen_*`` tokens. ``units`` restricts the work to the listed
    (sequence, query head) pairs; rows of other units stay zero.

    Returns (out [Tq, Hq, dv], lse [Hq, Tq] or None).
    """
    q, k, v = q.double(), k.double(), v.double()
    tq, hq, _ = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    grp = _group(hq, hkv)
    out = torch.zeros(tq, hq, dv, dtype=torch.float64)
    lse = torch.full((hq, tq), -math.inf, dtype=torch.float64) if act == "softmax" else None
    todo = units if units is not None else [(b, h) for b in range(batch) for h in range(hq)]
    for b, h in todo:
        q0, q1 = _bounds(cu_seqlens_q, b, max_seqlen_q)
        k0, k1 = _bounds(cu_seqlens_k, b, max_seqlen_k)
        g = h // grp
        f = unit_fwd(q[q0:q1, h], k[k0:k1, g], v[k0:k1, g], act, scale, causal, window)
        out[q0:q1, h] = f.out
        if lse is not None:
            lse[h, q0:q1] = f.lse
    return out, lse


def gdpa_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor,
             cu_seqlens_q: torch.Tensor | None, cu_seqlens_k: torch.Tensor | None,
             batch: int, max_seqlen_q: int, max_seqlen_k: int, act: str,
             scale: float, causal: bool = False, window: int = -1,
             units: list[tuple[int, int]] | None = None):
    """Packed GDPA backward in float64: returns (dq, dk, dv).

    dk and dv of kv head g sum the contributions of every query head in g's
    group (GQA/MQA). With ``units`` only those (sequence, query head) pairs
    contribute.
    """
    q, k, v, dout = q.double(), k.double(), v.double(), dout.double()
    tq, hq, dqk = q.shape
    tk, hkv, dv_dim = v.shape
    grp = _group(hq, hkv)
    dq = torch.zeros(tq, hq, dqk, dtype=torch.float64)
    dk = torch.zeros(tk, hkv, dqk, dtype=torch.float64)
    dv = torch.zeros(tk, hkv, dv_dim, dtype=torch.float64)
    todo = units if units is not None else [(b, h) for b in range(batch) for h in range(hq)]
    for b, h in todo:
        q0, q1 = _bounds(cu_seqlens_q, b, max_seqlen_q)
        k0, k1 = _bounds(cu_seqlens_k, b, max_seqlen_k)
        g = h // grp
        r = unit_bwd(q[q0:q1, h], k[k0:k1, g], v[k0:k1, g], dout[q0:q1, h], act, scale, causal, window)
        dq[q0:q1, h] = r.dq
        dk[k0:k1, g] += r.dk
        dv[k0:k1, g] += r.dv
    return dq, dk, dv
