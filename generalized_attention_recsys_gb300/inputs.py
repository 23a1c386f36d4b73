"""Seeded synthetic inputs for GDPA workloads.

This module is shared by the tests, the benchmark and the oracle checks. It
draws random numbers and encodes them in the requested storage type; it
holds none of the attention arithmetic.

Recipe (one ``torch.Generator`` on the CPU, seeded per call), in draw order:

1. query lengths (``torch.randint``, inclusive bounds), when jagged;
2. key lengths, when jagged and drawn independently of the query lengths;
3. q, k, v, dout with ``torch.randn`` in float32;
4. cast once to bf16/fp16, or quantise to FP8 E4M3 with a per-tensor scale
   ``s = amax / 448`` (round to nearest even, no overflow by construction).

The workloads mirror the benchmark scenarios on the gdpa/README.md page
("Benchmark Results": self-attention at sparsity 1.0 and 0.5, cross-attention
with short KV). "Sparsity 0.5" is read as lengths uniform in [1, max], so
that the mean length is about half the maximum.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_q: int
    h_kv: int
    d_qk: int
    d_v: int
    max_q: int
    max_k: int
    act: str
    causal: bool = False
    window: int = -1
    jagged_q: tuple[int, int] | None = None   # inclusive (lo, hi) when Q lengths are drawn
    jagged_k: tuple[int, int] | None = None   # inclusive (lo, hi) when K lengths are drawn independently
    k_follows_q: bool = False                 # self-attention: key length = query length
    dtype: str = "bf16"                       # "bf16", "fp16", "e4m3" or "mxe4m3" (MXFP8)
    scale: float | None = None                # None = 1/sqrt(d_qk)
    fwd_only: bool = False
    notes: str = field(default="", compare=False)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d_qk)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    "tiny_fixed": Workload(
        "tiny_fixed", batch=2, h_q=2, h_kv=2, d_qk=64, d_v=64, max_q=128, max_k=128,
        act="fast_gelu", scale=1.0 / 8.0,
        notes="B=2 H=2 N=128 d=64 bf16, fast_gelu, non-causal"),
    "jagged_self": Workload(
        "jagged_self", batch=64, h_q=4, h_kv=4, d_qk=128, d_v=128, max_q=2048, max_k=2048,
        act="gelu", jagged_q=(1, 2048), k_follows_q=True,
        notes="B=64 H=4 d=128 bf16, lengths U[1,2048] (Lq=Lk), gelu, non-causal"),
    "dense_causal": Workload(
        "dense_causal", batch=32, h_q=8, h_kv=8, d_qk=128, d_v=128, max_q=4096, max_k=4096,
        act="silu", causal=True,
        notes="B=32 H=8 N=4096 d=128 bf16, causal, silu"),
    "short_kv_cross": Workload(
        "short_kv_cross", batch=512, h_q=4, h_kv=4, d_qk=128, d_v=128, max_q=1024, max_k=128,
        act="relu2", jagged_q=(64, 1024),
        notes="B=512 H=4 d=128 bf16, Lq U[64,1024], Lk=128, relu2, non-causal"),
    "gqa_window_fp8": Workload(
        "gqa_window_fp8", batch=16, h_q=16, h_kv=2, d_qk=192, d_v=128, max_q=8192, max_k=8192,
        act="fast_gelu", causal=True, window=512, dtype="e4m3", fwd_only=True,
        notes="B=16 Hq=16 Hkv=2 dqk=192 dv=128 N=8192, causal window 512, e4m3, fast_gelu"),
    "gqa_window_mxfp8": Workload(
        "gqa_window_mxfp8", batch=16, h_q=16, h_kv=2, d_qk=192, d_v=128, max_q=8192, max_k=8192,
        act="fast_gelu", causal=True, window=512, dtype="mxe4m3", fwd_only=True,
        notes="the gqa_window_fp8 shapes with MXFP8 inputs (e4m3, E8M0 scale per 32 elements)"),
    "gqa_window_softmax": Workload(
        "gqa_window_softmax", batch=16, h_q=16, h_kv=2, d_qk=192, d_v=128, max_q=8192, max_k=8192,
        act="softmax", causal=True, window=512, dtype="bf16", fwd_only=True,
        notes="same shapes as gqa_window_fp8 in bf16 with softmax"),
}


@dataclass
class Inputs:
    wl: Workload
    lengths_q: torch.Tensor          # int64 [B]
    lengths_k: torch.Tensor          # int64 [B]
    cu_seqlens_q: torch.Tensor       # int32 [B+1]
    cu_seqlens_k: torch.Tensor       # int32 [B+1]
    q: torch.Tensor                  # storage dtype, [Tq, Hq, dqk]
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor | None        # bf16/fp16 [Tq, Hq, dv] (None when forward only)
    descale: tuple[float, float, float] | None = None   # e4m3: per-tensor scales of q, k, v
    fixed_length: bool = False       # every sequence has max_q / max_k tokens (no cu_seqlens)
    mx: tuple[torch.Tensor, torch.Tensor, torch.Tensor] | None = None  # MXFP8: E8M0 scales of q, k, v

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_seqlens_k[-1])

    @property
    def max_q(self) -> int:
        return int(self.lengths_q.max()) if self.lengths_q.numel() else 0

    @property
    def max_k(self) -> int:
        return int(self.lengths_k.max()) if self.lengths_k.numel() else 0

    def values(self, name: str) -> torch.Tensor:
        """The exact values the kernel sees, as float64 (dequantised for e4m3)."""
        t = getattr(self, name)
        if t.dtype == torch.float8_e4m3fn and self.mx is not None:
            sc = self.mx[("q", "k", "v").index(name)]
            return mx_values(t, sc, along_tokens=(name == "v"))
        if t.dtype == torch.float8_e4m3fn:
            s = self.descale[("q", "k", "v").index(name)]
            return t.double() * s
        return t.double()

    def is_fixed_length(self) -> bool:
        return self.fixed_length


def _cu(lengths: torch.Tensor) -> torch.Tensor:
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    return cu


def quantize_e4m3(x: torch.Tensor) -> tuple[torch.Tensor, float]:
    """Per-tensor FP8 E4M3 encoding: returns (codes, scale) with x ~ codes * scale."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    s = amax / E4M3_MAX if amax > 0 else 1.0
    return (x / s).to(torch.float8_e4m3fn), s


# OCP Microscaling (MX) v1.0 encoding of the MXFP8 inputs: blocks of 32
# elements share one E8M0 scale byte s (value 2^(s - 127)); the shared
# exponent is floor(log2(block amax)) - 8, 8 being the largest exponent of an
# e4m3 element, and elements are rounded to e4m3 with saturation at 448.
MX_BLOCK = 32
E8M0_BIAS = 127


def _mx_encode(blocks: torch.Tensor, dim: int) -> tuple[torch.Tensor, torch.Tensor]:
    amax = blocks.abs().amax(dim=dim, keepdim=True)
    e = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 8,
                    torch.full_like(amax, -E8M0_BIAS))
    e = e.clamp(-E8M0_BIAS, E8M0_BIAS)
    codes = (blocks / torch.exp2(e)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes, (e + E8M0_BIAS).to(torch.uint8).squeeze(dim)


def quantize_mx_rows(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """MX blocks along the last dim (q, k: [T, H, d], d % 32 == 0): (codes, scales [T, H, d / 32])."""
    t, h, d = x.shape
    codes, sc = _mx_encode(x.reshape(t, h, d // MX_BLOCK, MX_BLOCK), 3)
    return codes.reshape(t, h, d), sc


def quantize_mx_tokens(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """MX blocks along the token dim (v: [T, H, d]): blocks of 32 packed tokens, the last one
    zero-padded: (codes [T, H, d], scales [ceil(T / 32), H, d])."""
    t, h, d = x.shape
    nb = (t + MX_BLOCK - 1) // MX_BLOCK
    xp = torch.zeros(nb * MX_BLOCK, h, d, dtype=x.dtype)
    xp[:t] = x
    codes, sc = _mx_encode(xp.reshape(nb, MX_BLOCK, h, d), 1)
    return codes.reshape(nb * MX_BLOCK, h, d)[:t], sc


def mx_values(codes: torch.Tensor, scales: torch.Tensor, along_tokens: bool) -> torch.Tensor:
    """float64 values of MX codes: code * 2^(s - 127), s the scale of the code's block."""
    c = codes.double()
    f = torch.exp2(scales.double() - E8M0_BIAS)
    if along_tokens:
        return c * f.repeat_interleave(MX_BLOCK, dim=0)[: c.shape[0]]
    return c * f.repeat_interleave(MX_BLOCK, dim=2)


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "fp16":
        return x.to(torch.float16)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def make_inputs(wl: Workload, seed: int = 0, with_dout: bool | None = None) -> Inputs:
    """Draw a workload's inputs on the CPU following the module's recipe."""
    g = torch.Generator().manual_seed(seed)
    b = wl.batch
    if wl.jagged_q is not None:
        lo, hi = wl.jagged_q
        lq = torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int64)
    else:
        lq = torch.full((b,), wl.max_q, dtype=torch.int64)
    if wl.k_follows_q:
        lk = lq.clone()
    elif wl.jagged_k is not None:
        lo, hi = wl.jagged_k
        lk = torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int64)
    else:
        lk = torch.full((b,), wl.max_k, dtype=torch.int64)
    cu_q, cu_k = _cu(lq), _cu(lk)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q = torch.randn(tq, wl.h_q, wl.d_qk, generator=g)
    k = torch.randn(tk, wl.h_kv, wl.d_qk, generator=g)
    v = torch.randn(tk, wl.h_kv, wl.d_v, generator=g)
    need_dout = (not wl.fwd_only) if with_dout is None else with_dout
    dout = torch.randn(tq, wl.h_q, wl.d_v, generator=g) if need_dout else None
    descale = mx = None
    if wl.dtype == "e4m3":
        q, sq = quantize_e4m3(q)
        k, sk = quantize_e4m3(k)
        v, sv = quantize_e4m3(v)
        descale = (sq, sk, sv)
        if dout is not None:
            dout = dout.to(torch.bfloat16)
    elif wl.dtype == "mxe4m3":
        (q, sq), (k, sk), (v, sv) = quantize_mx_rows(q), quantize_mx_rows(k), quantize_mx_tokens(v)
        mx = (sq, sk, sv)
        if dout is not None:
            dout = dout.to(torch.bfloat16)
    else:
        q, k, v = _cast(q, wl.dtype), _cast(k, wl.dtype), _cast(v, wl.dtype)
        if dout is not None:
            dout = _cast(dout, wl.dtype)
    fixed = wl.jagged_q is None and wl.jagged_k is None and not wl.k_follows_q
    return Inputs(wl, lq, lk, cu_q, cu_k, q, k, v, dout, descale, fixed, mx)


def custom(batch: int, h_q: int, h_kv: int, d_qk: int, d_v: int, lengths_q, lengths_k,
           act: str, causal: bool = False, window: int = -1, dtype: str = "bf16",
           scale: float | None = None, seed: int = 0, with_dout: bool = True) -> Inputs:
    """Inputs with explicit per-sequence lengths (edge cases: 0, 1, ragged tails)."""
    lq = torch.as_tensor(lengths_q, dtype=torch.int64)
    lk = torch.as_tensor(lengths_k, dtype=torch.int64)
    assert lq.numel() == batch and lk.numel() == batch
    wl = Workload("custom", batch, h_q, h_kv, d_qk, d_v,
                  int(lq.max()) if batch else 0, int(lk.max()) if batch else 0,
                  act, causal, window, dtype=dtype, scale=scale)
    g = torch.Generator().manual_seed(seed)
    cu_q, cu_k = _cu(lq), _cu(lk)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q = torch.randn(tq, h_q, d_qk, generator=g)
    k = torch.randn(tk, h_kv, d_qk, generator=g)
    v = torch.randn(tk, h_kv, d_v, generator=g)
    dout = torch.randn(tq, h_q, d_v, generator=g) if with_dout else None
    descale = mx = None
    if dtype == "e4m3":
        q, sq = quantize_e4m3(q)
        k, sk = quantize_e4m3(k)
        v, sv = quantize_e4m3(v)
        descale = (sq, sk, sv)
        dout = dout.to(torch.bfloat16) if dout is not None else None
    elif dtype == "mxe4m3":
        (q, sq), (k, sk), (v, sv) = quantize_mx_rows(q), quantize_mx_rows(k), quantize_mx_tokens(v)
        mx = (sq, sk, sv)
        dout = dout.to(torch.bfloat16) if dout is not None else None
    else:
        q, k, v = _cast(q, dtype), _cast(k, dtype), _cast(v, dtype)
        dout = _cast(dout, dtype) if dout is not None else None
    return Inputs(wl, lq, lk, cu_q, cu_k, q, k, v, dout, descale, False, mx)
