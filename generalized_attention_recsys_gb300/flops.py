"""Useful-work accounting for GDPA throughput figures (host side).

Counts the (query, key) positions a mask allows, so that throughput excludes
masked and padded work. It computes no attention.
"""

from __future__ import annotations


def allowed_pairs(lengths_q, lengths_k, causal: bool, window: int) -> int:
    """Number of allowed (query, key) pairs summed over sequences, for one head.

    Used only to count useful FLOPs (masked and padded work excluded); it
    counts positions, it computes no attention.
    """
    total = 0
    for lq, lk in zip([int(x) for x in lengths_q], [int(x) for x in lengths_k]):
        if lq == 0 or lk == 0:
            continue
        off = lk - lq
        for_rows = 0
        if not causal and window <= 0:
            for_rows = lq * lk
        else:
            # per row i the allowed keys form one interval [lo_i, hi_i] of j
            for i in range(lq):
                d = i + off
                if causal:
                    hi_j = min(d, lk - 1)
                    lo_j = max(0, d - window + 1) if window > 0 else 0
                else:
                    hi_j = min(d + window - 1, lk - 1)
                    lo_j = max(0, d - window + 1)
                if hi_j >= lo_j:
                    for_rows += hi_j - lo_j + 1
        total += for_rows
    return total


def useful_flops(inp) -> tuple[float, float]:
    """(forward, backward) useful FLOPs: 2*A*(dqk+dv) and 2.5x that.

    A counts allowed pairs over all query heads. The backward figure counts
    five GEMMs (the recomputed S plus dV, dP, dQ, dK), the usual convention
    for attention backward throughput.
    """
    wl = inp.wl
    a = allowed_pairs(inp.lengths_q.tolist(), inp.lengths_k.tolist(), wl.causal, wl.window) * wl.h_q
    fwd = 2.0 * a * (wl.d_qk + wl.d_v)
    return fwd, 2.5 * fwd
