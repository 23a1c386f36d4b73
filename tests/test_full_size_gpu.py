"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (the same C-ABI calls on the whole packed batch).

The oracle cannot redo whole workloads in test time, so it checks sampled
units: (sequence, head) pairs, or, for the 8192-token windowed workloads, row
slices. A causal, windowed slice of query rows [r0, r1) only sees keys
[r0 - W + 1, r1), and the oracle's bottom-right alignment maps the slice
(queries r0..r1-1, keys k0..r1-1) back onto the same positions, so the slice is
computed exactly as in the full problem. The sample and its seed are fixed.
"""

import random

import pytest
import torch

import oracle
from generalized_attention_recsys_gb300 import inputs
from gpu_util import FP8_TOL, FWD_TOL, GRAD_TOL, assert_close, run_bwd, run_fwd

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _units(inp, n_random, seed):
    lens = inp.lengths_q.tolist()
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    picks = {order[0], order[-1]}
    rng = random.Random(seed)
    while len(picks) < 2 + n_random and len(picks) < len(lens):
        picks.add(rng.randrange(len(lens)))
    return [(b, h) for b in sorted(picks) for h in range(inp.wl.h_q)]


def _unit_rows(inp, t, b, h):
    s, e = int(inp.cu_seqlens_q[b]), int(inp.cu_seqlens_q[b + 1])
    return t[s:e, h]


@pytest.mark.parametrize("name,n_random", [("jagged_self", 2), ("short_kv_cross", 2), ("dense_causal", 0)])
def test_forward_and_backward_full_size(name, n_random):
    wl = inputs.WORKLOADS[name]
    inp = inputs.make_inputs(wl, seed=0)
    units = _units(inp, n_random, seed=1)
    if name == "dense_causal":
        units = [(0, 0), (7, 3), (19, 5), (31, 7)]  # 4 of the 256 (sequence, head) units
    out, _ = run_fwd(inp)
    dq, dk, dv = run_bwd(inp)
    out, dq, dk, dv = (t.cpu() for t in (out, dq, dk, dv))
    q, k, v, do = inp.values("q"), inp.values("k"), inp.values("v"), inp.dout.double()
    for b, h in units:
        qs, qe = int(inp.cu_seqlens_q[b]), int(inp.cu_seqlens_q[b + 1])
        ks, ke = int(inp.cu_seqlens_k[b]), int(inp.cu_seqlens_k[b + 1])
        f = oracle.unit_fwd(q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], wl.act, wl.softmax_scale, wl.causal, wl.window)
        assert_close(out[qs:qe, h], f.out, FWD_TOL, f"{name} out unit {(b, h)}")
        r = oracle.unit_bwd(q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], do[qs:qe, h], wl.act, wl.softmax_scale,
                            wl.causal, wl.window)
        # MHA: the unit alone determines dK, dV of its kv head
        assert_close(dq[qs:qe, h], r.dq, GRAD_TOL, f"{name} dq unit {(b, h)}")
        assert_close(dk[ks:ke, h], r.dk, GRAD_TOL, f"{name} dk unit {(b, h)}")
        assert_close(dv[ks:ke, h], r.dv, GRAD_TOL, f"{name} dv unit {(b, h)}")


@pytest.mark.parametrize("name,tol", [("gqa_window_fp8", FP8_TOL), ("gqa_window_softmax", FWD_TOL)])
def test_windowed_gqa_forward_full_size(name, tol):
    wl = inputs.WORKLOADS[name]
    inp = inputs.make_inputs(wl, seed=0)
    out, lse = run_fwd(inp)
    out = out.cpu()
    q, k, v = inp.values("q"), inp.values("k"), inp.values("v")
    n, w, grp = wl.max_q, wl.window, wl.h_q // wl.h_kv
    picks = [(0, 0, 0), (5, 7, 1000), (15, 15, n - 128), (9, 2, 4096 + 77)]
    for b, h, r0 in picks:
        r1 = min(r0 + 128, n)
        k0 = max(0, r0 - w + 1)
        base = b * n
        g = h // grp
        f = oracle.unit_fwd(q[base + r0:base + r1, h], k[base + k0:base + r1, g], v[base + k0:base + r1, g],
                            wl.act, wl.softmax_scale, True, w)
        assert_close(out[base + r0:base + r1, h], f.out, tol, f"{name} rows {r0}:{r1} of unit {(b, h)}")
        if lse is not None:
            got = lse.cpu()[h, base + r0:base + r1].double()
            assert (got - f.lse).abs().max() < 1e-3
