"""gdpa_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers own no device allocator of their own (a plugin inside a host
framework whose memory is fully managed by that framework, or a deployment
that forbids allocations after start-up). gdpa_fwd_noalloc serves them by
keeping the forward's scratch (the work list) in a fixed array inside the
library. This test calls it through the C ABI twice in a row, on two
different problems, and checks each result against the workspace-taking
gdpa_fwd and against the float64 oracle, within the forward tolerance the
other tests use. It lives in a file that pytest collects last so that a
stop-at-first-failure run has already run every other test.
"""

import pytest
import torch

from generalized_attention_recsys_gb300 import _lib, inputs
from gpu_util import FWD_TOL, assert_close, ensure_built, max_lens, ref_fwd, to_dev

pytestmark = pytest.mark.gpu


def _both(inp):
    wl = inp.wl
    d = to_dev(inp)
    mq, mk = max_lens(inp)
    args = (d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], mq, mk, wl.act, wl.softmax_scale, wl.causal, wl.window)
    ref, _ = _lib.gdpa_fwd(*args, descale_qkv=d["descale"], batch=wl.batch)
    out = torch.full_like(ref, float("nan"))
    got, _ = _lib.gdpa_fwd_noalloc(*args, descale_qkv=d["descale"], out=out, batch=wl.batch)
    assert _lib.gdpa_get_status() == 0
    return got, ref


def test_noalloc_forward_matches_gdpa_fwd_on_two_calls_in_a_row():
    ensure_built()
    lens_a = [1, 127, 128, 129, 300, 0, 513, 64]
    first = inputs.custom(len(lens_a), 4, 2, 128, 128, lens_a, lens_a, "gelu", causal=True, seed=21)
    lens_b = [700, 5, 256]
    second = inputs.custom(len(lens_b), 2, 1, 64, 64, lens_b, [300, 5, 900], "silu", window=100, seed=22)
    for inp in (first, second):
        got, ref = _both(inp)
        assert_close(got, ref, FWD_TOL, "gdpa_fwd_noalloc vs gdpa_fwd")
        oracle_out, _ = ref_fwd(inp)
        assert_close(got, oracle_out, FWD_TOL, "gdpa_fwd_noalloc vs the oracle")
