"""MXFP8 forward (gdpa_fwd_mxfp8): e4m3 codes with one E8M0 scale per 32
elements along each GEMM's contraction (q and k along the head dim, v along
the keys), applied by the block-scaled MMAs. Checked against the float64
oracle on the dequantised values at the FP8 tolerance: jagged query lengths
(empty, one row, ragged tails), key lengths that keep every key sequence on
a 32-key block boundary (the last sequence ragged), GQA/MQA, causal and
sliding-window masks, both supported head-dim pairs, head counts up to
64 (past what one shared-memory tile row of the scale rearrangement holds
at d_qk = 192, so it takes the heads in two chunks), and several
activations, softmax included. A key sequence that starts off a block is
reported through the device status word."""

import pytest
import torch

from generalized_attention_recsys_gb300 import _lib, inputs
from gpu_util import FP8_TOL, assert_close, ensure_built, ref_fwd, run_fwd, to_dev

pytestmark = pytest.mark.gpu

LQ = [200, 129, 1, 450, 0, 300, 77]
LK = [224, 128, 32, 448, 0, 320, 101]  # multiples of 32 but the last: every sequence starts on a block


@pytest.mark.parametrize("dims,h_q,h_kv,act,causal,window", [
    ((128, 128), 2, 2, "fast_gelu", False, -1),
    ((128, 128), 4, 1, "relu2", True, -1),
    ((128, 128), 4, 2, "softmax", True, 100),
    ((192, 128), 4, 2, "gelu", True, 130),
    ((192, 128), 4, 4, "identity", False, 60),
    ((192, 128), 4, 1, "silu", False, -1),
    ((192, 128), 2, 2, "softmax", False, -1),
    ((128, 128), 24, 3, "fast_gelu", True, -1),   # GQA 8 over an odd number of kv heads
    ((192, 128), 36, 18, "gelu", False, 200),     # many kv heads
    ((192, 128), 64, 1, "relu", True, -1),        # q heads past one staging tile row (two head chunks)
])
def test_mxfp8_forward_matches_oracle(dims, h_q, h_kv, act, causal, window):
    inp = inputs.custom(len(LQ), h_q, h_kv, dims[0], dims[1], LQ, LK, act, causal=causal, window=window,
                        dtype="mxe4m3", seed=31, with_dout=False)
    out, lse = run_fwd(inp)
    assert out.dtype == torch.bfloat16
    ref, ref_lse = ref_fwd(inp)
    assert_close(out, ref, FP8_TOL, f"out mxfp8 [{act}]")
    if act == "softmax":
        fin = torch.isfinite(ref_lse)
        assert (lse.cpu().double()[fin] - ref_lse[fin]).abs().max() < 2e-2


def test_mxfp8_fixed_length_workload_sample():
    # the benchmark's shapes, scaled down: fixed length, GQA 16/2, (192, 128), causal window
    wl = inputs.WORKLOADS["gqa_window_mxfp8"].with_(batch=2, max_q=1024, max_k=1024)
    inp = inputs.make_inputs(wl, seed=3, with_dout=False)
    assert inp.is_fixed_length()
    out, _ = run_fwd(inp)
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FP8_TOL, "out mxfp8 fixed length")


def test_mxfp8_key_sequence_off_a_block_is_reported():
    ensure_built()
    inp = inputs.custom(2, 2, 2, 128, 128, [64, 64], [40, 64], "gelu", dtype="mxe4m3", seed=32, with_dout=False)
    d = to_dev(inp)
    _lib.gdpa_fwd_mxfp8(d["q"], d["k"], d["v"], *d["mx"], d["cu_q"], d["cu_k"], 64, 64, "gelu", 0.1, batch=2)
    assert _lib.gdpa_get_status() == _lib.GDPA_ERR_INVALID
    # the device stays usable
    good = inputs.custom(2, 2, 2, 128, 128, [64, 64], [32, 64], "gelu", dtype="mxe4m3", seed=33, with_dout=False)
    out, _ = run_fwd(good)
    ref, _ = ref_fwd(good)
    assert_close(out, ref, FP8_TOL, "out mxfp8 after a reported call")
