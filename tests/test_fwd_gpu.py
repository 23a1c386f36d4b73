"""GPU forward parity: the CUDA path through the C-ABI against the float64 oracle,
element by element, on seeded inputs that span several tiles and ragged tails."""

import pytest
import torch

from generalized_attention_recsys_gb300 import inputs
from gpu_util import FP8_TOL, FWD_TOL, assert_close, ref_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

RAGGED = [1, 127, 128, 129, 300, 0, 513, 64]
ALL_ACTS = ["identity", "gelu", "gelu_tanh", "fast_gelu", "relu", "relu2", "leaky_relu", "silu",
            "hardswish", "softmax", "fast_gelu_bf16", "fast_silu"]


def test_tiny_fixed_length():
    inp = inputs.make_inputs(inputs.WORKLOADS["tiny_fixed"], seed=0)
    out, _ = run_fwd(inp)
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FWD_TOL, "out")


@pytest.mark.parametrize("act", ALL_ACTS)
def test_every_activation_jagged(act):
    inp = inputs.custom(len(RAGGED), 2, 2, 128, 128, RAGGED, RAGGED, act, seed=1)
    out, lse = run_fwd(inp)
    ref, ref_lse = ref_fwd(inp)
    assert_close(out, ref, FWD_TOL, f"out[{act}]")
    if act == "softmax":
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse.cpu()), fin)
        assert (lse.cpu().double()[fin] - ref_lse[fin]).abs().max() < 1e-3


@pytest.mark.parametrize("causal,window", [(True, -1), (True, 37), (False, 37), (True, 200), (False, 300)])
@pytest.mark.parametrize("h_kv", [4, 2, 1])
def test_masks_and_heads(causal, window, h_kv):
    lq = [100, 257, 3, 0, 130, 129]
    lk = [300, 257, 0, 5, 64, 400]
    inp = inputs.custom(6, 4, h_kv, 128, 128, lq, lk, "silu", causal=causal, window=window, seed=2)
    out, _ = run_fwd(inp)
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FWD_TOL, f"out causal={causal} window={window} h_kv={h_kv}")


@pytest.mark.parametrize("causal", [True, False])
def test_window_beyond_any_length_is_no_window(causal):
    # a window at the top of the int range must select the same keys as no window
    # (the library clamps it below 2^30, so the mask arithmetic cannot overflow)
    lq, lk = [100, 257, 3, 130], [300, 257, 9, 64]
    wide = inputs.custom(4, 2, 1, 128, 128, lq, lk, "gelu", causal=causal, window=2**31 - 1, seed=7)
    none = inputs.custom(4, 2, 1, 128, 128, lq, lk, "gelu", causal=causal, window=-1, seed=7)
    out_wide, _ = run_fwd(wide)
    out_none, _ = run_fwd(none)
    assert torch.equal(out_wide, out_none)
    ref, _ = ref_fwd(none)
    assert_close(out_wide, ref, FWD_TOL, f"out causal={causal} window=2^31-1")
    dq_w, dk_w, dv_w = run_bwd(wide)
    dq_n, dk_n, dv_n = run_bwd(none)
    assert torch.equal(dk_w, dk_n) and torch.equal(dv_w, dv_n)
    assert torch.allclose(dq_w.float(), dq_n.float(), rtol=0, atol=1e-2 * dq_n.float().abs().max().item())


@pytest.mark.parametrize("dims", [(64, 64), (96, 96), (192, 128)])
@pytest.mark.parametrize("act", ["gelu", "softmax"])
def test_head_dims(dims, act):
    inp = inputs.custom(5, 4, 2, dims[0], dims[1], [130, 1, 256, 300, 77], [130, 1, 256, 300, 77], act,
                        causal=True, seed=3)
    out, _ = run_fwd(inp)
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FWD_TOL, f"out dims={dims}")


@pytest.mark.parametrize("act", ["gelu_tanh", "softmax", "relu2"])
def test_fp16(act):
    inp = inputs.custom(4, 2, 2, 128, 128, [129, 256, 7, 400], [129, 256, 7, 400], act, dtype="fp16", seed=4)
    out, _ = run_fwd(inp)
    assert out.dtype == torch.float16
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FWD_TOL, "out fp16")


@pytest.mark.parametrize("act", ALL_ACTS)
def test_every_activation_fp16(act):
    # every fp16 kernel configuration: four activation groups (GELU, tanh GELU, SiLU), two groups
    # (the other elementwise activations) and the softmax kernel, each compiled for its own set
    inp = inputs.custom(len(RAGGED), 2, 1, 128, 128, RAGGED, RAGGED, act, dtype="fp16", seed=6, with_dout=False)
    out, lse = run_fwd(inp)
    assert out.dtype == torch.float16
    ref, ref_lse = ref_fwd(inp)
    assert_close(out, ref, FWD_TOL, f"out fp16 [{act}]")
    if act == "softmax":
        fin = torch.isfinite(ref_lse)
        assert (lse.cpu().double()[fin] - ref_lse[fin]).abs().max() < 1e-3


@pytest.mark.parametrize("act", ALL_ACTS)
def test_every_activation_fp8(act):
    # e4m3 runs every activation with two groups: the elementwise kernel and the softmax kernel
    lens = [200, 129, 1, 450, 0, 300]
    inp = inputs.custom(len(lens), 2, 2, 128, 128, lens, lens, act, dtype="e4m3", seed=7, with_dout=False)
    out, _ = run_fwd(inp)
    assert out.dtype == torch.bfloat16
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FP8_TOL, f"out e4m3 [{act}]")


@pytest.mark.parametrize("dims,h_kv,causal,window", [((128, 128), 4, False, -1), ((192, 128), 1, True, 100),
                                                    ((64, 64), 2, True, -1)])
def test_fp8(dims, h_kv, causal, window):
    lens = [200, 129, 1, 450]
    inp = inputs.custom(4, 4, h_kv, dims[0], dims[1], lens, lens, "fast_gelu", causal=causal, window=window,
                        dtype="e4m3", seed=5, with_dout=False)
    out, _ = run_fwd(inp)
    assert out.dtype == torch.bfloat16
    ref, _ = ref_fwd(inp)
    assert_close(out, ref, FP8_TOL, "out e4m3")


def test_zero_keys_give_zero_rows_and_empty_batch():
    inp = inputs.custom(3, 2, 2, 64, 64, [50, 0, 130], [0, 10, 0], "gelu", seed=6)
    out, _ = run_fwd(inp)
    assert torch.count_nonzero(out) == 0
    inp = inputs.custom(2, 2, 1, 64, 64, [0, 0], [0, 0], "gelu", seed=6)
    out, _ = run_fwd(inp)
    assert out.numel() == 0


@pytest.mark.parametrize("act", ["gelu", "relu2", "softmax"])
def test_repeat_calls_are_bitwise_stable(act):
    # four activation groups (gelu) and two groups with the staged epilogue (relu2, softmax)
    inp = inputs.custom(len(RAGGED), 2, 2, 128, 128, RAGGED, RAGGED, act, seed=7)
    a, la = run_fwd(inp)
    b, lb = run_fwd(inp)
    assert torch.equal(a, b)
    if act == "softmax":
        assert torch.equal(la, lb)
