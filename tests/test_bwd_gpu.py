"""GPU backward parity: dQ, dK, dV from the CUDA path through the C-ABI against
the float64 oracle, per tensor, on seeded jagged inputs with ragged tails."""

import pytest
import torch

from generalized_attention_recsys_gb300 import inputs
from gpu_util import GRAD_TOL, assert_close, ref_bwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

RAGGED = [1, 127, 128, 129, 300, 0, 513, 64]
ALL_ACTS = ["identity", "gelu", "gelu_tanh", "fast_gelu", "relu", "relu2", "leaky_relu", "silu",
            "hardswish", "softmax", "fast_gelu_bf16", "fast_silu"]


def _check(inp, what=""):
    out = lse = None
    if inp.wl.act == "softmax":
        out, lse = run_fwd(inp)
    dq, dk, dv = run_bwd(inp, out, lse)
    rq, rk, rv = ref_bwd(inp)
    assert_close(dq, rq, GRAD_TOL, f"dq {what}")
    assert_close(dk, rk, GRAD_TOL, f"dk {what}")
    assert_close(dv, rv, GRAD_TOL, f"dv {what}")


def test_tiny_fixed_length():
    _check(inputs.make_inputs(inputs.WORKLOADS["tiny_fixed"], seed=0), "tiny")


@pytest.mark.parametrize("act", ALL_ACTS)
def test_every_activation_jagged(act):
    _check(inputs.custom(len(RAGGED), 2, 2, 128, 128, RAGGED, RAGGED, act, seed=11), act)


@pytest.mark.parametrize("causal,window", [(True, -1), (True, 37), (False, 37), (True, 200), (False, 300)])
@pytest.mark.parametrize("h_kv", [4, 2, 1])
def test_masks_and_heads(causal, window, h_kv):
    lq = [100, 257, 3, 0, 130, 129]
    lk = [300, 257, 0, 5, 64, 400]
    _check(inputs.custom(6, 4, h_kv, 128, 128, lq, lk, "silu", causal=causal, window=window, seed=12),
           f"causal={causal} window={window} h_kv={h_kv}")


@pytest.mark.parametrize("dims", [(64, 64), (96, 96), (192, 128)])
@pytest.mark.parametrize("act", ["gelu", "softmax"])
def test_head_dims(dims, act):
    lens = [130, 1, 256, 300, 77]
    _check(inputs.custom(5, 4, 2, dims[0], dims[1], lens, lens, act, causal=True, seed=13), f"dims={dims}")


@pytest.mark.parametrize("act", ALL_ACTS)
def test_fp16(act):
    lens = [129, 256, 7, 400]
    _check(inputs.custom(4, 2, 2, 128, 128, lens, lens, act, dtype="fp16", seed=14), f"fp16 {act}")


def test_empty_and_unseen_blocks_give_zero_gradients():
    # Lk = 0 for a sequence: its dQ is zero; Lq = 0: its dK/dV are zero
    inp = inputs.custom(3, 2, 2, 64, 64, [50, 0, 130], [0, 10, 140], "gelu", seed=15)
    dq, dk, dv = run_bwd(inp)
    rq, rk, rv = ref_bwd(inp)
    assert torch.count_nonzero(dq[:50]) == 0
    assert torch.count_nonzero(dk[:10]) == 0 and torch.count_nonzero(dv[:10]) == 0
    for g, r, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert_close(g, r, GRAD_TOL, n)


# (192, 128): dK and dQ come from two column-part work items ([0, 128) with
# dV, and [128, 192)); GQA and MQA groups, causal and sliding-window masks on
# ragged lengths that leave key blocks without queries and queries without keys.
@pytest.mark.parametrize("act,causal,window,h_kv,dtype", [
    ("silu", True, 37, 2, "bf16"),
    ("fast_gelu", True, -1, 1, "bf16"),
    ("relu2", False, 200, 4, "bf16"),
    ("hardswish", False, -1, 2, "fp16"),
    ("softmax", True, 130, 2, "bf16"),
])
def test_d192(act, causal, window, h_kv, dtype):
    lq = [100, 257, 3, 0, 130, 129, 400]
    lk = [300, 257, 0, 5, 64, 400, 129]
    _check(inputs.custom(len(lq), 4, h_kv, 192, 128, lq, lk, act, causal=causal, window=window, dtype=dtype, seed=16),
           f"d192 {act} causal={causal} window={window} h_kv={h_kv} {dtype}")
