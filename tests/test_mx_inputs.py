"""The MXFP8 input encoding (OCP Microscaling v1.0, as the seeded input
generator applies it) pinned to definitions outside this repository: the
E8M0 scale byte against torch's float8_e8m0fnu type, and e4m3 codes against
torch's float8_e4m3fn. The encoder must reproduce every block within half an
e4m3 step of its scale, saturate at 448 times the scale, and keep blocks
along the right axis (head dim for q and k, packed tokens for v)."""

import pytest
import torch

from generalized_attention_recsys_gb300 import inputs


def test_e8m0_scale_byte_is_a_power_of_two_with_bias_127():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    s = torch.arange(0, 255, dtype=torch.uint8)
    lib = s.view(torch.float8_e8m0fnu).double()
    codes = torch.ones(1, 1, 255 * 32).to(torch.float8_e4m3fn)
    ours = inputs.mx_values(codes, s.reshape(1, 1, 255), along_tokens=False)[0, 0, ::32]
    assert torch.equal(ours, lib)


def test_row_blocks_reproduce_values_within_half_a_step():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(50, 3, 192, generator=g) * torch.exp2(torch.randint(-6, 6, (50, 3, 1), generator=g).float())
    codes, sc = inputs.quantize_mx_rows(x)
    assert codes.dtype == torch.float8_e4m3fn and sc.shape == (50, 3, 6) and sc.dtype == torch.uint8
    v = inputs.mx_values(codes, sc, along_tokens=False)
    blk = x.reshape(50, 3, 6, 32)
    amax = blk.abs().amax(3)
    e = torch.floor(torch.log2(amax)) - 8
    assert torch.equal(sc.double(), e.double() + 127)
    # e4m3 has 3 mantissa bits: half a step of |x| / 2^e, below the saturation point 448
    step = torch.exp2(torch.floor(torch.log2(blk.abs().clamp_min(1e-30) / torch.exp2(e)[..., None])) - 3)
    err = (v.reshape(50, 3, 6, 32) - blk.double()).abs() / torch.exp2(e.double())[..., None]
    sat = blk.abs() / torch.exp2(e)[..., None] > 448
    assert (err[~sat] <= 0.5 * step.double()[~sat] * 1.000001 + 2.0 ** -10).all()
    assert torch.equal(codes.float().reshape(50, 3, 6, 32).abs()[sat], torch.full_like(blk[sat], 448.0))


def test_token_blocks_run_along_packed_tokens():
    x = torch.zeros(70, 2, 128)
    x[33, 1, 5] = 3.0  # block 1 (tokens 32..63) of head 1, column 5
    x[69, 0, 0] = -0.5  # the last, partial block
    codes, sc = inputs.quantize_mx_tokens(x)
    assert sc.shape == (3, 2, 128)
    assert int(sc[1, 1, 5]) == 127 + 1 - 8 and int(sc[2, 0, 0]) == 127 - 1 - 8
    assert int(sc[0, 0, 0]) == 0  # an all-zero block: the smallest scale
    v = inputs.mx_values(codes, sc, along_tokens=True)
    assert torch.equal(v, x.double())
