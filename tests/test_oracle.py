"""Pins for the float64 oracle, each against something other than the oracle itself.

CPU only. The pins are: textbook constants and hand-worked examples
(tests/golden), PyTorch library routines for the activations and for textbook
softmax attention, closed forms (associativity), invariants (jagged vs
per-sequence, GQA vs repeated heads, window >= length, fully masked rows),
exact rational brute force on tiny inputs, autograd of the forward
definition, and central finite differences.
"""

import json
import math
import os
import random
from fractions import Fraction

import pytest
import torch
import torch.nn.functional as F

from oracle import (ACTIVATIONS, LEAKY_SLOPE, act_fwd, act_grad, allowed_mask, gdpa_bwd,
                    gdpa_fwd, unit_bwd, unit_fwd)
from generalized_attention_recsys_gb300 import flops, inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ELEMENTWISE = [a for a in ACTIVATIONS if a != "softmax"]
pytestmark = pytest.mark.filterwarnings("ignore")


def _t(x):
    return torch.tensor(x, dtype=torch.float64)


# ------------------------------------------------------------ golden fixtures

def test_golden_hand_example_relu_causal():
    g = json.load(open(os.path.join(GOLDEN, "hand_relu_causal.json")))
    q, k, v, do = (_t(g[n]) for n in ("q", "k", "v", "dout"))
    f = unit_fwd(q, k, v, g["act"], g["scale"], g["causal"], g["window"])
    assert torch.equal(f.out, _t(g["out"]))
    r = unit_bwd(q, k, v, do, g["act"], g["scale"], g["causal"], g["window"])
    assert torch.equal(r.dq, _t(g["dq"]))
    assert torch.equal(r.dk, _t(g["dk"]))
    assert torch.equal(r.dv, _t(g["dv"]))


def test_golden_scalar_activations():
    g = json.load(open(os.path.join(GOLDEN, "scalar_activations.json")))
    for c in g["cases"]:
        one = _t([[1.0]])
        f = unit_fwd(_t([[c["z"]]]), one, one, c["act"], 1.0, False, -1)
        assert abs(float(f.out) - c["value"]) < 1e-12, c


# ------------------------------------------------------------ activations vs library

_LIB = {
    "identity": lambda z: z,
    "gelu": lambda z: F.gelu(z, approximate="none"),
    "gelu_tanh": lambda z: F.gelu(z, approximate="tanh"),
    "fast_gelu": lambda z: F.gelu(z, approximate="tanh"),
    "relu": F.relu,
    "relu2": lambda z: F.relu(z) ** 2,
    "leaky_relu": lambda z: F.leaky_relu(z, LEAKY_SLOPE),
    "silu": F.silu,
    "hardswish": F.hardswish,
    "fast_gelu_bf16": lambda z: F.gelu(z, approximate="tanh"),
    "fast_silu": F.silu,
}


@pytest.mark.parametrize("act", ELEMENTWISE)
def test_activation_matches_torch(act):
    z = torch.linspace(-8, 8, 4001, dtype=torch.float64)
    z = torch.cat([z, _t([0.0, -3.0, 3.0, 1e-9, -1e-9])])
    assert torch.allclose(act_fwd(act, z), _LIB[act](z), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("act", ELEMENTWISE)
def test_activation_derivative_matches_autograd(act):
    # includes the kinks 0 and +-3, where PyTorch's backward conventions decide
    z = torch.cat([torch.linspace(-8, 8, 4001, dtype=torch.float64), _t([0.0, -3.0, 3.0])])
    z.requires_grad_(True)
    (g,) = torch.autograd.grad(_LIB[act](z).sum(), z)
    assert torch.allclose(act_grad(act, z.detach()), g, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ closed forms and invariants

def _rand(*shape, seed=0, lo=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float64)
    return x.abs() + lo if lo is not None else x


def _packed(lengths, h, d, seed):
    t = sum(lengths)
    return _rand(t, h, d, seed=seed)


def _cu(lengths):
    return torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()), dtype=torch.int32)


def test_identity_equals_associativity():
    lq = [5, 0, 9, 3]
    q = _packed(lq, 4, 6, 1)
    k = _packed(lq, 2, 6, 2)
    v = _packed(lq, 2, 5, 3)
    cu = _cu(lq)
    scale = 0.37
    out, _ = gdpa_fwd(q, k, v, cu, cu, 4, 9, 9, "identity", scale)
    for b in range(4):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        for h in range(4):
            g = h // 2
            ref = scale * q[s0:s1, h] @ (k[s0:s1, g].T @ v[s0:s1, g])
            assert torch.allclose(out[s0:s1, h], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act,expect", [("relu", "identity"), ("leaky_relu", "identity"),
                                         ("hardswish", None), ("relu2", "square")])
def test_relu_family_on_positive_scores(act, expect):
    q = _rand(7, 1, 4, seed=4, lo=0.1)
    k = _rand(6, 1, 4, seed=5, lo=0.1)
    v = _rand(6, 1, 3, seed=6)
    cu_q, cu_k = _cu([7]), _cu([6])
    out, _ = gdpa_fwd(q, k, v, cu_q, cu_k, 1, 7, 6, act, 1.0)
    z = q[:, 0] @ k[:, 0].T
    if expect == "identity":
        ref = z @ v[:, 0]
    elif expect == "square":
        ref = (z * z) @ v[:, 0]
    else:
        # hardswish on z >= 3 is the identity
        q3 = q * 3.0
        out, _ = gdpa_fwd(q3, k * 3.0, v, cu_q, cu_k, 1, 7, 6, act, 1.0)
        z3 = q3[:, 0] @ (k[:, 0] * 3.0).T
        assert (z3 > 3).all()
        ref = z3 @ v[:, 0]
    assert torch.allclose(out[:, 0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 3), (False, 2)])
def test_softmax_matches_textbook_attention(causal, window):
    lq, lk = 6, 8
    q, k, v, do = _rand(lq, 4, seed=7), _rand(lk, 4, seed=8), _rand(lk, 3, seed=9), _rand(lq, 3, seed=10)
    scale = 0.5
    m = allowed_mask(lq, lk, causal, window)
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, k, v))
    logits = (scale * qr @ kr.T).masked_fill(~m, -math.inf)
    ref = torch.softmax(logits, dim=-1) @ vr
    lse_ref = torch.logsumexp(logits, dim=-1)
    f = unit_fwd(q, k, v, "softmax", scale, causal, window)
    assert torch.allclose(f.out, ref.detach(), rtol=1e-12, atol=1e-12)
    assert torch.allclose(f.lse, lse_ref.detach(), rtol=1e-12, atol=1e-12)
    gq, gk, gv = torch.autograd.grad(ref, (qr, kr, vr), do)
    r = unit_bwd(q, k, v, do, "softmax", scale, causal, window)
    for a, b in ((r.dq, gq), (r.dk, gk), (r.dv, gv)):
        assert torch.allclose(a, b, rtol=1e-10, atol=1e-12)


def test_masked_rows_are_zero():
    # causal with Lq > Lk: query rows i < Lq - Lk see no key at all
    lq, lk = 7, 3
    q, k, v, do = _rand(lq, 4, seed=11), _rand(lk, 4, seed=12), _rand(lk, 2, seed=13), _rand(lq, 2, seed=14)
    for act in ("gelu", "silu", "softmax", "identity"):
        f = unit_fwd(q, k, v, act, 0.3, True, -1)
        assert torch.count_nonzero(f.out[: lq - lk]) == 0
        assert torch.count_nonzero(f.out[lq - lk:]) > 0
        if act == "softmax":
            assert torch.isneginf(f.lse[: lq - lk]).all()
        r = unit_bwd(q, k, v, do, act, 0.3, True, -1)
        assert torch.count_nonzero(r.dq[: lq - lk]) == 0


def test_jagged_equals_per_sequence_dense():
    lens = [3, 130, 1, 0, 64]
    q = _packed(lens, 2, 8, 20)
    k = _packed(lens, 2, 8, 21)
    v = _packed(lens, 2, 8, 22)
    do = _packed(lens, 2, 8, 23)
    cu = _cu(lens)
    out, _ = gdpa_fwd(q, k, v, cu, cu, 5, 130, 130, "gelu", 0.25, causal=True)
    dq, dk, dv = gdpa_bwd(q, k, v, do, cu, cu, 5, 130, 130, "gelu", 0.25, causal=True)
    for b, n in enumerate(lens):
        s = slice(int(cu[b]), int(cu[b + 1]))
        o1, _ = gdpa_fwd(q[s], k[s], v[s], None, None, 1, n, n, "gelu", 0.25, causal=True)
        g1 = gdpa_bwd(q[s], k[s], v[s], do[s], None, None, 1, n, n, "gelu", 0.25, causal=True)
        assert torch.equal(out[s], o1)
        for a, b_ in zip((dq[s], dk[s], dv[s]), g1):
            assert torch.equal(a, b_)


def test_gqa_equals_mha_with_repeated_kv_heads():
    lens = [9, 4]
    hq, hkv = 6, 2
    q = _packed(lens, hq, 5, 30)
    k = _packed(lens, hkv, 5, 31)
    v = _packed(lens, hkv, 7, 32)
    do = _packed(lens, hq, 7, 33)
    cu = _cu(lens)
    args = (cu, cu, 2, 9, 9, "silu", 0.4)
    out, _ = gdpa_fwd(q, k, v, *args, causal=True, window=3)
    dq, dk, dv = gdpa_bwd(q, k, v, do, *args, causal=True, window=3)
    kr = k.repeat_interleave(hq // hkv, dim=1)
    vr = v.repeat_interleave(hq // hkv, dim=1)
    out_r, _ = gdpa_fwd(q, kr, vr, *args, causal=True, window=3)
    dq_r, dk_r, dv_r = gdpa_bwd(q, kr, vr, do, *args, causal=True, window=3)
    assert torch.allclose(out, out_r, rtol=0, atol=1e-13)
    assert torch.allclose(dq, dq_r, rtol=0, atol=1e-13)
    assert torch.allclose(dk, dk_r.view(-1, hkv, hq // hkv, 5).sum(2), rtol=0, atol=1e-12)
    assert torch.allclose(dv, dv_r.view(-1, hkv, hq // hkv, 7).sum(2), rtol=0, atol=1e-12)


def test_window_at_least_length_is_no_window():
    lq, lk = 11, 11
    q, k, v = _rand(lq, 4, seed=40), _rand(lk, 4, seed=41), _rand(lk, 4, seed=42)
    for causal in (True, False):
        a = unit_fwd(q, k, v, "gelu_tanh", 0.5, causal, -1).out
        b = unit_fwd(q, k, v, "gelu_tanh", 0.5, causal, lk + 2).out
        assert torch.equal(a, b)
    # and a real window changes the answer
    c = unit_fwd(q, k, v, "gelu_tanh", 0.5, True, 4).out
    assert not torch.allclose(c, unit_fwd(q, k, v, "gelu_tanh", 0.5, True, -1).out)


def test_mask_shapes_by_counting():
    # causal square: lower triangle; window W causal: at most W per row, diagonal included
    m = allowed_mask(5, 5, True, -1)
    assert int(m.sum()) == 15 and bool(m.diagonal().all()) and not bool(m[0, 1])
    m = allowed_mask(6, 6, True, 2)
    assert m.sum(1).tolist() == [1, 2, 2, 2, 2, 2]
    m = allowed_mask(3, 5, True, -1)   # bottom-right: last query sees every key
    assert m.sum(1).tolist() == [3, 4, 5]
    m = allowed_mask(4, 4, False, 2)   # |i - j| < 2
    assert m.sum(1).tolist() == [2, 3, 3, 2]


# ------------------------------------------------------------ exact brute force

def _frac_act(name, z: Fraction) -> Fraction:
    if name == "identity":
        return z
    if name == "relu":
        return z if z > 0 else Fraction(0)
    if name == "relu2":
        return z * z if z > 0 else Fraction(0)
    if name == "leaky_relu":
        return z if z > 0 else Fraction(1, 100) * z
    if name == "hardswish":
        return z * min(max(z + 3, Fraction(0)), Fraction(6)) / 6
    raise ValueError(name)


def _frac_dact(name, z: Fraction) -> Fraction:
    if name == "identity":
        return Fraction(1)
    if name == "relu":
        return Fraction(1) if z > 0 else Fraction(0)
    if name == "relu2":
        return 2 * z if z > 0 else Fraction(0)
    if name == "leaky_relu":
        return Fraction(1) if z > 0 else Fraction(1, 100)
    if name == "hardswish":
        if z <= -3:
            return Fraction(0)
        return z / 3 + Fraction(1, 2) if z < 3 else Fraction(1)
    raise ValueError(name)


def _allowed_py(i, j, lq, lk, causal, window):
    d = i + lk - lq - j
    if causal:
        return d >= 0 and (window <= 0 or d < window)
    return window <= 0 or abs(d) < window


def _brute(lens_q, lens_k, hq, hkv, dqk, dv, act, scale, causal, window, seed):
    """Exact rational GDPA forward and backward with plain Python loops."""
    rng = random.Random(seed)
    tq, tk = sum(lens_q), sum(lens_k)

    def mat(t, h, d):
        return [[[Fraction(rng.randint(-4, 4), 4) for _ in range(d)] for _ in range(h)] for _ in range(t)]

    q, k, v, do = mat(tq, hq, dqk), mat(tk, hkv, dqk), mat(tk, hkv, dv), mat(tq, hq, dv)
    out = [[[Fraction(0)] * dv for _ in range(hq)] for _ in range(tq)]
    dq = [[[Fraction(0)] * dqk for _ in range(hq)] for _ in range(tq)]
    dk = [[[Fraction(0)] * dqk for _ in range(hkv)] for _ in range(tk)]
    dvv = [[[Fraction(0)] * dv for _ in range(hkv)] for _ in range(tk)]
    oq = ok = 0
    for lq, lk in zip(lens_q, lens_k):
        for h in range(hq):
            g = h // (hq // hkv)
            for i in range(lq):
                for j in range(lk):
                    if not _allowed_py(i, j, lq, lk, causal, window):
                        continue
                    z = scale * sum(q[oq + i][h][c] * k[ok + j][g][c] for c in range(dqk))
                    p = _frac_act(act, z)
                    dp = sum(do[oq + i][h][c] * v[ok + j][g][c] for c in range(dv))
                    ds = scale * dp * _frac_dact(act, z)
                    for c in range(dv):
                        out[oq + i][h][c] += p * v[ok + j][g][c]
                        dvv[ok + j][g][c] += p * do[oq + i][h][c]
                    for c in range(dqk):
                        dq[oq + i][h][c] += ds * k[ok + j][g][c]
                        dk[ok + j][g][c] += ds * q[oq + i][h][c]
        oq += lq
        ok += lk
    f = lambda x: torch.tensor([[[float(e) for e in r] for r in hh] for hh in x], dtype=torch.float64)
    return [f(x) for x in (q, k, v, do, out, dq, dk, dvv)]


@pytest.mark.parametrize("act", ["identity", "relu", "relu2", "leaky_relu", "hardswish"])
@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 2), (False, 2)])
def test_exact_rational_brute_force(act, causal, window):
    lens_q, lens_k = [3, 0, 4], [4, 2, 4]
    scale = Fraction(1, 2)
    # a fixed seed per case (string hashing is salted per process, so no hash())
    seed = 100 * ["identity", "relu", "relu2", "leaky_relu", "hardswish"].index(act) + 10 * int(causal) + max(window, 0)
    q, k, v, do, out_e, dq_e, dk_e, dv_e = _brute(lens_q, lens_k, 4, 2, 3, 2, act, scale, causal, window, seed=seed)
    cu_q, cu_k = _cu(lens_q), _cu(lens_k)
    out, _ = gdpa_fwd(q, k, v, cu_q, cu_k, 3, 4, 4, act, float(scale), causal, window)
    dq, dk, dv = gdpa_bwd(q, k, v, do, cu_q, cu_k, 3, 4, 4, act, float(scale), causal, window)
    for a, b in ((out, out_e), (dq, dq_e), (dk, dk_e), (dv, dv_e)):
        assert torch.allclose(a, b, rtol=0, atol=1e-12)


# ------------------------------------------------------------ gradients

@pytest.mark.parametrize("act", ACTIVATIONS)
def test_backward_matches_autograd_of_forward(act):
    lq, lk = 5, 7
    q, k, v, do = _rand(lq, 3, seed=50), _rand(lk, 3, seed=51), _rand(lk, 4, seed=52), _rand(lq, 4, seed=53)
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, k, v))
    f = unit_fwd(qr, kr, vr, act, 0.7, True, 4)
    gq, gk, gv = torch.autograd.grad(f.out, (qr, kr, vr), do)
    r = unit_bwd(q, k, v, do, act, 0.7, True, 4)
    for a, b in ((r.dq, gq), (r.dk, gk), (r.dv, gv)):
        assert torch.allclose(a, b, rtol=1e-10, atol=1e-12)


_KINKS = {"relu": [0.0], "relu2": [0.0], "leaky_relu": [0.0], "hardswish": [-3.0, 3.0]}


@pytest.mark.parametrize("act", ACTIVATIONS)
def test_gradients_match_central_differences(act):
    lq, lk, scale = 4, 5, 0.6
    for seed in range(60, 200):
        q, k, v, do = _rand(lq, 3, seed=seed), _rand(lk, 3, seed=seed + 1), _rand(lk, 2, seed=seed + 2), \
            _rand(lq, 2, seed=seed + 3)
        z = scale * q @ k.T
        if all((z - c).abs().min() > 1e-3 for c in _KINKS.get(act, [])):
            break
    r = unit_bwd(q, k, v, do, act, scale, True, 3)

    def loss(args):
        return float((unit_fwd(args["q"], args["k"], args["v"], act, scale, True, 3).out * do).sum())

    eps = 1e-6
    base = {"q": q, "k": k, "v": v}
    for name, t, g in (("q", q, r.dq), ("k", k, r.dk), ("v", v, r.dv)):
        num = torch.zeros_like(t)
        for idx in range(t.numel()):
            tp, tm = t.clone(), t.clone()
            tp.view(-1)[idx] += eps
            tm.view(-1)[idx] -= eps
            num.view(-1)[idx] = (loss({**base, name: tp}) - loss({**base, name: tm})) / (2 * eps)
        rel = (num - g).abs().max() / max(g.abs().max(), 1e-30)
        assert rel <= 1e-6, (act, name, float(rel))


# ------------------------------------------------------------ host helpers pinned to the oracle mask

@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 5), (False, 3)])
def test_allowed_pairs_counts_mask(causal, window):
    lens_q, lens_k = [7, 0, 12, 3, 30], [9, 4, 12, 1, 17]
    ref = sum(int(allowed_mask(a, b, causal, window).sum()) for a, b in zip(lens_q, lens_k))
    assert flops.allowed_pairs(lens_q, lens_k, causal, window) == ref


def test_e4m3_quantiser_roundtrip():
    x = _rand(4096, seed=70).float()
    codes, s = inputs.quantize_e4m3(x)
    back = codes.float() * s
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 for normals, absolute <= 2^-10 * s below 2^-6
    err = (back - x).abs()
    bound = torch.maximum(x.abs() * 2.0 ** -4, torch.full_like(x, s * 2.0 ** -10))
    assert bool((err <= bound).all())
    assert float(codes.float().abs().max()) == 448.0


def test_workload_recipe_is_deterministic_and_matches_sizes():
    a = inputs.make_inputs(inputs.WORKLOADS["tiny_fixed"], seed=0)
    b = inputs.make_inputs(inputs.WORKLOADS["tiny_fixed"], seed=0)
    assert torch.equal(a.q, b.q) and torch.equal(a.dout, b.dout)
    j = inputs.WORKLOADS["jagged_self"]
    g = torch.Generator().manual_seed(0)
    lens = torch.randint(1, 2049, (64,), generator=g)
    assert int(lens.sum()) == 62386
    fw, bw = flops.useful_flops(a)
    assert fw == 2 * 2 * 2 * 128 * 128 * 128 and bw == 2.5 * fw
    assert j.softmax_scale == 1 / math.sqrt(128)
