"""The C-ABI library builds, loads and exports what include/gdpa.h declares.

CPU only: these calls return before touching a GPU (host-side validation and
workspace sizing).
"""

import ctypes
import os
import re

import pytest

from generalized_attention_recsys_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "gdpa.h")).read()
    return sorted(set(re.findall(r"\b(gdpa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert sorted(_lib.EXPORTS) == _declared()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_error_strings(lib):
    for s in range(6):
        assert _lib.gdpa_error_string(s)
    assert _lib.gdpa_error_string(5) == "device-side wait timed out"


def _shape(**kw):
    d = dict(batch=2, total_q=256, total_k=256, h_q=4, h_kv=2, d_qk=128, d_v=128, dtype=0)
    d.update(kw)
    return _lib.GdpaShape(**d)


def test_workspace_bytes(lib):
    s = _shape()
    fwd = _lib.gdpa_workspace_bytes(s, 128, 128, False)
    bwd = _lib.gdpa_workspace_bytes(s, 128, 128, True)
    assert fwd >= 16 and fwd % 256 == 0
    # backward holds an fp32 dQ accumulator
    assert bwd >= 256 * 4 * 128 * 4
    assert _lib.gdpa_workspace_bytes(_shape(h_q=3), 128, 128, False) == 0
    # sequences of 2^30 tokens or more are refused (mask arithmetic stays within int)
    assert _lib.gdpa_workspace_bytes(s, 1 << 30, 128, False) == 0
    assert _lib.gdpa_workspace_bytes(s, 128, 1 << 30, False) == 0
    assert _lib.gdpa_workspace_bytes(s, (1 << 30) - 1, 128, False) > 0
    # the MXFP8 forward adds its scale atoms (512 bytes each): per work item (at most
    # total_q / 128 + batch + 1) and head, and per 32-key group and kv head, for q and k one
    # atom per four 32-element blocks of d_qk, for v one
    for d_qk, nqb in ((128, 1), (192, 2)):
        sm = _shape(d_qk=d_qk, dtype=2)
        r256 = lambda x: (x + 255) // 256 * 256
        atoms = r256((256 // 128 + 2 + 1) * 4 * nqb * 512) + r256(8 * 2 * nqb * 512) + r256(8 * 2 * 512)
        assert _lib.gdpa_workspace_bytes(sm, 128, 128, 3) - _lib.gdpa_workspace_bytes(sm, 128, 128, 0) == atoms
    # the deterministic backward adds one fp32 dQ slice per 128-key block of max_seqlen_k
    for max_k, nkv in ((128, 1), (129, 2), (300, 3)):
        det = _lib.gdpa_workspace_bytes(s, 128, max_k, 2)
        assert det - _lib.gdpa_workspace_bytes(s, 128, max_k, 1) == nkv * 256 * 4 * 128 * 4


@pytest.mark.parametrize("kw,status", [
    (dict(h_q=3, h_kv=2), _lib.GDPA_ERR_INVALID),
    (dict(h_kv=0), _lib.GDPA_ERR_INVALID),
    (dict(batch=-1), _lib.GDPA_ERR_INVALID),
    (dict(dtype=7), _lib.GDPA_ERR_INVALID),
    (dict(d_qk=80, d_v=80), _lib.GDPA_ERR_UNSUPPORTED),
    (dict(d_qk=128, d_v=64), _lib.GDPA_ERR_UNSUPPORTED),
])
def test_host_validation_rejects_before_launch(lib, kw, status):
    s = _shape(**kw)
    st = lib.gdpa_fwd(ctypes.byref(s), None, None, None, None, None, 128, 128, 1, 0.1, 0, -1,
                      None, None, None, None, 0, None)
    assert st == status


def test_bad_activation_and_fp8_backward(lib):
    s = _shape()
    assert max(_lib.ACTS.values()) == 11 and sorted(_lib.ACTS.values()) == list(range(12))
    for bad in (-1, 12, 42):  # just outside the enum on both sides, and far outside
        assert lib.gdpa_fwd(ctypes.byref(s), None, None, None, None, None, 128, 128, bad, 0.1, 0, -1,
                            None, None, None, None, 0, None) == _lib.GDPA_ERR_INVALID
        assert lib.gdpa_bwd(ctypes.byref(s), None, None, None, None, None, 128, 128, bad, 0.1, 0, -1,
                            None, None, None, None, None, None, 0, None, 0, None) == _lib.GDPA_ERR_INVALID
    s8 = _shape(dtype=2)
    assert lib.gdpa_bwd(ctypes.byref(s8), None, None, None, None, None, 128, 128, 1, 0.1, 0, -1,
                        None, None, None, None, None, None, 0, None, 0, None) == _lib.GDPA_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers_rejected(lib):
    s = _shape()
    buf = ctypes.create_string_buffer(64)
    base = ctypes.addressof(buf)
    aligned = (base + 15) & ~15
    # q missing
    assert lib.gdpa_fwd(ctypes.byref(s), None, aligned, aligned, None, None, 128, 128, 1, 0.1, 0, -1,
                        None, aligned, None, aligned, 1 << 20, None) == _lib.GDPA_ERR_INVALID
    # q misaligned
    assert lib.gdpa_fwd(ctypes.byref(s), aligned + 2, aligned, aligned, None, None, 128, 128, 1, 0.1, 0,
                        -1, None, aligned, None, aligned, 1 << 20, None) == _lib.GDPA_ERR_INVALID
    # softmax without lse
    assert lib.gdpa_fwd(ctypes.byref(s), aligned, aligned, aligned, None, None, 128, 128, 9, 0.1, 0, -1,
                        None, aligned, None, aligned, 1 << 20, None) == _lib.GDPA_ERR_INVALID
    # workspace too small
    assert lib.gdpa_fwd(ctypes.byref(s), aligned, aligned, aligned, None, None, 128, 128, 1, 0.1, 0, -1,
                        None, aligned, None, aligned, 8, None) == _lib.GDPA_ERR_WORKSPACE
    # fixed length with inconsistent totals
    s2 = _shape(total_q=250)
    assert lib.gdpa_fwd(ctypes.byref(s2), aligned, aligned, aligned, None, None, 128, 128, 1, 0.1, 0, -1,
                        None, aligned, None, aligned, 1 << 20, None) == _lib.GDPA_ERR_INVALID


def test_noalloc_forward_rejects_problems_beyond_its_scratch(lib):
    # the work list of 70,000 one-token sequences needs more than the fixed scratch
    s = _shape(batch=70000, total_q=70000, total_k=70000)
    assert _lib.gdpa_workspace_bytes(s, 1, 1, False) > _lib.NOALLOC_SCRATCH_BYTES
    st = lib.gdpa_fwd_noalloc(ctypes.byref(s), None, None, None, None, None, 1, 1, 1, 0.1, 0, -1, None, None,
                              None, None)
    assert st == _lib.GDPA_ERR_SCRATCH_LIMIT
    assert "scratch" in _lib.gdpa_error_string(st)
