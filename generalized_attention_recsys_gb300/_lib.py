"""ctypes binding of libgdpa.so: the C-ABI entry points under the same names.

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch supplies device memory (tensors and the workspace) and the
current stream. Loading fails loudly when the library is missing; there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdpa.so")

(GDPA_OK, GDPA_ERR_INVALID, GDPA_ERR_UNSUPPORTED, GDPA_ERR_CUDA, GDPA_ERR_WORKSPACE, GDPA_ERR_TIMEOUT,
 GDPA_ERR_SCRATCH_LIMIT) = range(7)
NOALLOC_SCRATCH_BYTES = 512 * 1024
DTYPES = {torch.bfloat16: 0, torch.float16: 1, torch.float8_e4m3fn: 2}
ACTS = {"identity": 0, "gelu": 1, "gelu_tanh": 2, "fast_gelu": 3, "relu": 4, "relu2": 5,
        "leaky_relu": 6, "silu": 7, "hardswish": 8, "softmax": 9, "fast_gelu_bf16": 10, "fast_silu": 11}
EXPORTS = ("gdpa_workspace_bytes", "gdpa_fwd", "gdpa_bwd", "gdpa_get_status", "gdpa_error_string",
           "gdpa_set_profile_events", "gdpa_fwd_noalloc", "gdpa_num_sms")


class GdpaShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("total_q", ctypes.c_int), ("total_k", ctypes.c_int),
                ("h_q", ctypes.c_int), ("h_kv", ctypes.c_int), ("d_qk", ctypes.c_int),
                ("d_v", ctypes.c_int), ("dtype", ctypes.c_int)]


class GdpaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"gdpa: {msg} (status {status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libgdpa.so (once) and declares the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libgdpa.so not found at {p}; build it with "
                               "`python -m generalized_attention_recsys_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sp = ctypes.POINTER(GdpaShape)
        lib.gdpa_workspace_bytes.argtypes = [sp, ci, ci, ci]
        lib.gdpa_workspace_bytes.restype = sz
        lib.gdpa_fwd.argtypes = [sp, vp, vp, vp, vp, vp, ci, ci, ci, cf, ci, ci, vp, vp, vp, vp, sz, vp]
        lib.gdpa_fwd.restype = ci
        lib.gdpa_bwd.argtypes = [sp, vp, vp, vp, vp, vp, ci, ci, ci, cf, ci, ci, vp, vp, vp, vp, vp, vp, ci,
                                 vp, sz, vp]
        lib.gdpa_bwd.restype = ci
        lib.gdpa_get_status.argtypes = [vp]
        lib.gdpa_get_status.restype = ci
        lib.gdpa_error_string.argtypes = [ci]
        lib.gdpa_error_string.restype = ctypes.c_char_p
        lib.gdpa_set_profile_events.argtypes = [vp, vp]
        lib.gdpa_set_profile_events.restype = ci
        lib.gdpa_fwd_mxfp8.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, cf, ci, ci, vp, vp, vp, sz,
                                       vp]
        lib.gdpa_fwd_mxfp8.restype = ci
        lib.gdpa_fwd_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, ci, ci, ci, cf, ci, ci, vp, vp, vp, vp]
        lib.gdpa_fwd_noalloc.restype = ci
        lib.gdpa_num_sms.argtypes = []
        lib.gdpa_num_sms.restype = ci
        _lib = lib
        return lib


def gdpa_error_string(status: int) -> str:
    return load().gdpa_error_string(status).decode()


def _check(status: int):
    if status != GDPA_OK:
        raise GdpaError(status, gdpa_error_string(status))


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _act(act) -> int:
    return ACTS[act] if isinstance(act, str) else int(act)


def make_shape(q, k, v, batch: int) -> GdpaShape:
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be packed [tokens, heads, head_dim]")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in DTYPES:
        raise ValueError("q, k, v must share one of bf16, fp16, float8_e4m3fn")
    return GdpaShape(batch, q.shape[0], k.shape[0], q.shape[1], k.shape[1], q.shape[2], v.shape[2],
                     DTYPES[q.dtype])


def gdpa_workspace_bytes(shape: GdpaShape, max_seqlen_q: int, max_seqlen_k: int, is_bwd: int) -> int:
    """is_bwd: 0 forward, 1 backward, 2 deterministic backward, 3 MXFP8 forward (C-ABI gdpa_workspace_bytes)."""
    return int(load().gdpa_workspace_bytes(ctypes.byref(shape), max_seqlen_q, max_seqlen_k, int(is_bwd)))


def _workspace(nbytes: int, device, workspace: torch.Tensor | None) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise GdpaError(GDPA_ERR_WORKSPACE, "workspace too small")
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def gdpa_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, act, scale: float,
             causal: bool = False, window: int = -1, descale_qkv=None, out=None, lse=None, batch=None,
             workspace=None, stream=None):
    """C-ABI gdpa_fwd. Returns (out, lse); lse is None unless act is softmax."""
    lib = load()
    if batch is None:
        batch = cu_seqlens_q.numel() - 1 if cu_seqlens_q is not None else q.shape[0] // max(max_seqlen_q, 1)
    shape = make_shape(q, k, v, batch)
    a = _act(act)
    if out is None:
        odt = torch.bfloat16 if q.dtype == torch.float8_e4m3fn else q.dtype
        out = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=odt, device=q.device)
    if a == ACTS["softmax"] and lse is None:
        lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
    nb = gdpa_workspace_bytes(shape, max_seqlen_q, max_seqlen_k, False)
    ws = _workspace(nb, q.device, workspace)
    st = lib.gdpa_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                      int(max_seqlen_q), int(max_seqlen_k), a, float(scale), int(bool(causal)), int(window),
                      _ptr(descale_qkv), _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(),
                      _stream(stream))
    _check(st)
    return out, (lse if a == ACTS["softmax"] else None)


def gdpa_fwd_mxfp8(q, k, v, q_scale, k_scale, v_scale, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                   max_seqlen_k: int, act, scale: float, causal: bool = False, window: int = -1, out=None, lse=None,
                   batch=None, workspace=None, stream=None):
    """C-ABI gdpa_fwd_mxfp8: q, k, v e4m3 codes; q_scale / k_scale [tokens, heads, d_qk / 32] and
    v_scale [ceil(total_k / 32), h_kv, d_v] E8M0 bytes (uint8). Returns (out, lse)."""
    lib = load()
    if batch is None:
        batch = cu_seqlens_q.numel() - 1 if cu_seqlens_q is not None else q.shape[0] // max(max_seqlen_q, 1)
    shape = make_shape(q, k, v, batch)
    a = _act(act)
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=torch.bfloat16, device=q.device)
    if a == ACTS["softmax"] and lse is None:
        lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
    for t in (q_scale, k_scale, v_scale):
        if t is not None and t.dtype != torch.uint8:
            raise TypeError("MX scales are E8M0 bytes (torch.uint8)")
    nb = gdpa_workspace_bytes(shape, max_seqlen_q, max_seqlen_k, 3)
    ws = _workspace(nb, q.device, workspace)
    st = lib.gdpa_fwd_mxfp8(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale),
                            _ptr(v_scale), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q),
                            int(max_seqlen_k), a, float(scale), int(bool(causal)), int(window), _ptr(out), _ptr(lse),
                            _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st)
    return out, (lse if a == ACTS["softmax"] else None)


def gdpa_bwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, act, scale: float,
             causal: bool, window: int, out, lse, dout, dq=None, dk=None, dv=None, deterministic: bool = False,
             batch=None, workspace=None, stream=None):
    """C-ABI gdpa_bwd. Returns (dq, dk, dv)."""
    lib = load()
    if batch is None:
        batch = cu_seqlens_q.numel() - 1 if cu_seqlens_q is not None else q.shape[0] // max(max_seqlen_q, 1)
    shape = make_shape(q, k, v, batch)
    if not dout.is_contiguous():
        dout = dout.contiguous()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nb = gdpa_workspace_bytes(shape, max_seqlen_q, max_seqlen_k, 2 if deterministic else 1)
    ws = _workspace(nb, q.device, workspace)
    st = lib.gdpa_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                      int(max_seqlen_q), int(max_seqlen_k), _act(act), float(scale), int(bool(causal)),
                      int(window), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                      int(bool(deterministic)), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st)
    return dq, dk, dv


def gdpa_get_status(stream=None) -> int:
    return int(load().gdpa_get_status(_stream(stream)))


def gdpa_num_sms() -> int:
    return int(load().gdpa_num_sms())


def gdpa_set_profile_events(before_main=None, after_main=None) -> None:
    """Brackets the main kernel of later calls on this thread with two events.

    Accepts torch.cuda.Event objects (they are recorded once here so that the
    underlying CUDA events exist) or raw handles; None, None clears the hook.
    """
    def handle(ev):
        if ev is None:
            return None
        if isinstance(ev, torch.cuda.Event):
            if ev.cuda_event == 0:
                ev.record()
            return ev.cuda_event
        return int(ev)

    _check(load().gdpa_set_profile_events(handle(before_main), handle(after_main)))


def gdpa_fwd_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, act,
                     scale: float, causal: bool = False, window: int = -1, descale_qkv=None, out=None, lse=None,
                     batch=None, stream=None):
    """C-ABI gdpa_fwd_noalloc: the forward with the library's fixed scratch
    instead of a workspace (for callers that cannot allocate device memory;
    the library itself allocates nothing). `out`/`lse` are allocated here only
    when not given. Calls sharing a device must not overlap on the GPU."""
    lib = load()
    if batch is None:
        batch = cu_seqlens_q.numel() - 1 if cu_seqlens_q is not None else q.shape[0] // max(max_seqlen_q, 1)
    shape = make_shape(q, k, v, batch)
    a = _act(act)
    if out is None:
        odt = torch.bfloat16 if q.dtype == torch.float8_e4m3fn else q.dtype
        out = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=odt, device=q.device)
    if a == ACTS["softmax"] and lse is None:
        lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
    st = lib.gdpa_fwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q),
                              _ptr(cu_seqlens_k), int(max_seqlen_q), int(max_seqlen_k), a, float(scale),
                              int(bool(causal)), int(window), _ptr(descale_qkv), _ptr(out), _ptr(lse),
                              _stream(stream))
    _check(st)
    return out, (lse if a == ACTS["softmax"] else None)
