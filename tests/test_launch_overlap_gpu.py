"""Kernels start before their predecessor on the stream has finished
(programmatic dependent launch) and must read nothing that predecessor
writes until their dependency wait returns. The work-list kernel writes
the list's entry count that the main kernels read: here every call gets a
zeroed workspace (a stale count of 0) and outputs pre-filled with a
sentinel, so a main kernel that read the count early would process no item
and leave the sentinel in place. Forward and backward, several calls back
to back, each checked for status and against the oracle."""

import pytest
import torch

from generalized_attention_recsys_gb300 import _lib, inputs
from gpu_util import FWD_TOL, GRAD_TOL, assert_close, ensure_built, max_lens, ref_bwd, ref_fwd, to_dev

pytestmark = pytest.mark.gpu


def test_stale_workspace_bytes_are_never_read():
    ensure_built()
    inp = inputs.custom(6, 4, 2, 128, 128, [700, 130, 1, 512, 300, 64], [700, 130, 1, 512, 300, 64], "gelu",
                        seed=41)
    wl = inp.wl
    d = to_dev(inp)
    mq, mk = max_lens(inp)
    shape = _lib.make_shape(d["q"], d["k"], d["v"], wl.batch)
    nf = _lib.gdpa_workspace_bytes(shape, mq, mk, False)
    nb = _lib.gdpa_workspace_bytes(shape, mq, mk, True)
    ref_out, _ = ref_fwd(inp)
    rq, rk, rv = ref_bwd(inp)
    for _ in range(4):
        ws_f = torch.zeros(nf, dtype=torch.uint8, device="cuda")
        out = torch.full((d["q"].shape[0], wl.h_q, wl.d_v), 7.0, dtype=torch.bfloat16, device="cuda")
        _lib.gdpa_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], mq, mk, wl.act, wl.softmax_scale, wl.causal,
                      wl.window, out=out, batch=wl.batch, workspace=ws_f)
        ws_b = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        dq, dk, dv = (torch.full_like(d[n], 7.0) for n in ("q", "k", "v"))
        _lib.gdpa_bwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], mq, mk, wl.act, wl.softmax_scale, wl.causal,
                      wl.window, None, None, d["dout"], dq=dq, dk=dk, dv=dv, batch=wl.batch, workspace=ws_b)
        assert _lib.gdpa_get_status() == 0
        assert_close(out, ref_out, FWD_TOL, "out")
        assert_close(dq, rq, GRAD_TOL, "dq")
        assert_close(dk, rk, GRAD_TOL, "dk")
        assert_close(dv, rv, GRAD_TOL, "dv")
