"""Child process of test_abort_gpu.py (not collected by pytest): loads only the
test-only build of the library given on the command line (a process holds one
copy of the library), makes one bounded wait run out in the forward or the
backward, checks that the call reports GDPA_ERR_TIMEOUT, then checks the next
call on the same device against the float64 oracle. Exit status 0 on success.

    python abort_child.py <libgdpa_test.so> fwd|bwd <activation>
"""

import ctypes
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import gpu_util  # noqa: E402
from generalized_attention_recsys_gb300 import _lib, inputs  # noqa: E402

FWD, BWD = 0, 1


def main(path: str, kernel: str, act: str) -> None:
    lib = _lib.load(path)  # the only copy of the library in this process
    gpu_util._built = True  # the tests' helpers use the loaded library as it is
    lib.gdpa_test_set_skip.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.gdpa_test_set_skip.restype = ctypes.c_int
    # one long sequence so that CTA 0 (the heaviest work item first) walks several steps
    lens = [1024, 300, 77, 129]
    inp = inputs.custom(len(lens), 2, 2, 128, 128, lens, lens, act, causal=act == "softmax", seed=41)
    wl = inp.wl
    q, k, v, do, cq, ck = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.dout, inp.cu_seqlens_q, inp.cu_seqlens_k))
    args = (q, k, v, cq, ck, inp.max_q, inp.max_k, wl.act, wl.softmax_scale, wl.causal, wl.window)
    if kernel == "fwd":
        assert lib.gdpa_test_set_skip(FWD, 1) == 0
        _lib.gdpa_fwd(*args, batch=wl.batch)
        status = _lib.gdpa_get_status()
        assert status == _lib.GDPA_ERR_TIMEOUT, f"forward status {status}, expected a timeout"
        assert lib.gdpa_test_set_skip(FWD, -1) == 0
        out, _ = gpu_util.run_fwd(inp)  # asserts a clean status
        ref, _ = gpu_util.ref_fwd(inp)
        gpu_util.assert_close(out, ref, gpu_util.FWD_TOL, f"out after an aborted {act} forward")
    else:
        out, lse = gpu_util.run_fwd(inp) if act == "softmax" else (None, None)
        assert lib.gdpa_test_set_skip(BWD, 1) == 0
        _lib.gdpa_bwd(*args, out, lse, do, batch=wl.batch)
        status = _lib.gdpa_get_status()
        assert status == _lib.GDPA_ERR_TIMEOUT, f"backward status {status}, expected a timeout"
        assert lib.gdpa_test_set_skip(BWD, -1) == 0
        dq, dk, dv = gpu_util.run_bwd(inp, out, lse)
        rq, rk, rv = gpu_util.ref_bwd(inp)
        for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
            gpu_util.assert_close(got, ref, gpu_util.GRAD_TOL, f"{name} after an aborted {act} backward")
    print("ok")


if __name__ == "__main__":
    main(*sys.argv[1:4])
