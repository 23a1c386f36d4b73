"""Failure detection on the device, without faulting the GPU.

Every wait in the kernels is bounded: a wait that gives up raises a
shared-memory abort flag, every role leaves its loop, lets its own TMA loads
and MMAs in flight land (time-bounded waits), TMEM is freed and the status
word reports GDPA_ERR_TIMEOUT. These tests make one such wait run out on
purpose, in a test-only build of the library (GDPA_TEST_HOOKS: waits give up
after 1 ms, and gdpa_test_set_skip() makes CTA 0 skip one mbarrier arrive, a
phase that then never completes). The kernel must return, gdpa_get_status
must report the timeout, and the next call on the same device must pass
parity against the oracle. Each case runs in a child process that loads only
the test build (a process holds one copy of the library).
"""

import os
import subprocess
import sys

import pytest

from generalized_attention_recsys_gb300 import build

pytestmark = pytest.mark.gpu

CHILD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "abort_child.py")


@pytest.fixture(scope="module")
def test_lib_path():
    return build.build(test_hooks=True)


@pytest.mark.parametrize("kernel,act", [("fwd", "gelu"), ("fwd", "relu2"), ("fwd", "softmax"), ("bwd", "gelu"),
                                        ("bwd", "softmax")])
def test_wait_runs_out_then_next_call_is_correct(test_lib_path, kernel, act):
    r = subprocess.run([sys.executable, CHILD, test_lib_path, kernel, act], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), f"child failed:\n{r.stdout}\n{r.stderr}"
