"""A bounded device wait that runs out, on the GPU, without faulting it.

The test-hook build of the library (mixed_precision_attention_gb300.build.
build_test_hooks: APA_TEST_HOOKS and a ~0.5 s wait limit) has a switch that points
the pass-1 producer's wait for the in-launch K/V quantizer's tile flags at a word
that nothing sets.  That wait gives up, sets the CTA's abort flag and the device
error word; the producer lets its copies land, the issuers drain their tcgen05
operations, the softmax warps leave their loops and TMEM is freed (the unwind
modelled in test_pass1_protocol.py).  The call must report APA_ERR_DEVICE through
apa_check_error, and the next call on the same context must succeed and match the
oracle.  It runs in a child process, so the test-hook build stays out of this one."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_wait_that_runs_out_reports_and_leaves_the_gpu_usable():
    from mixed_precision_attention_gb300 import build
    lib = build.build_test_hooks()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_timeout_child.py"), lib],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["stuck_status"] == -7, res          # APA_ERR_DEVICE: the wait gave up
    assert res["stuck_seconds"] >= 0.2, res          # after its limit, not at once
    assert res["after_status"] == 0, res             # the context is still usable
    assert res["after_finite"] and res["after_max_err"] <= 1e-2, res
