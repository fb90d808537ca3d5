"""Failure detection without a GPU fault: a pipeline wait that nothing
satisfies gives up after its limit, the kernel reports
SFA_DEVSTAT_WAIT_TIMEOUT in the status word and returns, and the context
stays usable (a forward afterwards still matches the oracle); a launch
failure injected on the host (SFA_TEST_FAULT=launch) reaches the Python
caller as an exception with nothing launched."""
import time

import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api
from oracle import oracle
from _helpers import TOL, draw, gpu_forward, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu

SFA_DEVSTAT_WAIT_TIMEOUT = 0x1


def test_wait_timeout_is_reported_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.sfa_selftest_wait_timeout(status)
    word = api.sfa_read_status(status)
    dt = time.perf_counter() - t0
    assert word & SFA_DEVSTAT_WAIT_TIMEOUT
    assert 0.2 <= dt < 10.0, dt  # the wait limit is 0.25 s
    # the same stream keeps working and computing the right thing
    x, f = draw(1, 200, "bf16", layer=90)
    o, lse = gpu_forward(to_dev(x), alpha=0.87, W=12, rungs=api.FIBONACCI_BASE)
    o_ref, _ = oracle.forward(f["q"], f["k"], f["v"], W=12, rungs=api.FIBONACCI_BASE, alpha=0.87)
    assert max_abs(np64(o), o_ref) <= TOL["bf16"]["o"]


def test_clean_runs_leave_the_status_word_clear():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x, _ = draw(2, 300, "bf16", layer=91, with_dO=True)
    xd = to_dev(x)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=1.1, W=12, status=status)
    api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, alpha=1.1, W=12, status=status)
    assert api.sfa_read_status(status) == 0


def test_injected_launch_fault_raises_in_the_binding():
    """SFA_TEST_FAULT=launch (a host-side hook, no device fault): the Python
    binding raises on the library's SFA_ERR_CUDA and no kernel is launched."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = r"""
import json, torch
from fibonacci_spaced_sparse_gb300 import api
q = torch.randn(1, 64, 8, 64, device="cuda").bfloat16()
k = torch.randn(1, 64, 2, 64, device="cuda").bfloat16()
v = torch.randn(1, 64, 2, 64, device="cuda").bfloat16()
n0 = api.launch_count()
try:
    api.sfa_forward(q, k, v, alpha=1.0, W=12, rope_theta=0.0)
    raised = ""
except RuntimeError as e:
    raised = str(e)
print(json.dumps({"raised": raised, "launches": api.launch_count() - n0}))
"""
    env = dict(os.environ, SFA_TEST_FAULT="launch", PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got["raised"] and got["launches"] == 0, got
