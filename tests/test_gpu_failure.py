"""Failure detection without a GPU fault: a pipeline wait that nothing
satisfies gives up after its limit, the kernel reports
SFA_DEVSTAT_WAIT_TIMEOUT in the status word and returns, and the context
stays usable (a forward afterwards still matches the oracle)."""
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
