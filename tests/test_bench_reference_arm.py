"""The CPU legs of bench.py (the reference arm and the CPU baseline) take the
schedules and base offsets from the oracle and never load the CUDA library;
the reference arm's line carries the same config object as the GPU arm's."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import io, json, sys, contextlib
sys.path.insert(0, ROOT)
import bench
from oracle import oracle
from fibonacci_spaced_sparse_gb300 import workloads as w
bench.REFERENCE_BUDGET_S = 0.5
class A: pass
args = A(); args.workload = "model-shape"; args.steps = 1; args.warmup = 3
out = io.StringIO()
with contextlib.redirect_stdout(out):
    bench.run_reference(args, 0, 1)
line = json.loads(out.getvalue().strip().splitlines()[-1])
maps = open("/proc/self/maps").read()
print(json.dumps({"line": line, "libsfa": "libsfa" in maps, "liboracle": "liboracle" in maps,
                  "alphas": bench.oracle_alphas(w.MODEL_SHAPE), "ramp": oracle.schedule_linear(16),
                  "config": bench.config_of(w.MODEL_SHAPE, 1)}))
"""


def test_reference_arm_runs_the_oracle_only():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], capture_output=True, text=True,
                       timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    assert not rec["libsfa"] and rec["liboracle"]
    assert rec["alphas"] == rec["ramp"]
    line = rec["line"]
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"] == rec["config"]


def test_source_digest_ignores_comments_only():
    """The traffic record stays valid across an edit to a comment, and is
    dropped by any change to the code."""
    sys.path.insert(0, ROOT)
    import bench
    src = "int a = 1; // one\n\n/* block\n   comment */\nint b = 2;   \n"
    assert bench.code_only(src) == "int a = 1;\nint b = 2;"
    assert bench.code_only(src.replace("// one", "// the first")) == bench.code_only(src)
    assert bench.code_only(src.replace("2", "3")) != bench.code_only(src)


def test_forward_kernel_label_follows_the_selection(monkeypatch):
    """The bench line names the forward kernel the library's environment
    switch selects; the committed DRAM-traffic record belongs to the default
    kernel only."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("SFA_FORWARD_KERNEL", raising=False)
    assert bench.forward_kernel() == "fwd_mma_kernel"
    monkeypatch.setenv("SFA_FORWARD_KERNEL", "tc")
    assert bench.forward_kernel() == "fwd_tc_kernel"
    monkeypatch.setenv("SFA_FORWARD_KERNEL", "simple")
    assert bench.forward_kernel() == "fwd_simple_kernel"
