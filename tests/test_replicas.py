"""The N > 1 path of bench.py on the CPU: two gloo ranks on 127.0.0.1.

The method shards over sequences with no exchange, so with one process per
GPU every rank runs its own batch (weak scaling) and the job's time is the
slowest rank's; these tests check that host logic without a GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from fibonacci_spaced_sparse_gb300 import inputs  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    assert bench.init_dist(world, backend="gloo")
    bench.barrier()
    # rank r "took" 10 + 5 r ms: every rank must see the slowest
    ms = bench.max_over_ranks(10.0 + 5.0 * rank)
    # each rank's own batch
    q = inputs.qkv(1, 8, seed=bench.replica_seed(rank))["q"].float()
    gathered = [torch.zeros_like(q) for _ in range(world)]
    dist.all_gather(gathered, q)
    rate = bench.aggregate_rate(1000, world, ms)
    out[rank] = (ms, rate, all(not torch.equal(gathered[a], gathered[b])
                              for a in range(world) for b in range(a + 1, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_independent_batches():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(world):
        ms, rate, distinct = res[r]
        assert ms == 15.0                      # the slowest rank's time on every rank
        assert rate == pytest.approx(1000 * 2 / 0.015)
        assert distinct                         # replicas draw different sequences


def test_single_process_helpers_are_identity():
    assert not bench.init_dist(1)
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_rate(500, 1, 2.0) == pytest.approx(250000.0)


def test_torchrun_two_ranks_reference_arm_prints_one_line():
    """bench.py under torchrun with two ranks: rank 0 alone runs the
    reference arm (the oracle on a bounded sample) and prints one JSON line;
    rank 1 exits 0 without output."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "model-shape"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
