"""Benchmark: sparse-attention forward query-tokens/s on the model-shape workload.

One step = the forward of all 16 layers of B=32 sequences of T=1024 tokens
(W=12, linear stagger alpha_l = 0.5 + l/15, Fibonacci base, bf16, 8 query / 2
key-value heads, d=64), each layer its own seeded inputs already resident in
HBM, through one sfa_forward_layers call (one attention launch per layer,
each also rotating the next layer's keys, plus one RoPE launch for layer 0).
The 16 layers' inputs (1.34 GB) are larger than L2, so no flush is needed
between steps.  ``value`` counts query tokens of every layer.

Also reported: ``e2e`` (the same step through the C ABI with pinned host
buffers, host->device inputs and device->host outputs inside the timed
region), ``roofline`` (the forward kernel's ideal bytes -- one read of Q, K, V
and one write of O -- over its average launch time from CUDA events on its
stream, against the measured HBM copy bandwidth), ``cpu_baseline`` (the fp64
CPU oracle on a bounded sample), and SM clocks sampled during the timed
region.

``--impl reference`` times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-attn fwd query-tokens/s (T=1024,W=12,bf16); HBM GB/s as % of GB300 peak"
UNIT = "query-tokens/s"
IDEAL_BYTES_PER_TOKEN = 2 * (8 * 64 + 2 * 64 + 2 * 64 + 8 * 64)  # bf16 Q, K, V read + O write
FALLBACK_HBM_GBS = 6800.0
E2E_MAX_STEPS = 20
SOAK_S = 1.0  # untimed run of the step right before the timed region (clock samples)
REFERENCE_BUDGET_S = 90.0  # oracle time of a whole --impl reference run


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="model-shape",
                    choices=["model-shape", "extrapolation", "pow2", "train-step", "long-forward",
                             "decode", "front-end"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------- replicas --
#
# With N > 1 (one process per GPU under torchrun) every rank runs its own
# independent batch of sequences -- the path shards over sequences with no
# exchange -- and the job's time is the slowest rank's.

def replica_seed(rank: int) -> int:
    """Seed of a rank's inputs: each rank draws its own batch."""
    return 42 + 1000 * int(rank)


def init_dist(world: int, dev=None, backend: str = "nccl") -> bool:
    """Joins the process group when world > 1 (127.0.0.1 rendezvous from the
    launcher's environment); returns whether there is one."""
    if world <= 1:
        return False
    import torch.distributed as dist
    if not dist.is_initialized():
        if backend == "nccl":
            dist.init_process_group(backend, device_id=dev)
        else:
            dist.init_process_group(backend)
    return True


def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time, returned on every rank (as is without a
    process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    """All ranks meet (and the device is idle) before and after a timed region."""
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()
    if device is not None and torch.cuda.is_available():
        torch.cuda.synchronize(device)


def aggregate_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time in milliseconds."""
    return float(units_per_rank) * int(world) / (float(ms) / 1e3)


def workload_of(name):
    from fibonacci_spaced_sparse_gb300 import workloads as w
    return {"model-shape": w.MODEL_SHAPE, "extrapolation": w.EXTRAPOLATION, "pow2": w.POW2,
            "train-step": w.TRAIN_STEP, "long-forward": w.LONG_FORWARD, "decode": w.DECODE}[name]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured (copy test)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if self.proc is None:
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------- traffic record --

# The sources that decide what the forward attention kernel does: its own
# file, the ring and PTX helpers it includes, and the host code that plans
# rungs and launches it.
FORWARD_SOURCES = ("sfa_fwd_mma.cu", "sfa_ring.cuh", "sfa_mma.cuh", "sfa_internal.cuh", "sfa_api.cu")


def code_only(text):
    """The source with its comments, trailing blanks and empty lines removed,
    so that a change to a comment leaves the digest as it was."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.split("\n") if line.strip())


def kernel_source_digest(sources=FORWARD_SOURCES):
    """First 16 hex digits of SHA-256 over the code of `sources`, in order."""
    from fibonacci_spaced_sparse_gb300 import build
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(build.CSRC, name), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def forward_kernel():
    """The bf16 forward kernel the library selects for this run's windows
    (all <= 16): the environment variable it reads picks the tcgen05 or the
    fp32-arithmetic kernel instead of the default."""
    return {"tc": "fwd_tc_kernel", "simple": "fwd_simple_kernel"}.get(
        os.environ.get("SFA_FORWARD_KERNEL", ""), "fwd_mma_kernel")


def recorded_traffic(workload_name):
    """DRAM bytes per launch of the forward kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"fwd_{workload_name}_traffic.txt")
    try:
        kv = {}
        with open(path) as fh:
            for line in fh:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_digest") != kernel_source_digest():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------- CPU baseline --

def oracle_alphas(wl):
    """The workload's per-layer alphas as the oracle states the schedules (the
    CPU arms never load the CUDA library)."""
    from oracle import oracle
    from fibonacci_spaced_sparse_gb300 import inputs
    if wl.schedule == "learned":
        return oracle.schedule_learned(inputs.thetas(wl.layers, wl.theta_sigma, seed=42))
    if wl.schedule == "linear":
        return oracle.schedule_linear(wl.layers)
    if wl.schedule == "coprime":
        return oracle.schedule_coprime(wl.layers, 7)
    return oracle.schedule_fixed(wl.layers)


def oracle_rungs(wl):
    """The workload's base offsets from the oracle's own tables."""
    from oracle import oracle
    return oracle.FIBONACCI_BASE if wl.base == "fibonacci" else oracle.pow2_base(wl.T)


def config_of(wl, world):
    """The ``config`` object of a bench line (the same for both arms)."""
    L = wl.layers
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "W": list(wl.W),
            "layers": L, "schedule": wl.schedule, "base": wl.base,
            "heads": "8q/2kv", "head_dim": 64,
            "backward": wl.backward,
            "l2": f"inputs larger than L2 ({L * 50.3 * wl.tokens / 32768:.0f} MB of "
                  "Q/K/V per step), no flush",
            "parallelism": f"replicas x{world}"}


def host_cpu() -> str:
    """The host CPU as /proc/cpuinfo names it (model name on x86; implementer
    and part number on Arm, e.g. 0x41/0xd4f for a Neoverse V2 / Grace core)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        return (f"{platform.machine()} implementer {fields.get('cpu implementer', '?')} "
                f"part {fields['cpu part']}")
    return platform.machine() or "unknown"


def cpu_baseline(wl, budget_s=12.0):
    """The fp64 oracle as it stands on the host cores: whole layers of the
    workload (all B sequences), cycling through its first four layers until
    about budget_s seconds of oracle time are spent."""
    import torch
    from fibonacci_spaced_sparse_gb300 import inputs
    from oracle import oracle
    oracle.build()
    alphas, rungs = oracle_alphas(wl), oracle_rungs(wl)
    cores = oracle.default_threads()
    data = {}
    tokens, spent, calls = 0, 0.0, 0
    nl = min(4, wl.layers)
    while spent < budget_s and calls < 8 * wl.layers:
        l = calls % nl
        if l not in data:
            x = inputs.qkv(wl.B, wl.T, dtype=torch.bfloat16, layer=l)
            data[l] = {k: v.to(torch.float64).numpy() for k, v in x.items()}
        f = data[l]
        t0 = time.perf_counter()
        oracle.forward(f["q"], f["k"], f["v"], W=wl.window(l), rungs=rungs, alpha=alphas[l],
                       nthreads=cores)
        spent += time.perf_counter() - t0
        tokens += wl.B * wl.T
        calls += 1
    return {"value": tokens / spent, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu": host_cpu(), "sample": f"{calls} whole-layer forwards ({wl.B}x{wl.T} query tokens each, "
                      f"layers 0..{nl - 1} in turn), {spent:.1f} s of oracle time"}


# --------------------------------------------------------------- our arm --

def run_ours(args, rank, world, local):
    import torch
    from fibonacci_spaced_sparse_gb300 import api, inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of(args.workload)
    alphas, _ = wl.alphas()
    L = wl.layers
    bf = torch.bfloat16
    # every rank holds its own batch (weak scaling: replicas over independent sequences)
    host = [inputs.qkv(wl.B, wl.T, dtype=bf, seed=replica_seed(rank), layer=l, with_dO=wl.backward)
            for l in range(L)]
    dv = [{k: v.to(dev) for k, v in h.items()} for h in host]
    outs = [torch.empty_like(d["q"]) for d in dv]
    lses = [torch.empty((wl.B, wl.T, 8), dtype=torch.float32, device=dev) for _ in range(L)]
    api.rope_table(wl.T, dev)
    stream = torch.cuda.current_stream(dev)
    ws = None
    if wl.backward:
        need = max(api.sfa_backward_workspace_size(wl.B, wl.T, alpha=a, W=wl.window(l),
                                                   rungs=wl.rungs()) for l, a in enumerate(alphas))
        ws = torch.empty(need, dtype=torch.uint8, device=dev)

    windows = [wl.window(l) for l in range(L)]
    qs, ks, vs = [d["q"] for d in dv], [d["k"] for d in dv], [d["v"] for d in dv]

    def step(events=None):
        # the forward of every layer in one call; with a backward, layer by
        # layer (the backward needs each layer's O and LSE)
        if events is not None:
            events[0].record(stream)
        api.sfa_forward_layers(qs, ks, vs, alphas=alphas, W=windows, rungs=wl.rungs(), outs=outs,
                               lses=lses)
        if events is not None:
            events[1].record(stream)
        if wl.backward:
            for l in range(L):
                if events is not None:
                    events[2 + 2 * l].record(stream)
                api.sfa_backward(dv[l]["q"], dv[l]["k"], dv[l]["v"], outs[l], dv[l]["dO"], lses[l],
                                 alpha=alphas[l], W=wl.window(l), rungs=wl.rungs(), workspace=ws)
                if events is not None:
                    events[3 + 2 * l].record(stream)

    use_dist = init_dist(world, dev)

    t_warm = time.perf_counter()
    for _ in range(max(3, args.warmup)):
        step()
    barrier(dev)
    step_s = (time.perf_counter() - t_warm) / max(3, args.warmup)

    # device-timed region: K steps, per-launch events on the launching stream
    nev = 2 + (2 * L if wl.backward else 0)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = -1
    with ClockSampler(local) as clk:
        # the same step, untimed, for about SOAK_S seconds right before the
        # timed region, so that the clock record has enough samples under this
        # load even when K steps take only milliseconds
        soak(step, step_s, dev)
        barrier(dev)
        n0 = api.launch_count()
        start.record(stream)
        for s in range(args.steps):
            step(ev[s])
        stop.record(stream)
        barrier(dev)
    launches = api.launch_count() - n0
    elapsed_ms = start.elapsed_time(stop)
    # per-layer average of the forward (the multi-layer call's time / L)
    fwd_ms = [st[0].elapsed_time(st[1]) / L for st in ev]
    bwd_ms = [st[2 + 2 * l].elapsed_time(st[3 + 2 * l]) for st in ev for l in range(L)] if wl.backward else []
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    value = aggregate_rate(wl.B * wl.T * L * args.steps, world, elapsed_ms)

    # roofline of the forward kernel
    peak, peak_kind = measured_peak()
    avg_launch_s = statistics.mean(fwd_ms) / 1e3
    ideal = IDEAL_BYTES_PER_TOKEN * wl.B * wl.T
    achieved = ideal / avg_launch_s / 1e9
    kernel = forward_kernel()
    # the committed DRAM-traffic record is of the default kernel
    traffic = recorded_traffic(args.workload) if kernel == "fwd_mma_kernel" else None

    # end to end through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, alphas, host, dev, stream, world, use_dist)

    cpu = None
    if rank == 0 and not args.no_cpu and world == 1:
        cpu = cpu_baseline(wl)

    if args.workload == "model-shape" and not args.no_backward:
        # the training step's backward, timed beside the headline forward
        backward = time_backward(dev, stream, rank)
    elif wl.backward:
        bwd_avg = statistics.mean(bwd_ms) / 1e3
        # backward ideal bytes: read Q, K, V, O, dO and write dQ, dK, dV once (bf16)
        bwd_ideal = 2 * (8 * 64 + 2 * 64 + 2 * 64 + 8 * 64 + 8 * 64 + 8 * 64 + 2 * 64 + 2 * 64) * wl.B * wl.T
        backward = {"avg_launch_us": bwd_avg * 1e6, "ideal_bytes_per_call": bwd_ideal,
                    "achieved": bwd_ideal / bwd_avg / 1e9, "peak": peak, "unit": "GB/s",
                    "frac": bwd_ideal / bwd_avg / 1e9 / peak}
    else:
        backward = None
    clocks = clk.summary()
    if clocks:
        clocks["window"] = f"{SOAK_S:.1f} s of the same step untimed, then the timed region"
        clocks["ms_per_step_x_sm_mhz"] = elapsed_ms / args.steps * clocks["sm_mhz"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(wl, world),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": f"forward attention ({kernel})",
                         "ideal_bytes_per_launch": ideal,
                         "avg_launch_us": avg_launch_s * 1e6,
                         "avg_launch_note": "per-layer average of the timed multi-layer calls "
                                            "(CUDA events on the launching stream), including "
                                            "layer 0's RoPE launch and launch gaps",
                         "peak_kind": peak_kind},
            "cpu_baseline": cpu,
            "backward": backward,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if use_dist:
        import torch.distributed as dist
        dist.destroy_process_group()


def soak(step, step_s, dev):
    """Runs ``step`` untimed for about SOAK_S seconds (at least one step)."""
    import torch
    n = max(1, int(SOAK_S / max(step_s, 1e-4)))
    for _ in range(n):
        step()
    torch.cuda.synchronize(dev)


def time_backward(dev, stream, rank, layers=4, iters=10):
    """The backward of the training-step workload (B=32, T=1024, W=12,
    Fibonacci base, learned-style alpha = 0.5 + sigmoid(theta), theta ~ N(0,
    0.5)), timed layer by layer with CUDA events on the launching stream after
    a forward of each layer: the per-layer time and its fraction of HBM peak
    on the ideal bytes (one read of Q, K, V, O, dO and one write of dQ, dK,
    dV).  ``layers`` of the 16 layers, each its own seeded inputs."""
    import torch
    from fibonacci_spaced_sparse_gb300 import api, inputs
    wl = workload_of("train-step")
    alphas, _ = wl.alphas()
    W, rungs = wl.window(0), wl.rungs()
    d = [{k: v.to(dev) for k, v in inputs.qkv(wl.B, wl.T, dtype=torch.bfloat16, seed=replica_seed(rank),
                                              layer=l, with_dO=True).items()} for l in range(layers)]
    outs, lses = [], []
    for l in range(layers):
        o, lse = api.sfa_forward(d[l]["q"], d[l]["k"], d[l]["v"], alpha=alphas[l], W=W, rungs=rungs)
        outs.append(o)
        lses.append(lse)
    need = max(api.sfa_backward_workspace_size(wl.B, wl.T, alpha=alphas[l], W=W, rungs=rungs)
               for l in range(layers))
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    grads = [(torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]),
              torch.empty(1, dtype=torch.float32, device=dev), torch.empty(1, dtype=torch.float32, device=dev))
             for x in d]

    def one(l):
        api.sfa_backward(d[l]["q"], d[l]["k"], d[l]["v"], outs[l], d[l]["dO"], lses[l], alpha=alphas[l],
                         W=W, rungs=rungs, workspace=ws, out=grads[l])

    for _ in range(3):
        for l in range(layers):
            one(l)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters * layers)]
    for it in range(iters):
        for l in range(layers):
            a, b = ev[it * layers + l]
            a.record(stream)
            one(l)
            b.record(stream)
    torch.cuda.synchronize(dev)
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    ideal = 2 * (8 * 64 * 4 + 2 * 64 * 4) * wl.B * wl.T
    peak, peak_kind = measured_peak()
    return {"workload": wl.name + " (backward only)", "layers_timed": layers, "calls": iters * layers,
            "avg_launch_us": us, "ideal_bytes_per_call": ideal, "achieved": ideal / (us * 1e-6) / 1e9,
            "peak": peak, "unit": "GB/s", "frac": ideal / (us * 1e-6) / 1e9 / peak, "peak_kind": peak_kind,
            "note": "per-layer sfa_backward call (all its launches), CUDA events on the launching stream, "
                    "inputs larger than L2"}


def run_e2e(args, wl, alphas, host, dev, stream, world, use_dist):
    """Same step through the C ABI from pinned host buffers: each step copies
    every layer's Q, K, V host->device, runs the layer, and copies O back.
    Copies run on their own streams through NB device staging buffers used in
    turn (across steps too), so the uploads run ahead of the attention and the
    downloads follow it; events order each layer's three stages.  The only
    waits are the hazards: an upload into a buffer waits for the attention
    launch that last read it, an attention launch waits for the download that
    last read its output buffer."""
    import torch
    from fibonacci_spaced_sparse_gb300 import api
    L = wl.layers
    pin = [{k: host[l][k].pin_memory() for k in ("q", "k", "v")} for l in range(L)]
    o_host = [torch.empty_like(pin[l]["q"]).pin_memory() for l in range(L)]
    NB = 3
    dq = [{k: torch.empty_like(pin[0][k], device=dev) for k in ("q", "k", "v")} for _ in range(NB)]
    do = [torch.empty_like(dq[0]["q"]) for _ in range(NB)]
    lse = [torch.empty((wl.B, wl.T, 8), dtype=torch.float32, device=dev) for _ in range(NB)]
    h2d = sum(pin[l][k].numel() * pin[l][k].element_size() for l in range(L) for k in pin[l])
    d2h = sum(o.numel() * o.element_size() for o in o_host)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    read_in = [None] * NB    # per buffer: the attention launch that last read its inputs
    read_out = [None] * NB   # per buffer: the download that last read its output
    turn = [0]

    def step():
        for l in range(L):
            s = turn[0] % NB
            turn[0] += 1
            with torch.cuda.stream(up):
                if read_in[s] is not None:
                    up.wait_event(read_in[s])
                for k in ("q", "k", "v"):
                    dq[s][k].copy_(pin[l][k], non_blocking=True)
                loaded = ev()
                loaded.record(up)
            stream.wait_event(loaded)
            if read_out[s] is not None:
                stream.wait_event(read_out[s])
            api.sfa_forward(dq[s]["q"], dq[s]["k"], dq[s]["v"], alpha=alphas[l], W=wl.window(l),
                            rungs=wl.rungs(), out=do[s], lse=lse[s], stream=stream)
            read_in[s] = ev()
            read_in[s].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(read_in[s])
                o_host[l].copy_(do[s], non_blocking=True)
                read_out[s] = ev()
                read_out[s].record(down)

    def drain():
        stream.wait_stream(up)
        stream.wait_stream(down)

    for _ in range(max(3, min(args.warmup, 5))):
        step()
    drain()
    torch.cuda.synchronize(dev)
    steps = min(args.steps, E2E_MAX_STEPS)  # each step moves 1.3 GB over the host link
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    for _ in range(steps):
        step()
    drain()
    stop.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(start.elapsed_time(stop), dev)
    return {"value": aggregate_rate(wl.B * wl.T * L * steps, world, ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps}


# ------------------------------------------------------------ decode arm --

def run_decode(args, rank, world, local):
    """Single-token decode: one step = one new token for each of B sequences
    through all 16 layers (16 sfa_decode calls, captured once in a CUDA graph
    and replayed), every layer with its own
    4096-row key/value cache (seeded N(0, 1) bf16, drawn on the device) and
    the sequences at seeded positions in the cache's second half.  The
    caches (8.6 GB) dwarf L2, so every step reads cold rows."""
    import torch
    from fibonacci_spaced_sparse_gb300 import api
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of("decode")
    alphas, _ = wl.alphas()
    L, B, Tc, W = wl.layers, wl.B, wl.T, wl.window(0)
    use_dist = init_dist(world, dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(replica_seed(rank))
    shape = (B, Tc, 2, 64)
    kc = [torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16) for _ in range(L)]
    vc = [torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16) for _ in range(L)]
    qs = [torch.randn((B, 8, 64), generator=gen, device=dev).to(torch.bfloat16) for _ in range(L)]
    pos = torch.randint(Tc // 2, Tc, (B,), generator=gen, device=dev, dtype=torch.int32)
    outs = [torch.empty_like(q) for q in qs]
    lses = [torch.empty((B, 8), dtype=torch.float32, device=dev) for _ in range(L)]
    api.rope_table(Tc, dev)
    stream = torch.cuda.current_stream(dev)

    def layers(s):
        for l in range(L):
            api.sfa_decode(qs[l], kc[l], vc[l], pos, alpha=alphas[l], W=W, out=outs[l], lse=lses[l],
                           stream=s)

    # the 16 calls of a step are captured once in a CUDA graph (a step is
    # ~16 short launches; replaying the graph keeps the host out of the timing)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        layers(side)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        layers(side)

    def step():
        graph.replay()

    t_warm = time.perf_counter()
    for _ in range(max(3, args.warmup)):
        step()
    barrier(dev)
    step_s = (time.perf_counter() - t_warm) / max(3, args.warmup)
    steps = max(1, args.steps)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        soak(step, step_s, dev)
        barrier(dev)
        start.record(stream)
        for _ in range(steps):
            step()
        stop.record(stream)
        barrier(dev)
    launches = L * steps  # graph replays: the library's counter sees only the capture
    ms = max_over_ranks(start.elapsed_time(stop), dev)
    # bytes one step must move: every layer's Q and O rows, and the distinct
    # cache rows (key and value, both kv heads) of each sequence's key list
    p_host = pos.cpu().numpy()
    rows = 0
    for l in range(L):
        plan = api.rung_plan(T=Tc, W=W, alpha=alphas[l])
        for i in p_host:
            used = set(range(max(0, i - W), i + 1))
            for (_, n, t, c) in plan:
                if i - c >= 0:
                    used.add(i - n)
                    if t > 0:
                        used.add(i - n - 1)
            rows += len(used)
    step_bytes = rows * 2 * 2 * 64 * 2 + L * B * 2 * (8 * 64 * 2)
    peak, peak_kind = measured_peak()
    per_layer_s = ms / 1e3 / steps / L
    achieved = step_bytes / L / per_layer_s / 1e9
    line = {
        "metric": "sparse-attn decode tokens/s (one new token per sequence through 16 layers)",
        "value": aggregate_rate(B * steps, world, ms), "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "B": B, "cache_rows": Tc, "W": [W], "layers": L,
                   "schedule": wl.schedule, "base": wl.base,
                   "l2": "caches of 8.6 GB, rows read cold each step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "decode_fast_kernel",
                     "ideal_bytes_per_launch": step_bytes / L, "avg_launch_us": per_layer_s * 1e6,
                     "peak_kind": peak_kind},
        "gpu_launches": launches, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if use_dist:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------- front-end arm --

def measured_tflops(kind="bf16_tflops_sustained"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)[kind]), f"measured ({kind})"
    except Exception:
        return 1700.0, "fallback"


def run_front_end(args, rank, world, local):
    """A layer with its fused front end: one step = for each of the 16
    model-shape layers (B=32, T=1024, W=12, linear stagger), sfa_qkv_rope on
    that layer's hidden states X [32, 1024, 512] with its weight Wqkv [768, 512]
    (RoPE in the epilogue), then sfa_forward on the rotated tensors with the
    rotation off.  Every layer has its own seeded X and Wqkv resident in HBM
    (537 MB of X per step, larger than L2).  ``value`` counts query tokens;
    the roofline is the front-end kernel's (a dense contraction: tensor-bound,
    2 x 768 x 512 flops per token) against the sustained cuBLAS bf16 rate."""
    import torch
    from fibonacci_spaced_sparse_gb300 import api, inputs
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of("model-shape")
    alphas, _ = wl.alphas()
    L, B, T, dm = wl.layers, wl.B, wl.T, 512
    use_dist = init_dist(world, dev)
    xw = [inputs.hidden_and_weight(B, T, dm, seed=replica_seed(rank), layer=l) for l in range(L)]
    xs = [x.to(dev) for x, _ in xw]
    wts = [w.to(dev) for _, w in xw]
    bf = torch.bfloat16
    bufs = [(torch.empty((B, T, 8, 64), dtype=bf, device=dev),
             torch.empty((B, T, 2, 64), dtype=bf, device=dev),
             torch.empty((B, T, 2, 64), dtype=bf, device=dev)) for _ in range(2)]
    outs = [torch.empty((B, T, 8, 64), dtype=bf, device=dev) for _ in range(L)]
    lses = [torch.empty((B, T, 8), dtype=torch.float32, device=dev) for _ in range(L)]
    api.rope_table(T, dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        for l in range(L):
            if ev is not None:
                ev[3 * l].record(stream)
            qh, kh, v = api.sfa_qkv_rope(xs[l], wts[l], out=bufs[l & 1])
            if ev is not None:
                ev[3 * l + 1].record(stream)
            api.sfa_forward(qh, kh, v, alpha=alphas[l], W=wl.window(l), rope_theta=0.0,
                            out=outs[l], lse=lses[l])
            if ev is not None:
                ev[3 * l + 2].record(stream)

    t_warm = time.perf_counter()
    for _ in range(max(3, args.warmup)):
        step()
    barrier(dev)
    step_s = (time.perf_counter() - t_warm) / max(3, args.warmup)
    steps = max(1, args.steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 * L)] for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        soak(step, step_s, dev)
        barrier(dev)
        n0 = api.launch_count()
        start.record(stream)
        for s_ in range(steps):
            step(ev[s_])
        stop.record(stream)
        barrier(dev)
    launches = api.launch_count() - n0
    ms = max_over_ranks(start.elapsed_time(stop), dev)
    qkv_us = statistics.mean(e[3 * l].elapsed_time(e[3 * l + 1]) for e in ev for l in range(L)) * 1e3
    att_us = statistics.mean(e[3 * l + 1].elapsed_time(e[3 * l + 2]) for e in ev for l in range(L)) * 1e3
    flops = 2.0 * 768 * dm * B * T
    tpeak, tkind = measured_tflops()
    hpeak, hkind = measured_peak()
    achieved = flops / (qkv_us * 1e-6) / 1e12
    io_bytes = (dm * 2 + 768 * 2) * B * T  # read X, write Qhat, Khat, V (bf16)
    line = {
        "metric": "layer with fused QKV+RoPE front end, query-tokens/s (T=1024,W=12,bf16)",
        "value": aggregate_rate(B * T * L * steps, world, ms), "unit": UNIT, "n_gpus": world,
        "steps": steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "model-shape layers with the QKV+RoPE front end", "B": B, "T": T,
                   "W": list(wl.W), "layers": L, "d_model": dm, "schedule": wl.schedule,
                   "l2": "537 MB of X per step, larger than L2, no flush"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                     "frac": achieved / tpeak, "traffic": None, "kernel": "qkv_rope_kernel",
                     "flops_per_launch": flops, "avg_launch_us": qkv_us, "peak_kind": tkind,
                     "hbm": {"ideal_bytes_per_launch": io_bytes,
                             "achieved_gbs": io_bytes / (qkv_us * 1e-6) / 1e9, "peak": hpeak,
                             "peak_kind": hkind}},
        "attention_rope_off_us": att_us,
        "e2e": None, "gpu_launches": launches, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if use_dist:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------- reference arm --

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the host cores: each step is a
    bounded sample of the workload -- a slice of whole sequences of one layer
    (layers 0..3 in turn) -- sized from a one-sequence calibration so that the
    warm-up and timed steps together take about REFERENCE_BUDGET_S seconds of
    oracle time, whatever --steps is."""
    if rank != 0:
        return
    import torch
    from fibonacci_spaced_sparse_gb300 import inputs
    from oracle import oracle
    oracle.build()
    wl = workload_of(args.workload)
    alphas, rungs = oracle_alphas(wl), oracle_rungs(wl)
    cores = oracle.default_threads()
    nl = min(wl.layers, 4)
    data = []
    for l in range(nl):
        x = inputs.qkv(wl.B, wl.T, dtype=torch.bfloat16, layer=l)
        data.append({k: v.to(torch.float64).numpy() for k, v in x.items()})

    def run(l, b0, n):
        f = data[l]
        oracle.forward(f["q"][b0:b0 + n], f["k"][b0:b0 + n], f["v"][b0:b0 + n], W=wl.window(l),
                       rungs=rungs, alpha=alphas[l], nthreads=cores)

    t0 = time.perf_counter()
    run(0, 0, 1)
    t_seq = time.perf_counter() - t0
    warm, steps = max(3, args.warmup), max(1, args.steps)
    n_seq = int(max(1, min(wl.B, REFERENCE_BUDGET_S / ((warm + steps) * max(t_seq, 1e-6)))))

    def step(i):
        run(i % nl, (i * n_seq) % (wl.B - n_seq + 1), n_seq)

    for i in range(warm):
        step(i)
    t0 = time.perf_counter()
    for i in range(steps):
        step(warm + i)
    dt = time.perf_counter() - t0
    value = n_seq * wl.T * steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu": host_cpu(), "sample": f"{n_seq} of {wl.B} sequences ({n_seq * wl.T} query tokens) of one "
                                   f"layer per step, layers 0..{nl - 1} in turn, sized for about "
                                   f"{REFERENCE_BUDGET_S:.0f} s over {warm + steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    from fibonacci_spaced_sparse_gb300 import build
    build.build()
    if args.workload == "decode":
        run_decode(args, rank, world, local)
        return
    if args.workload == "front-end":
        run_front_end(args, rank, world, local)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
