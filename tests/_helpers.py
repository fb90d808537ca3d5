"""Shared helpers of the GPU parity tests: seeded inputs on both sides, oracle
calls, sampled rows and the tolerances of the checks."""
from __future__ import annotations

import numpy as np
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs
from oracle import oracle

# Tolerances.  fp32 path: max abs error 1e-4 on O (and LSE).  bf16 inputs with
# fp32 accumulation: max abs error 2e-2 on O and LSE; input gradients within
# 2e-2 * max(1, max |oracle|) per tensor; dtheta within 5e-2 relative.
TOL = {
    "f32": {"o": 1e-4, "lse": 1e-4, "grad": 1e-4, "dtheta": 1e-3},
    "bf16": {"o": 2e-2, "lse": 2e-2, "grad": 2e-2, "dtheta": 5e-2},
}

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def draw(B, T, dtype, layer=0, seed=42, with_dO=False):
    """The same bytes for both sides: CPU tensors in ``dtype`` and their exact
    fp64 copies for the oracle."""
    x = inputs.qkv(B, T, dtype=DT[dtype], seed=seed, layer=layer, with_dO=with_dO)
    f64 = {k: v.to(torch.float64).numpy() for k, v in x.items()}
    return x, f64


def to_dev(x):
    return {k: v.cuda() for k, v in x.items()}


def gpu_forward(xd, *, alpha, W, rungs, rope_theta=1e4, **kw):
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=W, rungs=rungs,
                             rope_theta=rope_theta, **kw)
    torch.cuda.synchronize()
    return o, lse


def np64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def sample_rows(B, T, n, seed=0):
    """(b, i) pairs: the first and last query of every sequence, the queries
    where rungs start to apply, and random ones."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(B):
        rows.add((b, 0))
        rows.add((b, T - 1))
    for i in (1, 12, 13, 14, 20, 21, 22, 34, 35, 89, 90, 144, 145, 233, 377, 610, 987, 988, 1480,
              1481, 1482):
        if i < T:
            rows.add((int(rng.integers(0, B)), i))
    while len(rows) < n:
        rows.add((int(rng.integers(0, B)), int(rng.integers(0, T))))
    return np.array(sorted(rows), dtype=np.int32)


def max_abs(a, b):
    return float(np.max(np.abs(a - b))) if a.size else 0.0
