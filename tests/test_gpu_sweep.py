"""A seeded sweep of forward and backward parity against the fp64 oracle over
the parameter space at small sizes: sequence lengths from 1 to a few tiles
with ragged tails, windows 0..30, alpha over [0.5, 1.5] including integer and
half-integer values (every t = 0, and t = 1/2), both bases, RoPE on and off,
rounded offsets on and off, both dtypes.  Each case is drawn from its own
seed, so a failure names a reproducible configuration."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api
from oracle import oracle
from _helpers import TOL, cancellation_limit, check_dalpha_dtheta, draw, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu

N_CASES = 48


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.choice([1, 2, 13, 29, 57, 100, 171, 256, 333]))
    B = int(rng.integers(1, 4))
    W = int(rng.choice([0, 1, 3, 6, 8, 10, 12, 16, 24, 30]))
    alpha = float(rng.choice([0.5, 1.0, 1.5, 2.0 / 3.0, float(np.round(rng.uniform(0.5, 1.5), 4))]))
    base = "pow2" if rng.random() < 0.3 else "fib"
    rope = 0.0 if rng.random() < 0.2 else 1e4
    rnd = bool(rng.random() < 0.25)
    dtype = "f32" if rng.random() < 0.25 else "bf16"
    return dict(B=B, T=T, W=W, alpha=alpha, base=base, rope=rope, rnd=rnd, dtype=dtype)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_sweep_forward_backward(seed):
    c = _case(seed)
    B, T, W, alpha = c["B"], c["T"], c["W"], c["alpha"]
    rungs = api.pow2_base(max(T, 2)) if c["base"] == "pow2" else api.FIBONACCI_BASE
    x, f = draw(B, T, c["dtype"], layer=200 + seed, with_dO=True)
    xd = to_dev(x)
    kw = dict(alpha=alpha, W=W, rungs=rungs, rope_theta=c["rope"], round_offsets=c["rnd"])
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], **kw)
    dq, dk, dv, da, dth = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, **kw)
    torch.cuda.synchronize()
    okw = dict(W=W, rungs=rungs, alpha=alpha, rope_theta=c["rope"], round_offsets=c["rnd"])
    o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], **okw)
    tol = TOL[c["dtype"]]
    assert max_abs(np64(o), o_ref) <= tol["o"], c
    assert max_abs(np64(lse), lse_ref) <= tol["lse"], c
    ref = oracle.backward(f["q"], f["k"], f["v"], f["dO"], **okw)
    for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        bound = tol["grad"] * max(1.0, float(np.abs(want).max()) if want.size else 1.0)
        assert max_abs(np64(got), want) <= bound, (name, c)
    # dL/dalpha and dL/dtheta to the relative tolerance (exact zeros on both
    # sides with rounded offsets)
    got_da, got_dth = float(da.item()), float(dth.item())
    if c["rnd"]:
        assert got_da == 0.0 and ref[3] == 0.0, c
    check_dalpha_dtheta(got_da, got_dth, ref[3], ref[4], c["dtype"], c,
                        known_limit=cancellation_limit(rungs, ref[5], ref[3], c["dtype"]))
