"""Rounded rung distances (round_offsets): every d_k = alpha * f_k replaced by
the nearest integer, halves up, as the static schedules "with integer offsets"
of section 2 "Implementation notes" take it.  The CUDA path against the fp64
oracle run with the same rounding: forward (bf16 and fp32), backward (dL/dalpha
is exactly zero), the multi-layer launch and decode."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api
from oracle import oracle
from _helpers import TOL, draw, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE


def _forward(B, T, dtype, alpha, W, rungs=FIB, layer=0, rope_theta=1e4):
    x, f = draw(B, T, dtype, layer=layer)
    xd = to_dev(x)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=W, rungs=rungs,
                             rope_theta=rope_theta, round_offsets=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], W=W, rungs=rungs, alpha=alpha,
                                    rope_theta=rope_theta, round_offsets=True)
    assert max_abs(np64(o), o_ref) <= TOL[dtype]["o"], (alpha, W)
    assert max_abs(np64(lse), lse_ref) <= TOL[dtype]["lse"], (alpha, W)
    return o_ref


# 0.61: distances 1.83, 3.05, 4.88, 7.93, 12.8, ... (none integer); 0.5: 1.5,
# 2.5, 4.0, 6.5 (halves round up); 1.37 with W = 13: 13.7 -> 14 is kept,
# 1.37 * 8 = 10.96 -> 11 is inside the window; 2.1: the fp32 product 2.1 * 55 is
# just below 115.5 and rounds down
@pytest.mark.parametrize("alpha,W", [(0.61, 6), (0.5, 1), (1.37, 13), (0.9, 12), (2.1, 4)])
def test_forward_bf16(alpha, W):
    _forward(2, 333, "bf16", alpha, W, layer=60)


@pytest.mark.parametrize("alpha,W", [(0.61, 6), (1.2345, 8)])
def test_forward_fp32(alpha, W):
    _forward(1, 300, "f32", alpha, W, layer=61)


def test_forward_pow2_base_no_rope():
    _forward(3, 517, "bf16", 0.77, 10, rungs=api.pow2_base(517), layer=62, rope_theta=0.0)


def test_rounding_changes_the_result():
    """At alpha = 0.61 the rounded and interpolated attentions differ well
    beyond the tolerance: the flag reaches the kernels."""
    x, _ = draw(2, 256, "bf16", layer=63)
    xd = to_dev(x)
    a, _ = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=0.61, W=6)
    b, _ = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=0.61, W=6, round_offsets=True)
    torch.cuda.synchronize()
    assert max_abs(np64(a), np64(b)) > 10 * TOL["bf16"]["o"]


@pytest.mark.parametrize("dtype,alpha,W", [("bf16", 0.61, 6), ("bf16", 1.37, 13),
                                           ("f32", 0.83, 8)])
def test_backward(dtype, alpha, W):
    B, T = 2, 301
    x, f = draw(B, T, dtype, layer=64, with_dO=True)
    xd = to_dev(x)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=W, round_offsets=True)
    dq, dk, dv, da, dth = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse,
                                           alpha=alpha, W=W, round_offsets=True)
    torch.cuda.synchronize()
    ref = oracle.backward(f["q"], f["k"], f["v"], f["dO"], W=W, rungs=FIB, alpha=alpha,
                          round_offsets=True)
    tol = TOL[dtype]
    for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        err = max_abs(np64(got), want)
        bound = tol["grad"] * max(1.0, float(np.abs(want).max()))
        assert err <= bound, (name, err, bound)
    assert ref[3] == 0.0 and ref[4] == 0.0
    assert float(da.item()) == 0.0 and float(dth.item()) == 0.0


def test_layers_equal_single_calls():
    B, T, L = 2, 400, 4
    alphas = [0.55, 0.71, 0.9, 1.13]
    xs = [to_dev(draw(B, T, "bf16", layer=70 + l)[0]) for l in range(L)]
    outs, lses = api.sfa_forward_layers([x["q"] for x in xs], [x["k"] for x in xs],
                                        [x["v"] for x in xs], alphas=alphas, W=12,
                                        round_offsets=True)
    for l in range(L):
        o, lse = api.sfa_forward(xs[l]["q"], xs[l]["k"], xs[l]["v"], alpha=alphas[l], W=12,
                                 round_offsets=True)
        torch.cuda.synchronize()
        assert torch.equal(outs[l], o) and torch.equal(lses[l], lse), l


def test_decode():
    B, Tc, alpha, W = 10, 500, 0.61, 6
    x, _ = draw(B, Tc, "bf16", layer=75)
    pos = np.array([0, 2, 5, 8, 13, 21, 34, 100, 377, Tc - 1], dtype=np.int32)
    qd = torch.stack([x["q"][b, p] for b, p in enumerate(pos)])
    o, lse = api.sfa_decode(qd.cuda(), x["k"].cuda(), x["v"].cuda(), torch.from_numpy(pos).cuda(),
                            alpha=alpha, W=W, round_offsets=True)
    torch.cuda.synchronize()
    rows = np.stack([np.arange(B, dtype=np.int32), pos], axis=1)
    f = {n: x[n].to(torch.float64).numpy() for n in ("q", "k", "v")}
    o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=W, rungs=FIB,
                                         alpha=alpha, round_offsets=True)
    assert max_abs(np64(o), o_ref) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse), lse_ref) <= TOL["bf16"]["lse"]
