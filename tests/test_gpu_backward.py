"""Backward parity: dQ, dK, dV, dalpha and dtheta from the CUDA path against the
fp64 oracle on the same seeded inputs (small sizes element by element, the
training-step workload at full size)."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs, workloads
from oracle import oracle
from _helpers import TOL, cancellation_limit, check_dalpha_dtheta, kernel_rotation, draw, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE


def run(B, T, dtype, *, alpha, W, rungs=FIB, layer=0, rope_theta=1e4):
    x, f = draw(B, T, dtype, layer=layer, with_dO=True)
    xd = to_dev(x)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=W, rungs=rungs,
                             rope_theta=rope_theta)
    dq, dk, dv, da, dth = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse,
                                           alpha=alpha, W=W, rungs=rungs, rope_theta=rope_theta)
    torch.cuda.synchronize()
    ref = oracle.backward(f["q"], f["k"], f["v"], f["dO"], W=W, rungs=rungs, alpha=alpha,
                          rope_theta=rope_theta)
    tol = TOL[dtype]
    for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        err = max_abs(np64(got), want)
        bound = tol["grad"] * max(1.0, float(np.abs(want).max()) if want.size else 1.0)
        assert err <= bound, (name, err, bound)
    check_dalpha_dtheta(float(da.item()), float(dth.item()), ref[3], ref[4], dtype)
    return ref


@pytest.mark.parametrize("alpha", [0.61, 1.0, 1.2345])
def test_fp32_small(alpha):
    run(2, 150, "f32", alpha=alpha, W=8, layer=2)


@pytest.mark.parametrize("alpha,W", [(0.5, 12), (0.873, 12), (1.31, 6), (1.5, 12)])
def test_bf16_small(alpha, W):
    run(2, 300, "bf16", alpha=alpha, W=W, layer=3)


def test_pow2_and_edges():
    run(1, 257, "bf16", alpha=api.alpha_from_theta(0.4), W=10, rungs=api.pow2_base(257))
    run(2, 1, "f32", alpha=0.7, W=12)                      # single token
    run(2, 40, "f32", alpha=0.9, W=64)                     # dense limit
    run(2, 40, "f32", alpha=0.9, W=5, rungs=())            # window only
    run(2, 64, "f32", alpha=1.11, W=8, rope_theta=0.0)     # pre-rotated inputs


def test_integer_distance_rung_at_sequence_start():
    """alpha = 1: every t = 0; the query i = f_k uses row 0 only and the
    t-derivative there has no row -1 (zero by convention)."""
    run(1, 120, "f32", alpha=1.0, W=8)


@pytest.mark.parametrize("layer", [0, 9])
def test_train_step_full(layer):
    wl = workloads.TRAIN_STEP
    alphas, _ = wl.alphas()
    run(wl.B, wl.T, "bf16", alpha=alphas[layer], W=12, layer=layer)


def test_autograd_theta_matches_library():
    x, _ = draw(1, 96, "f32", layer=7, with_dO=True)
    xd = to_dev(x)
    q, k, v = (xd[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    theta = torch.tensor(0.31, device="cuda", requires_grad=True)
    o = api.SparseAttention.apply(q, k, v, theta, 8)
    (o * xd["dO"]).sum().backward()
    alpha = api.alpha_from_theta(0.31)
    _, _, _, _, dth_ref, _ = oracle.backward(*(x[n].double().numpy() for n in ("q", "k", "v", "dO")),
                                              W=8, rungs=FIB, alpha=alpha)
    assert abs(theta.grad.item() - dth_ref) <= 1e-3 * max(1.0, abs(dth_ref))


# ------------------------------------------- tensor-core backward edges --


@pytest.mark.parametrize("W", [0, 5, 13, 14, 17, 30])
def test_bf16_window_widths(W):
    """Window tiles beyond the first (W > 12) and windows narrower than the tile."""
    run(2, 160, "bf16", alpha=1.13, W=W, layer=4)


@pytest.mark.parametrize("T", [2, 29, 33, 97])
def test_bf16_short_and_ragged_sequences(T):
    """Sequences shorter than a tile and ragged last tiles (queries past T masked)."""
    run(3, T, "bf16", alpha=0.77, W=12, layer=6)


def test_bf16_without_rope_and_many_rungs():
    run(2, 200, "bf16", alpha=0.9, W=8, rope_theta=0.0, layer=8)
    rungs = tuple(range(9, 41))                       # 32 rungs: 8 groups of the ring
    run(1, 240, "bf16", alpha=1.07, W=8, rungs=rungs, layer=9)


def _oracle_grads(x, f, dtype, rope, **kw):
    """(dq, dk, dv, dalpha, dtheta) of the fp64 oracle for the kernels'
    inputs.  bf16 with RoPE: the oracle differentiates at the rows the kernels
    score (the bf16-rounded rotation of kernel_rotation) with its own rotation
    off, and its gradients with respect to those rotated rows are turned back
    into gradients of Q and K by the inverse rotation, in fp64."""
    if dtype == "bf16" and rope > 0:
        qr, kr = kernel_rotation(x["q"], rope), kernel_rotation(x["k"], rope)
        ref = oracle.backward(qr.double().numpy(), kr.double().numpy(), f["v"], f["dO"], rope_theta=0.0, **kw)
        return (oracle.rope(ref[0], rope, inverse=True), oracle.rope(ref[1], rope, inverse=True), ref[2],
                ref[3], ref[4], ref[5])
    return oracle.backward(f["q"], f["k"], f["v"], f["dO"], rope_theta=rope, **kw)


def _check_grads(got, ref, dtype, rungs=FIB):
    tol = TOL[dtype]
    for name, g, want in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        bound = tol["grad"] * max(1.0, float(np.abs(want).max()))
        err = max_abs(np64(g), want)
        assert err <= bound, (name, err, bound)
    check_dalpha_dtheta(float(got[3].item()), float(got[4].item()), ref[3], ref[4], dtype,
                        known_limit=cancellation_limit(rungs, ref[5], ref[3], dtype))


@pytest.mark.parametrize("dtype,rope", [("bf16", 0.0), ("bf16", 1e4), ("f32", 1e4)])
def test_sharp_softmax_gradients(dtype, rope):
    """Q and K scaled by 6 (scores spread over about 50 log2 units): the
    recomputed probabilities exp(s - LSE) are close to 0 or 1 and dS is large.
    bf16 with RoPE against the oracle at the kernels' rounded rotation (see
    _oracle_grads)."""
    x, _ = draw(2, 300, dtype, layer=32, with_dO=True)
    for n in ("q", "k"):
        x[n] = (x[n].float() * 6.0).to(x[n].dtype)
    f = {n: v.to(torch.float64).numpy() for n, v in x.items()}
    xd = to_dev(x)
    kw = dict(alpha=1.21, W=12, rungs=FIB)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], rope_theta=rope, **kw)
    got = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, rope_theta=rope, **kw)
    torch.cuda.synchronize()
    _check_grads(got, _oracle_grads(x, f, dtype, rope, **kw), dtype)


@pytest.mark.parametrize("dtype,scale,rope", [("bf16", 0.05, 1e4), ("bf16", 0.3, 0.0), ("bf16", 0.3, 1e4),
                                              ("f32", 0.2, 1e4)])
def test_explicit_softmax_scale_gradients(dtype, scale, rope):
    """dQ, dK, dV, dL/dalpha and dL/dtheta with a caller-given softmax scale."""
    x, f = draw(2, 150, dtype, layer=62, with_dO=True)
    xd = to_dev(x)
    kw = dict(alpha=0.83, W=12, rungs=FIB, scale=scale)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], rope_theta=rope, **kw)
    got = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, rope_theta=rope, **kw)
    torch.cuda.synchronize()
    _check_grads(got, _oracle_grads(x, f, dtype, rope, **kw), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fractional_unsorted_duplicate_base_offsets(dtype):
    """Any finite positive base offsets: fractional, given out of order, one
    repeated (the rung plan sorts by distance and keeps repeats as separate
    entries, as the oracle's key list does)."""
    rungs = (19.1, 2.5, 7.3, 7.3, 40.25, 13.0)
    ref = run(2, 140, dtype, alpha=1.11, W=8, rungs=rungs, layer=66)
    assert np.isfinite(ref[3])


def test_fractional_base_offsets_decode():
    rungs = (19.1, 2.5, 7.3, 7.3, 40.25, 13.0)
    x, f = draw(4, 120, "bf16", layer=67)
    pos = np.array([0, 9, 60, 119], dtype=np.int32)
    qd = torch.stack([x["q"][b, p] for b, p in enumerate(pos)])
    o, lse = api.sfa_decode(qd.cuda(), x["k"].cuda(), x["v"].cuda(), torch.from_numpy(pos).cuda(),
                            alpha=1.11, W=8, rungs=rungs)
    torch.cuda.synchronize()
    rows = np.stack([np.arange(4, dtype=np.int32), pos], axis=1)
    o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=8, rungs=rungs, alpha=1.11)
    assert max_abs(np64(o), o_ref) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse), lse_ref) <= TOL["bf16"]["lse"]
