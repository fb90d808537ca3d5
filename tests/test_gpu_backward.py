"""Backward parity: dQ, dK, dV, dalpha and dtheta from the CUDA path against the
fp64 oracle on the same seeded inputs (small sizes element by element, the
training-step workload at full size)."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs, workloads
from oracle import oracle
from _helpers import TOL, draw, max_abs, np64, to_dev

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
    da_ref, dth_ref = ref[3], ref[4]
    assert abs(float(dth.item()) - dth_ref) <= tol["dtheta"] * max(abs(dth_ref), 1e-3), (
        float(dth.item()), dth_ref)
    assert abs(float(da.item()) - da_ref) <= tol["dtheta"] * max(abs(da_ref), 1e-3)
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


@pytest.mark.parametrize("dtype,rope", [("bf16", 0.0), ("f32", 1e4)])
def test_sharp_softmax_gradients(dtype, rope):
    """Q and K scaled by 6 (scores spread over about 50 log2 units): the
    recomputed probabilities exp(s - LSE) are close to 0 or 1 and dS is large.
    bf16 without RoPE, so that both sides score the identical bf16 bytes."""
    x, _ = draw(2, 300, dtype, layer=32, with_dO=True)
    for n in ("q", "k"):
        x[n] = (x[n].float() * 6.0).to(x[n].dtype)
    f = {n: v.to(torch.float64).numpy() for n, v in x.items()}
    xd = to_dev(x)
    kw = dict(alpha=1.21, W=12, rungs=FIB, rope_theta=rope)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], **kw)
    dq, dk, dv, da, dth = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, **kw)
    torch.cuda.synchronize()
    ref = oracle.backward(f["q"], f["k"], f["v"], f["dO"], W=12, rungs=FIB, alpha=1.21, rope_theta=rope)
    tol = TOL[dtype]
    for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        err = max_abs(np64(got), want)
        bound = tol["grad"] * max(1.0, float(np.abs(want).max()))
        assert err <= bound, (name, err, bound)
    # dL/dalpha = sum_k f_k dL/dt_k: the bound scales with sum_k f_k |dL/dt_k|
    terms = float(np.sum(np.asarray(FIB, dtype=np.float64) * np.abs(ref[5])))
    assert abs(float(da.item()) - ref[3]) <= tol["dtheta"] * max(terms, abs(ref[3])) + 1e-6


@pytest.mark.parametrize("dtype,scale", [("bf16", 0.05), ("bf16", 0.3), ("f32", 0.2)])
def test_explicit_softmax_scale_gradients(dtype, scale):
    """dQ, dK, dV and dL/dalpha with a caller-given softmax scale."""
    x, f = draw(2, 150, dtype, layer=62, with_dO=True)
    xd = to_dev(x)
    kw = dict(alpha=0.83, W=12, rungs=FIB, scale=scale)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], **kw)
    dq, dk, dv, da, dth = api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, **kw)
    torch.cuda.synchronize()
    ref = oracle.backward(f["q"], f["k"], f["v"], f["dO"], W=12, rungs=FIB, alpha=0.83, scale=scale)
    tol = TOL[dtype]
    for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        bound = tol["grad"] * max(1.0, float(np.abs(want).max()))
        assert max_abs(np64(got), want) <= bound, name
    terms = float(np.sum(np.asarray(FIB, dtype=np.float64) * np.abs(ref[5])))
    assert abs(float(da.item()) - ref[3]) <= tol["dtheta"] * max(terms, abs(ref[3])) + 1e-6


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
