"""Forward parity of the tcgen05 forward kernel (sfa_fwd_tc.cu, selected with
SFA_FORWARD_KERNEL=tc) against the fp64 oracle: small shapes element by
element (ragged tiles of 31 queries, every window width it takes, rung groups
of 4 up to 32 rungs, integer and fractional distances, rounded offsets), the
online maximum across rung groups at sharp scores, sampled rows at the
model-shape workload, and the multi-layer call with the next layer's keys
rotated inside the kernel."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, workloads
from oracle import oracle
from _helpers import TOL, draw, gpu_forward, kernel_rotation, max_abs, np64, sample_rows, to_dev

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE


@pytest.fixture(autouse=True)
def tc_kernel(monkeypatch):
    monkeypatch.setenv("SFA_FORWARD_KERNEL", "tc")


def check(B, T, *, alpha, W, rungs=FIB, layer=0, rope_theta=1e4, round_offsets=False, factor=1.0):
    x, _ = draw(B, T, "bf16", layer=layer)
    if factor != 1.0:
        for n in ("q", "k"):
            x[n] = (x[n].float() * factor).to(torch.bfloat16)
    f = {n: v.to(torch.float64).numpy() for n, v in x.items()}
    o, lse = gpu_forward(to_dev(x), alpha=alpha, W=W, rungs=rungs, rope_theta=rope_theta,
                         round_offsets=round_offsets)
    kw = dict(W=W, rungs=rungs, alpha=alpha, round_offsets=round_offsets)
    if rope_theta > 0 and factor != 1.0:
        # sharp scores: the oracle scores the rows the kernels score (the
        # bf16-rounded rotation)
        qr, kr = kernel_rotation(x["q"], rope_theta), kernel_rotation(x["k"], rope_theta)
        o_ref, lse_ref = oracle.forward(qr.double().numpy(), kr.double().numpy(), f["v"], rope_theta=0.0, **kw)
    else:
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], rope_theta=rope_theta, **kw)
    assert max_abs(np64(o), o_ref) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse), lse_ref) <= TOL["bf16"]["lse"]
    return lse_ref


@pytest.mark.parametrize("T", [1, 2, 30, 31, 32, 62, 63, 100, 333])
def test_ragged_tiles(T):
    check(2, T, alpha=1.13, W=12, layer=70)


@pytest.mark.parametrize("W", [0, 1, 5, 6, 8, 10, 12, 15, 16])
def test_window_widths(W):
    check(2, 160, alpha=0.87, W=W, layer=71)


@pytest.mark.parametrize("alpha", [0.5, 0.61, 1.0, 1.2345, 1.5])
def test_linear_range(alpha):
    check(2, 300, alpha=alpha, W=12, layer=72)


def test_pow2_base_and_rounded_offsets():
    check(2, 333, alpha=api.alpha_from_theta(0.3), W=8, rungs=api.pow2_base(333), layer=73)
    check(2, 333, alpha=1.37, W=12, round_offsets=True, layer=74)


def test_many_rungs_in_groups_of_four():
    """32 rungs: eight rung groups per tile, so the output is accumulated over
    eight probability-times-value steps with the running maximum carried
    across them."""
    check(1, 260, alpha=1.07, W=8, rungs=tuple(range(9, 41)), layer=75)


def test_without_rope():
    check(2, 200, alpha=0.9, W=12, rope_theta=0.0, layer=76)


@pytest.mark.parametrize("rope", [0.0, 1e4])
def test_sharp_scores_raise_the_maximum_across_groups(rope):
    """Q and K scaled by 6: a later rung group often beats the row maximum of
    the window and the first group by more than 2^8, so the output already in
    TMEM is rescaled."""
    lse_ref = check(2, 300, alpha=1.21, W=12, rope_theta=rope, factor=6.0, layer=77)
    assert float(np.median(lse_ref)) > 30.0


def test_model_shape_sampled_rows():
    wl = workloads.MODEL_SHAPE
    alphas, _ = wl.alphas()
    for layer in (0, 15):
        x, f = draw(wl.B, wl.T, wl.dtype, layer=layer)
        o, lse = gpu_forward(to_dev(x), alpha=alphas[layer], W=12, rungs=wl.rungs())
        rows = sample_rows(wl.B, wl.T, 256, seed=layer)
        o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=12, rungs=wl.rungs(),
                                             alpha=alphas[layer])
        assert max_abs(np64(o)[rows[:, 0], rows[:, 1]], o_ref) <= TOL["bf16"]["o"]
        assert max_abs(np64(lse)[rows[:, 0], rows[:, 1]], lse_ref) <= TOL["bf16"]["lse"]


def test_layers_match_single_layer_calls():
    """The multi-layer call (each launch rotating the next layer's keys) gives
    the same bits as one call per layer."""
    xs = [to_dev(draw(2, 130, "bf16", layer=78 + l)[0]) for l in range(3)]
    alphas = [0.8, 1.0, 1.3]
    outs, lses = api.sfa_forward_layers([x["q"] for x in xs], [x["k"] for x in xs], [x["v"] for x in xs],
                                        alphas=alphas, W=12)
    for l, x in enumerate(xs):
        o, lse = gpu_forward(x, alpha=alphas[l], W=12, rungs=FIB)
        assert torch.equal(outs[l], o) and torch.equal(lses[l], lse)


def test_agrees_with_the_mma_kernel(monkeypatch):
    x = to_dev(draw(4, 500, "bf16", layer=79)[0])
    o1, l1 = gpu_forward(x, alpha=1.17, W=12, rungs=FIB)
    monkeypatch.setenv("SFA_FORWARD_KERNEL", "mma")
    o2, l2 = gpu_forward(x, alpha=1.17, W=12, rungs=FIB)
    assert max_abs(np64(o1), np64(o2)) <= TOL["bf16"]["o"]
    assert max_abs(np64(l1), np64(l2)) <= TOL["bf16"]["lse"]
