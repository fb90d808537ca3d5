"""Forward parity: the CUDA path through the C ABI against the fp64 oracle on
the same seeded inputs, element by element at sizes the oracle finishes in
seconds, and on sampled rows at the workloads' full sizes."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, workloads
from oracle import oracle
from _helpers import kernel_rotation, rope_rounding_bound, TOL, draw, gpu_forward, max_abs, np64, sample_rows, to_dev

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE


def check_full(B, T, dtype, *, alpha, W, rungs, layer=0, rope_theta=1e4):
    x, f = draw(B, T, dtype, layer=layer)
    o, lse = gpu_forward(to_dev(x), alpha=alpha, W=W, rungs=rungs, rope_theta=rope_theta)
    o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], W=W, rungs=rungs, alpha=alpha,
                                    rope_theta=rope_theta)
    eo, el = max_abs(np64(o), o_ref), max_abs(np64(lse), lse_ref)
    assert eo <= TOL[dtype]["o"], (eo, alpha, W)
    assert el <= TOL[dtype]["lse"], (el, alpha, W)
    return eo


def check_sampled(wl, layer, nrows=384):
    alphas, _ = wl.alphas()
    alpha, W = alphas[layer], wl.window(layer)
    x, f = draw(wl.B, wl.T, wl.dtype, layer=layer)
    o, lse = gpu_forward(to_dev(x), alpha=alpha, W=W, rungs=wl.rungs())
    rows = sample_rows(wl.B, wl.T, nrows, seed=layer)
    o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=W, rungs=wl.rungs(),
                                         alpha=alpha)
    og = np64(o)[rows[:, 0], rows[:, 1]]
    lg = np64(lse)[rows[:, 0], rows[:, 1]]
    assert max_abs(og, o_ref) <= TOL[wl.dtype]["o"]
    assert max_abs(lg, lse_ref) <= TOL[wl.dtype]["lse"]
    # properties that hold at any size: finite, rows are convex combinations
    on = np64(o)
    assert np.isfinite(on).all()
    vmax = np.abs(x["v"].float().numpy()).max()
    assert np.abs(on).max() <= vmax * (1 + 1e-2)


# ------------------------------------------------ element-wise, small sizes --


def test_tiny_fp32_alpha1():
    """B=1, T=256, W=8, alpha=1, fp32: within 1e-4 of the oracle."""
    check_full(1, 256, "f32", alpha=1.0, W=8, rungs=FIB)


@pytest.mark.parametrize("layer", [0, 3, 7, 11, 15])
def test_linear_stagger_small(layer):
    alpha = api.alpha_schedule("linear", 16)[layer]
    check_full(2, 300, "bf16", alpha=alpha, W=12, rungs=FIB, layer=layer)


@pytest.mark.parametrize("layer", [1, 2, 9])
def test_coprime_small(layer):
    alpha = api.alpha_schedule("coprime", 16, 7)[layer]
    check_full(1, 1200, "bf16", alpha=alpha, W=12, rungs=FIB, layer=layer)


@pytest.mark.parametrize("W", [6, 8, 10, 12])
def test_pow2_small(W):
    alpha = api.alpha_from_theta(0.21 * W - 1.9)
    check_full(2, 333, "bf16", alpha=alpha, W=W, rungs=api.pow2_base(333))


@pytest.mark.parametrize("alpha", [0.5, 0.51234, 1.0, 1.37, 1.5])
def test_fp32_fractional(alpha):
    check_full(2, 200, "f32", alpha=alpha, W=10, rungs=FIB, layer=4)


# ------------------------------------------------------------- edge cases --


def test_single_token_and_first_query():
    x, f = draw(3, 1, "bf16")
    o, lse = gpu_forward(to_dev(x), alpha=1.0, W=12, rungs=FIB)
    for h in range(8):
        assert torch.equal(o[:, 0, h].cpu(), x["v"][:, 0, h // 4])
    ref = (x["q"].double()[:, 0] * x["k"].double()[:, 0].repeat_interleave(4, 1)).sum(-1) / 8
    assert max_abs(np64(lse[:, 0]), ref.numpy()) <= TOL["bf16"]["lse"]


def test_empty_inputs_launch_nothing():
    z = torch.empty((0, 16, 8, 64), dtype=torch.bfloat16, device="cuda")
    zk = torch.empty((0, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    n0 = api.launch_count()
    o, lse = api.sfa_forward(z, zk, zk, alpha=1.0, W=12)
    assert o.shape == z.shape and api.launch_count() == n0
    z = torch.empty((2, 0, 8, 64), dtype=torch.bfloat16, device="cuda")
    zk = torch.empty((2, 0, 2, 64), dtype=torch.bfloat16, device="cuda")
    api.sfa_forward(z, zk, zk, alpha=1.0, W=12)
    assert api.launch_count() == n0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_window_only_and_dense_limit(dtype):
    check_full(2, 96, dtype, alpha=0.8, W=12, rungs=())          # no rungs at all
    check_full(2, 96, dtype, alpha=0.8, W=200, rungs=FIB)        # W >= T: causal dense
    check_full(2, 96, dtype, alpha=1.3, W=0, rungs=FIB)          # self + rungs only


def test_rungs_all_masked_short_sequence():
    check_full(3, 20, "bf16", alpha=1.5, W=12, rungs=FIB)


def test_without_rope():
    check_full(2, 128, "f32", alpha=0.91, W=8, rungs=FIB, rope_theta=0.0)


def test_deterministic_and_status_word():
    x, _ = draw(2, 257, "bf16", layer=5)
    xd = to_dev(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n0 = api.launch_count()
    o1, l1 = gpu_forward(xd, alpha=1.17, W=12, rungs=FIB, status=status)
    o2, l2 = gpu_forward(xd, alpha=1.17, W=12, rungs=FIB, status=status)
    assert api.launch_count() - n0 == 4          # RoPE on the keys + attention, per call
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert api.sfa_read_status(status) == 0


# -------------------------------------------- full sizes, sampled rows --


@pytest.mark.parametrize("layer", [0, 7, 15])
def test_model_shape_full(layer):
    check_sampled(workloads.MODEL_SHAPE, layer)


@pytest.mark.parametrize("layer", [0, 5])
def test_extrapolation_full(layer):
    check_sampled(workloads.EXTRAPOLATION, layer)


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_pow2_full(layer):
    check_sampled(workloads.POW2, layer)


def test_long_forward_full():
    check_sampled(workloads.LONG_FORWARD, 3, nrows=256)


# ---------------------------------------- tensor-core path specific shapes --


@pytest.mark.parametrize("W", [0, 1, 5, 13, 14, 15, 16, 17, 22, 30, 31])
def test_window_widths(W):
    """One or two window M tiles (W + 2 rows), and the fp32-arithmetic kernel
    beyond W = 30."""
    check_full(2, 200, "bf16", alpha=1.23, W=W, rungs=FIB, layer=W)


def test_many_rungs_wrap_the_slot_ring():
    """32 rungs (the maximum): eight groups of four rungs per query tile, so
    the two group slots of the ring are reused four times each."""
    base = [13 + 7 * k for k in range(32)]
    check_full(2, 300, "bf16", alpha=1.1, W=12, rungs=base, layer=21)


@pytest.mark.parametrize("T", [2, 31, 32, 33, 65, 97])
def test_short_and_ragged_sequences(T):
    check_full(3, T, "bf16", alpha=0.77, W=12, rungs=FIB, layer=T)


def test_integer_offsets_bf16():
    """alpha = 1: every t = 0 (rows i - f only)."""
    check_full(2, 512, "bf16", alpha=1.0, W=8, rungs=FIB, layer=30)


def test_without_rope_bf16():
    check_full(2, 160, "bf16", alpha=0.91, W=12, rungs=FIB, rope_theta=0.0)


@pytest.mark.parametrize("alpha,W", [(1.0, 0), (1.0, 12), (2.0, 6), (3.0, 20), (1.0, 30)])
def test_integer_offset_tiles(alpha, W):
    """Every kept distance an integer (t = 0): the rung tiles that read rows a
    only (two query pairs per tile), with ragged tiles and partial groups."""
    check_full(2, 333, "bf16", alpha=alpha, W=W, rungs=FIB, layer=40 + W)


def test_integer_offset_tiles_pow2_base():
    check_full(3, 517, "bf16", alpha=1.0, W=8, rungs=api.pow2_base(517), layer=47)


# ------------------------------------------------- sharp softmax (rescales) --


def _scaled(B, T, dtype, layer, factor, with_dO=False):
    """Seeded inputs with Q and K multiplied by ``factor`` (rounded once to the
    dtype), and their exact fp64 copies."""
    x, _ = draw(B, T, dtype, layer=layer, with_dO=with_dO)
    for n in ("q", "k"):
        x[n] = (x[n].float() * factor).to(x[n].dtype)
    return x, {n: v.to(torch.float64).numpy() for n, v in x.items()}


def _check_against_oracle(x, f, o, lse, dtype, rope, **kw):
    """O and LSE of the kernels against the fp64 oracle, to the dtype's
    tolerance.  bf16 with RoPE: the oracle scores the rows the kernels score
    (the bf16-rounded rotation, restated in kernel_rotation) with its own
    rotation off; the rounding itself is then checked on the LSE against the
    bound it implies (rope_rounding_bound) with the oracle's exact rotation."""
    if dtype == "bf16" and rope > 0:
        qr, kr = kernel_rotation(x["q"], rope), kernel_rotation(x["k"], rope)
        o_ref, lse_ref = oracle.forward(qr.double().numpy(), kr.double().numpy(), f["v"], rope_theta=0.0, **kw)
        o_ex, lse_ex = oracle.forward(f["q"], f["k"], f["v"], rope_theta=rope, **kw)
        scale = kw.get("scale") or 0.125
        delta = rope_rounding_bound(x["q"], x["k"], scale, rope)
        assert np.all(np.abs(np64(lse) - lse_ex) <= delta + TOL[dtype]["lse"])
    else:
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], rope_theta=rope, **kw)
    assert max_abs(np64(o), o_ref) <= TOL[dtype]["o"]
    assert max_abs(np64(lse), lse_ref) <= TOL[dtype]["lse"]
    return o_ref, lse_ref


@pytest.mark.parametrize("dtype,rope", [("bf16", 0.0), ("bf16", 1e4), ("f32", 1e4)])
def test_sharp_softmax_raises_the_running_max(dtype, rope):
    """Q and K scaled by 6: scores spread over about 50 log2 units, so the
    running max is raised many times inside the window and rung tiles (the
    lazy rescale fires whenever a score beats the max by 2^8).  With RoPE the
    bf16 kernels round the rotated rows to bf16 (a score moves by up to about
    scale |q| |k| 2^-7), so the oracle is given those rows (see
    _check_against_oracle)."""
    x, f = _scaled(2, 300, dtype, 31, 6.0)
    o, lse = gpu_forward(to_dev(x), alpha=1.21, W=12, rungs=FIB, rope_theta=rope)
    _, lse_ref = _check_against_oracle(x, f, o, lse, dtype, rope, W=12, rungs=FIB, alpha=1.21)
    # the reference itself is sharp: most rows put over half their weight on one entry
    assert float(np.median(lse_ref)) > 30.0


@pytest.mark.parametrize("dtype,scale,rope", [("bf16", 0.05, 1e4), ("bf16", 0.15, 1e4), ("bf16", 0.3, 0.0),
                                              ("bf16", 0.3, 1e4), ("f32", 0.2, 1e4)])
def test_explicit_softmax_scale(dtype, scale, rope):
    """A caller-given softmax scale (sfa_params.scale) instead of 1/sqrt(64),
    with and without RoPE."""
    x, f = draw(2, 150, dtype, layer=61)
    o, lse = gpu_forward(to_dev(x), alpha=1.17, W=12, rungs=FIB, scale=scale, rope_theta=rope)
    _check_against_oracle(x, f, o, lse, dtype, rope, W=12, rungs=FIB, alpha=1.17, scale=scale)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_without_lse_output(dtype):
    """LSE is optional (a NULL pointer): the output is the same as with it."""
    x, f = draw(2, 150, dtype, layer=64)
    xd = to_dev(x)
    o1, _ = gpu_forward(xd, alpha=0.97, W=12, rungs=FIB)
    o2, l2 = gpu_forward(xd, alpha=0.97, W=12, rungs=FIB, need_lse=False)
    assert l2 is None
    assert torch.equal(o1, o2)
    o_ref, _ = oracle.forward(f["q"], f["k"], f["v"], W=12, rungs=FIB, alpha=0.97)
    assert max_abs(np64(o2), o_ref) <= TOL[dtype]["o"]


def test_layers_and_decode_without_lse_output():
    """The multi-layer forward and the decode with no LSE output give the same
    outputs as with it."""
    xs = [draw(2, 130, "bf16", layer=65 + l)[0] for l in range(3)]
    xd = [to_dev(x) for x in xs]
    alphas = [0.8, 1.0, 1.3]
    a_outs, _ = api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd], [x["v"] for x in xd],
                                       alphas=alphas, W=12)
    b_outs, b_lses = api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd],
                                            [x["v"] for x in xd], alphas=alphas, W=12, need_lse=False)
    torch.cuda.synchronize()
    assert b_lses is None
    for a, b in zip(a_outs, b_outs):
        assert torch.equal(a, b)
    pos = torch.tensor([0, 129], dtype=torch.int32, device="cuda")
    q = torch.stack([xd[0]["q"][0, 0], xd[0]["q"][1, 129]])
    o1, _ = api.sfa_decode(q, xd[0]["k"], xd[0]["v"], pos, alpha=0.8, W=12)
    o2, l2 = api.sfa_decode(q, xd[0]["k"], xd[0]["v"], pos, alpha=0.8, W=12, need_lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(o1, o2)
