"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test names what fixes the expected value: a value printed by the paper
(tests/golden/paper_tables.txt), a library routine the special case reduces to
(torch's scaled_dot_product_attention in fp64), a closed form, an invariant, or
a finite difference.  Paper: "Depth-Staggered Fibonacci Spacing for Sparse
Attention" (arXiv 2606.28560), section 2 "Method".
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle
from fibonacci_spaced_sparse_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paper_tables.txt")


def golden():
    out = {}
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = [s.strip() for s in line.split("=", 1)]
            vals = [float(x) for x in val.split()]
            out[key] = vals if len(vals) > 1 else vals[0]
    return out


def f64(x):
    return x.to(torch.float64).numpy()


def union_mask(T, W, dists):
    """Boolean [T, T] mask: key j allowed for query i iff i - j is a window
    distance 0..W or one of the (integer) rung distances ``dists``."""
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    dd = i - j
    m = (dd >= 0) & (dd <= W)
    for d in dists:
        m |= dd == d
    return m


def sdpa_masked(qh, kh, v, mask, scale):
    """Library attention (torch SDPA, fp64, CPU) with a boolean mask and the
    GQA head map h -> h // G; also returns the log-sum-exp of the masked scores."""
    q = torch.from_numpy(qh).permute(0, 2, 1, 3)          # B,H,T,D
    k = torch.from_numpy(kh).permute(0, 2, 1, 3)
    vv = torch.from_numpy(v).permute(0, 2, 1, 3)
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    vv = vv.repeat_interleave(G, dim=1)
    m = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, vv, attn_mask=m, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    s = s.masked_fill(~m, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.permute(0, 2, 1).numpy()


FIB = oracle.FIBONACCI_BASE


# ------------------------------------------------------------- tables ----


def test_tables_match_printed_values():
    g = golden()
    assert list(FIB) == [int(x) for x in g["fibonacci_base"]]
    assert len(FIB) == g["fibonacci_K"] == 15
    assert FIB[-1] == g["fibonacci_last"] == 987
    # section 4.2: consecutive rungs are spaced by the rung two below
    for k in range(2, len(FIB) - 1):
        assert FIB[k + 1] - FIB[k] == FIB[k - 1]
    assert oracle.alpha_from_theta(0.0) == g["alpha_at_init"]
    for th in (-50.0, -3.0, 0.3, 4.0, 50.0):
        a = oracle.alpha_from_theta(th)
        assert g["alpha_min"] <= a <= g["alpha_max"]
    lin = oracle.schedule_linear(int(g["layers"]))
    assert lin[0] == g["linear_first"] and lin[-1] == g["linear_last"]
    assert np.all(np.diff(lin) > 0)
    assert oracle.schedule_fixed(16) == [1.0] * 16
    p2 = oracle.pow2_base(4096)
    assert all(x in p2 for x in g["pow2_new_offsets_at_4096"])
    assert max(p2) < 4096 and 1024 not in oracle.pow2_base(1024)
    assert oracle.pow2_base(1024) == tuple(2 ** k for k in range(10))


def test_coprime_schedule_is_permutation_of_ramp():
    g = golden()
    L, S = int(g["layers"]), int(g["coprime_stride"])
    assert math.gcd(S, L) == 1
    lin = oracle.schedule_linear(L)
    cop = oracle.schedule_coprime(L, S)
    assert sorted(cop) == sorted(lin)                      # same multiset
    perm = [(S * l) % L for l in range(L)]
    assert sorted(perm) == list(range(L))                  # a permutation
    for l in range(L):
        assert cop[l] == lin[perm[l]]
    # adjacent layers land 7/15 or 9/15 apart on the ramp
    gaps = sorted({round(abs(cop[l + 1] - cop[l]) * 15) for l in range(L - 1)})
    assert gaps == [7, 9]


def test_learned_schedule_init_and_monotone():
    assert oracle.schedule_learned([0.0, 0.0]) == [1.0, 1.0]
    a = oracle.schedule_learned(np.linspace(-6, 6, 13))
    assert np.all(np.diff(a) > 0)


# --------------------------------------------------------------- RoPE ----


def test_rope_angles_closed_form():
    """Per pair (m, m+32) the rotation at position p is by p * 1e4^(-2m/64):
    recovered from cos = <y, x> and sin = y[m+32] x[m] - y[m] x[m+32]."""
    rng = np.random.default_rng(0)
    T, D = 300, 64
    x = np.broadcast_to(rng.standard_normal(D), (1, T, 1, D)).copy()
    y = oracle.rope(x, 1e4)
    h = D // 2
    for p in (0, 1, 7, 123, 299):
        for m in range(h):
            r2 = x[0, p, 0, m] ** 2 + x[0, p, 0, m + h] ** 2
            c = (y[0, p, 0, m] * x[0, p, 0, m] + y[0, p, 0, m + h] * x[0, p, 0, m + h]) / r2
            s = (y[0, p, 0, m + h] * x[0, p, 0, m] - y[0, p, 0, m] * x[0, p, 0, m + h]) / r2
            ang = p * 10000.0 ** (-2.0 * m / D)
            assert abs(c - math.cos(ang)) < 1e-12 and abs(s - math.sin(ang)) < 1e-12


def test_rope_relative_and_inverse():
    rng = np.random.default_rng(1)
    T, D = 64, 64
    q = rng.standard_normal((1, T, 1, D))
    k = rng.standard_normal((1, T, 1, D))
    q2 = np.roll(q, 5, axis=1)   # same vectors five positions later
    k2 = np.roll(k, 5, axis=1)
    a = np.einsum("d,d->", oracle.rope(q)[0, 20, 0], oracle.rope(k)[0, 11, 0])
    b = np.einsum("d,d->", oracle.rope(q2)[0, 25, 0], oracle.rope(k2)[0, 16, 0])
    assert abs(a - b) < 1e-10
    back = oracle.rope(oracle.rope(q), inverse=True)
    assert np.max(np.abs(back - q)) < 1e-12
    assert np.allclose(np.linalg.norm(oracle.rope(q), axis=-1), np.linalg.norm(q, axis=-1))


# ------------------------------------------------------ forward pins ----


def _inputs(B, T, dtype=torch.float32, layer=0):
    t = inputs.qkv(B, T, dtype=dtype, layer=layer, with_dO=True)
    return {k: f64(v) for k, v in t.items()}


def test_alpha1_equals_dense_boolean_mask():
    """At alpha = 1 every rung distance is an integer, and the sparse attention
    equals dense attention under the boolean mask of the union set (section 2,
    "Implementation notes": the fused boolean-mask path is numerically the
    same).  Tiny fp32 workload: B=1, T=256, W=8."""
    x = _inputs(1, 256)
    W = 8
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=FIB, alpha=1.0)
    qh, kh = oracle.rope(x["q"]), oracle.rope(x["k"])
    mask = union_mask(256, W, [f for f in FIB if f > W])
    o_ref, lse_ref = sdpa_masked(qh, kh, x["v"], mask, 1 / 8)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


@pytest.mark.parametrize("W", [0, 6, 12])
def test_alpha1_dense_mask_batched(W):
    x = _inputs(2, 160, layer=3)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=FIB, alpha=1.0)
    mask = union_mask(160, W, [f for f in FIB if f > W])
    o_ref, lse_ref = sdpa_masked(oracle.rope(x["q"]), oracle.rope(x["k"]), x["v"], mask, 1 / 8)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_explicit_scale_equals_dense_mask_with_that_scale(scale):
    """A caller-given softmax scale multiplies every score: at alpha = 1 the
    sparse attention equals masked dense attention at that scale."""
    x = _inputs(1, 160, layer=5)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=6, rungs=FIB, alpha=1.0, scale=scale)
    mask = union_mask(160, 6, [f for f in FIB if f > 6])
    o_ref, lse_ref = sdpa_masked(oracle.rope(x["q"]), oracle.rope(x["k"]), x["v"], mask, scale)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_lerp_limit_from_below_is_plain_gather():
    """As alpha -> 1 from below, each rung's fraction t -> 1 and the lerp tends
    to the plain gather of row i - f_k (weight t on the row at distance n + 1)."""
    x = _inputs(1, 200, layer=1)
    W = 8
    eps = 2.0 ** -32
    o, _ = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=FIB, alpha=1.0 - eps, d_fp32=False)
    mask = union_mask(200, W, [f for f in FIB if f > W])
    o_ref, _ = sdpa_masked(oracle.rope(x["q"]), oracle.rope(x["k"]), x["v"], mask, 1 / 8)
    assert np.max(np.abs(o - o_ref)) < 1e-6


def test_lerp_limit_from_above_shifts_the_mask():
    """As alpha -> 1 from above, t -> 0 and the lerp tends to row i - f_k, but
    ceil(d_k) = f_k + 1, so the first query that may use rung k is f_k + 1."""
    x = _inputs(1, 200, layer=2)
    W = 10                      # no base offset equals W (see the next test)
    eps = 2.0 ** -32
    o, _ = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=FIB, alpha=1.0 + eps, d_fp32=False)
    T = 200
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    dd = i - j
    mask = (dd >= 0) & (dd <= W)
    for f in FIB:
        if f > W:
            mask |= (dd == f) & (i >= f + 1)
    o_ref, _ = sdpa_masked(oracle.rope(x["q"]), oracle.rope(x["k"]), x["v"], mask, 1 / 8)
    assert np.max(np.abs(o - o_ref)) < 1e-6


def test_rung_just_outside_window_duplicates_a_window_row():
    """W < d_k < W + 1 keeps the rung although its row i - floor(d_k) = i - W is
    also a window row: the two stay separate entries.  With t -> 0 the rung
    entry tends to a second copy of key i - W, i.e. dense attention in which
    that key's logit carries an extra log(2) (two equal terms in the softmax)."""
    T, W = 64, 8
    x = _inputs(1, T, layer=15)
    eps = 2.0 ** -36
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=[8], alpha=1.0 + eps, d_fp32=False)
    qh, kh = oracle.rope(x["q"]), oracle.rope(x["k"])
    q = torch.from_numpy(qh).permute(0, 2, 1, 3)
    k = torch.from_numpy(kh).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    v = torch.from_numpy(x["v"]).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    i = np.arange(T)[:, None]
    dd = i - np.arange(T)[None, :]
    allowed = (dd >= 0) & (dd <= W)
    bias = np.where(allowed, 0.0, -np.inf)
    bias = bias + np.where((dd == W) & (i >= W + 1), math.log(2.0), 0.0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=torch.from_numpy(bias), scale=1 / 8)
    assert np.max(np.abs(o - ref.permute(0, 2, 1, 3).numpy())) < 1e-6


def test_repeated_rung_is_a_second_entry():
    """A base offset given twice is two entries of the key list: at alpha = 1
    (integer distance 13, beyond W = 6) that key's logit carries an extra
    log(2) in dense attention, from the position where the rung applies."""
    T, W = 80, 6
    x = _inputs(1, T, layer=16)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=[13, 13], alpha=1.0)
    qh, kh = oracle.rope(x["q"]), oracle.rope(x["k"])
    q = torch.from_numpy(qh).permute(0, 2, 1, 3)
    k = torch.from_numpy(kh).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    v = torch.from_numpy(x["v"]).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    dd = np.arange(T)[:, None] - np.arange(T)[None, :]
    bias = np.where(((dd >= 0) & (dd <= W)) | (dd == 13), 0.0, -np.inf)
    bias = bias + np.where(dd == 13, math.log(2.0), 0.0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=torch.from_numpy(bias), scale=1 / 8)
    assert np.max(np.abs(o - ref.permute(0, 2, 1, 3).numpy())) < 1e-12


def test_order_of_base_offsets_does_not_matter():
    """The key list is a set of entries: listing the base offsets in another
    order changes only the summation order (fractional offsets, alpha != 1)."""
    x = _inputs(2, 120, layer=17)
    a = (2.5, 7.3, 13.0, 19.1, 40.25)
    b = (19.1, 2.5, 40.25, 13.0, 7.3)
    oa, la = oracle.forward(x["q"], x["k"], x["v"], W=8, rungs=a, alpha=1.11)
    ob, lb = oracle.forward(x["q"], x["k"], x["v"], W=8, rungs=b, alpha=1.11)
    assert np.max(np.abs(oa - ob)) < 1e-12 and np.max(np.abs(la - lb)) < 1e-12
    ga = oracle.backward(x["q"], x["k"], x["v"], x["dO"], W=8, rungs=a, alpha=1.11)
    gb = oracle.backward(x["q"], x["k"], x["v"], x["dO"], W=8, rungs=b, alpha=1.11)
    for u, w in zip(ga[:3], gb[:3]):
        assert np.max(np.abs(u - w)) < 1e-11
    assert abs(ga[3] - gb[3]) < 1e-9 * max(1.0, abs(ga[3]))


def test_integer_rungs_at_alpha_1p5_even_offsets():
    """alpha = 1.5 makes the even offsets integral (3, 12, 51, 216, 915) and the
    odd ones half-integral; with W = 12, every rung is integral or dropped when
    the base holds only even offsets beyond the window, so the result is a
    dense boolean-mask attention again."""
    x = _inputs(1, 256, layer=4)
    W = 12
    base = [2, 8, 34, 144]               # distances 3, 12 (dropped), 51, 216
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=base, alpha=1.5)
    mask = union_mask(256, W, [51, 216])
    o_ref, lse_ref = sdpa_masked(oracle.rope(x["q"]), oracle.rope(x["k"]), x["v"], mask, 1 / 8)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_dense_limit_is_causal_attention():
    """W >= T - 1: every rung is dropped or masked and the result is plain
    causal attention (torch SDPA with is_causal)."""
    T = 96
    x = _inputs(2, T, layer=5)
    o, _ = oracle.forward(x["q"], x["k"], x["v"], W=T - 1, rungs=FIB, alpha=0.73)
    q = torch.from_numpy(oracle.rope(x["q"])).permute(0, 2, 1, 3)
    k = torch.from_numpy(oracle.rope(x["k"])).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    v = torch.from_numpy(x["v"]).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1 / 8)
    assert np.max(np.abs(o - ref.permute(0, 2, 1, 3).numpy())) < 1e-12
    # without rotation the oracle reads the raw inputs
    o2, _ = oracle.forward(x["q"], x["k"], x["v"], W=T + 5, rungs=FIB, alpha=1.2, rope_theta=0.0)
    q = torch.from_numpy(x["q"]).permute(0, 2, 1, 3)
    k = torch.from_numpy(x["k"]).permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    ref2 = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1 / 8)
    assert np.max(np.abs(o2 - ref2.permute(0, 2, 1, 3).numpy())) < 1e-12


def test_first_query_sees_only_itself():
    """Query 0 has only its own key (no rung reaches before the start), so
    O = v_0 and LSE = scale * q_0 . k_0 (RoPE at position 0 is the identity)."""
    x = _inputs(3, 40, layer=6)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=6, rungs=FIB, alpha=0.61)
    for b in range(3):
        for h in range(8):
            g = h // 4
            assert np.max(np.abs(o[b, 0, h] - x["v"][b, 0, g])) < 1e-14
            assert abs(lse[b, 0, h] - x["q"][b, 0, h] @ x["k"][b, 0, g] / 8) < 1e-12


def test_rungs_inside_window_are_dropped():
    """alpha = 1.5, W = 12: offsets 1, 2, 3, 5, 8 map to 1.5 .. 12 <= W and are
    dropped, so removing them from the table changes nothing."""
    x = _inputs(1, 300, layer=7)
    a = oracle.forward(x["q"], x["k"], x["v"], W=12, rungs=FIB, alpha=1.5)
    b = oracle.forward(x["q"], x["k"], x["v"], W=12, rungs=FIB[5:], alpha=1.5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_causality_and_prefix_invariance():
    x = _inputs(1, 128, layer=8)
    kw = dict(W=10, rungs=FIB, alpha=0.87)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], **kw)
    k2, v2 = x["k"].copy(), x["v"].copy()
    k2[:, 70:] += 3.0
    v2[:, 70:] -= 2.0
    o2, _ = oracle.forward(x["q"], k2, v2, **kw)
    assert np.array_equal(o[:, :70], o2[:, :70])
    assert not np.allclose(o[:, 70:], o2[:, 70:])
    o3, lse3 = oracle.forward(x["q"][:, :50], x["k"][:, :50], x["v"][:, :50], **kw)
    assert np.max(np.abs(o3 - o[:, :50])) < 1e-14


def test_forward_rows_matches_full():
    x = _inputs(2, 128, layer=9)
    kw = dict(W=12, rungs=FIB, alpha=1.37)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], **kw)
    rows = [(0, 0), (1, 127), (0, 64), (1, 13)]
    o_r, lse_r = oracle.forward_rows(x["q"], x["k"], x["v"], rows, **kw)
    for n, (b, i) in enumerate(rows):
        assert np.array_equal(o_r[n], o[b, i]) and np.array_equal(lse_r[n], lse[b, i])


def test_fp32_rung_distance_rule():
    """d_k is one fp32 multiply: alpha = 0.1000000005 times 130 rounds to
    exactly 13.0 in fp32 but is 13.000000065 in fp64, which decides whether the
    rung lies on the window edge W = 13 (dropped) or just outside (kept)."""
    x = _inputs(1, 64, layer=10)
    a = 0.1000000005
    a32 = oracle.forward(x["q"], x["k"], x["v"], W=13, rungs=[130], alpha=a, d_fp32=True)
    a64 = oracle.forward(x["q"], x["k"], x["v"], W=13, rungs=[130], alpha=a, d_fp32=False)
    none = oracle.forward(x["q"], x["k"], x["v"], W=13, rungs=[], alpha=a)
    assert np.float32(np.float32(a) * np.float32(130.0)) == np.float32(13.0)
    assert a * 130.0 > 13.0
    assert np.array_equal(a32[0], none[0])
    assert not np.array_equal(a64[0], none[0])


# ------------------------------------------------------ backward pins ----


def _loss(x, dO, **kw):
    o, _ = oracle.forward(x["q"], x["k"], x["v"], **kw)
    return float(np.sum(o * dO))


def _safe_alpha(alpha, W, base, h):
    for f in base:
        for a in (alpha - h, alpha + h):
            d = a * f
            assert abs(d - round(d)) > 1e-3 and abs(d - W) > 1e-3
    return alpha


def test_dalpha_finite_difference():
    """dL/dalpha (through the lerp fraction) against a central difference of
    the fp64 forward; no distance crosses an integer or the window edge."""
    x = _inputs(1, 48, layer=11)
    base = FIB[:10]
    W = 4
    alpha = _safe_alpha(0.8137, W, base, 1e-4)
    kw = dict(W=W, rungs=base, d_fp32=False)
    _, _, _, da, dth, dt = oracle.backward(x["q"], x["k"], x["v"], x["dO"], alpha=alpha, **kw)
    h = 1e-5
    fd = (_loss(x, x["dO"], alpha=alpha + h, **kw) - _loss(x, x["dO"], alpha=alpha - h, **kw)) / (2 * h)
    assert abs(da - fd) <= 1e-6 * max(1.0, abs(fd))
    assert abs(dth - da * (alpha - 0.5) * (1.5 - alpha)) < 1e-12 * max(1.0, abs(da))


def test_dtheta_finite_difference():
    """dL/dtheta with alpha = 0.5 + sigmoid(theta), against a central difference
    taken in theta itself."""
    x = _inputs(1, 40, layer=12)
    base = FIB[:9]
    W = 3
    theta = -0.437
    alpha = oracle.alpha_from_theta(theta)
    _safe_alpha(alpha, W, base, 1e-4)
    kw = dict(W=W, rungs=base, d_fp32=False)
    _, _, _, da, dth, _ = oracle.backward(x["q"], x["k"], x["v"], x["dO"], alpha=alpha, **kw)
    h = 1e-5
    lp = _loss(x, x["dO"], alpha=oracle.alpha_from_theta(theta + h), **kw)
    lm = _loss(x, x["dO"], alpha=oracle.alpha_from_theta(theta - h), **kw)
    fd = (lp - lm) / (2 * h)
    assert abs(dth - fd) <= 1e-6 * max(1.0, abs(fd))


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_input_gradients_finite_difference(which):
    x = _inputs(1, 36, layer=13)
    base = FIB[:9]
    W = 3
    alpha = _safe_alpha(1.2371, W, base, 0.0)
    kw = dict(W=W, rungs=base, alpha=alpha, d_fp32=False)
    dq, dk, dv, _, _, _ = oracle.backward(x["q"], x["k"], x["v"], x["dO"], **kw)
    grad = {"q": dq, "k": dk, "v": dv}[which]
    rng = np.random.default_rng(3)
    shp = x[which].shape
    h = 1e-6
    for _ in range(12):
        idx = tuple(int(rng.integers(0, s)) for s in shp)
        xp = {k: v.copy() for k, v in x.items()}
        xm = {k: v.copy() for k, v in x.items()}
        xp[which][idx] += h
        xm[which][idx] -= h
        fd = (_loss(xp, x["dO"], **kw) - _loss(xm, x["dO"], **kw)) / (2 * h)
        assert abs(grad[idx] - fd) <= 1e-7 * max(1.0, abs(fd)), (idx, grad[idx], fd)


@pytest.mark.parametrize("scale", [1 / 8, 0.3])
def test_backward_alpha1_matches_autograd_dense_mask(scale):
    """At alpha = 1 the input gradients equal autograd through torch SDPA with
    the union boolean mask (fp64), with RoPE undone by the chain rule; also at
    a caller-given softmax scale."""
    T, W = 96, 8
    x = _inputs(1, T, layer=14)
    dq, dk, dv, _, _, _ = oracle.backward(x["q"], x["k"], x["v"], x["dO"], W=W, rungs=FIB, alpha=1.0,
                                          scale=scale)
    mask = torch.from_numpy(union_mask(T, W, [f for f in FIB if f > W]))
    qh = torch.from_numpy(oracle.rope(x["q"])).requires_grad_(True)
    kh = torch.from_numpy(oracle.rope(x["k"])).requires_grad_(True)
    v = torch.from_numpy(x["v"]).requires_grad_(True)
    q_ = qh.permute(0, 2, 1, 3)
    k_ = kh.permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    v_ = v.permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q_, k_, v_, attn_mask=mask, scale=scale)
    (o.permute(0, 2, 1, 3) * torch.from_numpy(x["dO"])).sum().backward()
    dq_ref = oracle.rope(qh.grad.numpy(), inverse=True)
    dk_ref = oracle.rope(kh.grad.numpy(), inverse=True)
    assert np.max(np.abs(dq - dq_ref)) < 1e-11
    assert np.max(np.abs(dk - dk_ref)) < 1e-11
    assert np.max(np.abs(dv - v.grad.numpy())) < 1e-11


# ------------------------------------------- rounded (integer) offsets ----


def _rounded_dists(alpha, W, base):
    """fl32(alpha) * fl32(f) rounded to the nearest integer, halves up, kept
    when beyond the window -- computed here without the oracle."""
    d = np.float32(alpha) * np.asarray(base, dtype=np.float32)
    r = np.floor(d.astype(np.float64) + 0.5).astype(int)
    return sorted(int(x) for x in r if x > W)


@pytest.mark.parametrize("alpha,W", [(1.37, 8), (1.0, 6), (1.5, 12), (2.2, 0)])
def test_round_offsets_equals_dense_mask(alpha, W):
    """With every distance rounded ("static schedules have integer offsets",
    section 2 "Implementation notes") the attention is dense attention under
    the boolean mask of the window and the rounded distances (alpha >= 1
    keeps the rounded distances distinct)."""
    T = 200
    x = _inputs(2, T, layer=15)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], W=W, rungs=FIB, alpha=alpha,
                            round_offsets=True)
    mask = union_mask(T, W, _rounded_dists(alpha, W, FIB))
    o_ref, lse_ref = sdpa_masked(oracle.rope(x["q"]), oracle.rope(x["k"]), x["v"], mask, 1 / 8)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_round_offsets_no_change_at_integer_alpha():
    x = _inputs(1, 180, layer=16)
    a = oracle.forward(x["q"], x["k"], x["v"], W=8, rungs=FIB, alpha=1.0, round_offsets=True)
    b = oracle.forward(x["q"], x["k"], x["v"], W=8, rungs=FIB, alpha=1.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_round_offsets_backward_matches_autograd_and_dalpha_is_zero():
    """Rounded distances do not depend on alpha (zero derivative), and the
    input gradients are those of dense attention under the rounded mask."""
    T, W, alpha = 96, 8, 1.29
    x = _inputs(1, T, layer=17)
    dq, dk, dv, da, dth, _ = oracle.backward(x["q"], x["k"], x["v"], x["dO"], W=W, rungs=FIB,
                                             alpha=alpha, round_offsets=True)
    assert da == 0.0 and dth == 0.0
    mask = torch.from_numpy(union_mask(T, W, _rounded_dists(alpha, W, FIB)))
    qh = torch.from_numpy(oracle.rope(x["q"])).requires_grad_(True)
    kh = torch.from_numpy(oracle.rope(x["k"])).requires_grad_(True)
    v = torch.from_numpy(x["v"]).requires_grad_(True)
    q_ = qh.permute(0, 2, 1, 3)
    k_ = kh.permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    v_ = v.permute(0, 2, 1, 3).repeat_interleave(4, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q_, k_, v_, attn_mask=mask, scale=1 / 8)
    (o.permute(0, 2, 1, 3) * torch.from_numpy(x["dO"])).sum().backward()
    assert np.max(np.abs(dq - oracle.rope(qh.grad.numpy(), inverse=True))) < 1e-11
    assert np.max(np.abs(dk - oracle.rope(kh.grad.numpy(), inverse=True))) < 1e-11
    assert np.max(np.abs(dv - v.grad.numpy())) < 1e-11


# ------------------------------------------------- the QKV front end ----


def test_qkv_front_end_brute_force_and_complex_rotation():
    """oracle.qkv_rope against explicit loops for the projection and complex
    multiplication z e^{i p w_m} (z = x_m + i x_{m+32}, w_m = 1e4^(-2m/64)) for
    the rotation, on a tiny case."""
    rng = np.random.default_rng(5)
    B, T, dm = 1, 3, 64
    x = rng.standard_normal((B, T, dm))
    w = rng.standard_normal((768, dm)) / 8.0
    q, k, v = oracle.qkv_rope(x, w, rope_theta=1e4)
    y = np.zeros((T, 768))
    for t in range(T):
        for r in range(768):
            acc = 0.0
            for c in range(dm):
                acc += x[0, t, c] * w[r, c]
            y[t, r] = acc
    freq = 10000.0 ** (-2.0 * np.arange(32) / 64)
    for t in range(T):
        rot = np.exp(1j * t * freq)
        for blk, got in ((range(8), q), (range(8, 10), k)):
            for n, h in enumerate(blk):
                z = (y[t, 64 * h:64 * h + 32] + 1j * y[t, 64 * h + 32:64 * h + 64]) * rot
                assert np.max(np.abs(got[0, t, n, :32] - z.real)) < 1e-12
                assert np.max(np.abs(got[0, t, n, 32:] - z.imag)) < 1e-12
        for g in range(2):
            assert np.max(np.abs(v[0, t, g] - y[t, 640 + 64 * g:704 + 64 * g])) < 1e-12
    q0, k0, v0 = oracle.qkv_rope(x, w, rope_theta=0.0)
    assert np.max(np.abs(q0[0, :, 3] - y[:, 192:256])) < 1e-12
    assert np.array_equal(v0, v)


def test_front_end_then_unrotated_attention_equals_attention_with_rope():
    """Rotating in the front end and attending with the rotation off gives the
    attention with RoPE inside (the rotation is applied once, before the
    gather, at true positions)."""
    x, w = inputs.hidden_and_weight(1, 40, 128, dtype=torch.float32, layer=3)
    q, k, v = oracle.qkv_rope(f64(x), f64(w), rope_theta=0.0)
    qh, kh, v2 = oracle.qkv_rope(f64(x), f64(w), rope_theta=1e4)
    o1, l1 = oracle.forward(q, k, v, W=4, rungs=oracle.FIBONACCI_BASE, alpha=0.83, rope_theta=1e4)
    o2, l2 = oracle.forward(qh, kh, v2, W=4, rungs=oracle.FIBONACCI_BASE, alpha=0.83, rope_theta=0.0)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12
