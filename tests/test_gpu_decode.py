"""Single-token decode over a key/value cache (sfa_decode): each sequence's
new query at position i = positions[b] against the fp64 oracle's row (b, i),
with every cache row after i poisoned with NaN (the decode must not read
it); a position outside the cache reports SFA_DEVSTAT_BAD_INDEX."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api
from oracle import oracle
from _helpers import DT, TOL, draw, max_abs, np64

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE


def _positions(B, Tc, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 12, 13, 14, 21, 22, 89, 90, Tc - 1]
    pos = [p for p in fixed if p < Tc][:B]
    while len(pos) < B:
        pos.append(int(rng.integers(0, Tc)))
    return np.array(pos, dtype=np.int32)


def _case(B, Tc, dtype, alpha, W, rungs=FIB, seed=0):
    x, _ = draw(B, Tc, dtype, layer=11 + seed)
    pos = _positions(B, Tc, seed)
    k = x["k"].clone()
    v = x["v"].clone()
    for b, p in enumerate(pos):          # rows after the new token are never read
        k[b, p + 1:] = float("nan")
        v[b, p + 1:] = float("nan")
    qd = torch.stack([x["q"][b, p] for b, p in enumerate(pos)])
    o, lse = api.sfa_decode(qd.cuda(), k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(),
                            alpha=alpha, W=W, rungs=rungs)
    torch.cuda.synchronize()
    rows = np.stack([np.arange(B, dtype=np.int32), pos], axis=1)
    f = {n: x[n].to(torch.float64).numpy() for n in ("q", "k", "v")}
    o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=W, rungs=rungs,
                                         alpha=alpha)
    assert max_abs(np64(o), o_ref) <= TOL[dtype]["o"], (alpha, W)
    assert max_abs(np64(lse), lse_ref) <= TOL[dtype]["lse"], (alpha, W)


@pytest.mark.parametrize("alpha", [0.61, 1.0, 1.37])
def test_decode_bf16_against_oracle(alpha):
    _case(24, 700, "bf16", alpha, 12)


@pytest.mark.parametrize("alpha,W", [(1.0, 8), (0.83, 6)])
def test_decode_fp32_against_oracle(alpha, W):
    _case(12, 300, "f32", alpha, W)


def test_decode_pow2_base_long_cache():
    _case(8, 4096, "bf16", api.alpha_from_theta(-0.2), 10, rungs=api.pow2_base(4096), seed=3)


def test_decode_matches_forward_last_row():
    """The decode of the last position equals the forward's last row."""
    B, T = 6, 512
    x, _ = draw(B, T, "bf16", layer=5)
    xd = {n: t.cuda() for n, t in x.items()}
    alpha = 1.13
    o_full, lse_full = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=12)
    pos = torch.full((B,), T - 1, dtype=torch.int32, device="cuda")
    o, lse = api.sfa_decode(xd["q"][:, T - 1].contiguous(), xd["k"], xd["v"], pos, alpha=alpha,
                            W=12)
    torch.cuda.synchronize()
    assert max_abs(np64(o), np64(o_full[:, T - 1])) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse), np64(lse_full[:, T - 1])) <= TOL["bf16"]["lse"]


def test_decode_bad_position_reports_and_zeroes():
    B, Tc = 4, 64
    x, _ = draw(B, Tc, "bf16", layer=2)
    qd = x["q"][:, 5].contiguous().cuda()
    pos = torch.tensor([5, Tc, -1, 7], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = api.sfa_decode(qd, x["k"].cuda(), x["v"].cuda(), pos, alpha=1.0, W=8,
                            status=status)
    word = api.sfa_read_status(status)
    assert word & 0x2
    on = np64(o)
    assert np.all(on[1] == 0) and np.all(on[2] == 0)
    assert np.isfinite(on).all() and np.abs(on[0]).max() > 0


@pytest.mark.parametrize("alpha,W", [(1.0, 30), (0.7, 24), (1.0, 20), (1.3, 16)])
def test_decode_long_key_lists(alpha, W):
    """Key lists longer than 32 entries (W = 24, 30) take the general kernel,
    shorter ones the one-pass kernel; both against the oracle."""
    _case(16, 1200, "bf16", alpha, W, seed=7)


def test_decode_explicit_softmax_scale():
    B, Tc = 6, 400
    x, _ = draw(B, Tc, "bf16", layer=63)
    pos = np.array([0, 7, 13, 150, 398, 399], dtype=np.int32)
    qd = torch.stack([x["q"][b, p] for b, p in enumerate(pos)])
    o, lse = api.sfa_decode(qd.cuda(), x["k"].cuda(), x["v"].cuda(), torch.from_numpy(pos).cuda(),
                            alpha=1.2, W=12, rungs=FIB, scale=0.3)
    torch.cuda.synchronize()
    rows = np.stack([np.arange(B, dtype=np.int32), pos], axis=1)
    f = {n: x[n].to(torch.float64).numpy() for n in ("q", "k", "v")}
    o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=12, rungs=FIB, alpha=1.2,
                                         scale=0.3)
    assert max_abs(np64(o), o_ref) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse), lse_ref) <= TOL["bf16"]["lse"]


def test_decode_bench_shape_from_graph_replay():
    """The benchmark's launch configuration: 256 sequences over 4096-row
    caches, the per-layer calls captured once in a CUDA graph on a side stream
    and replayed; sampled sequences of every layer against the oracle."""
    from fibonacci_spaced_sparse_gb300 import inputs
    B, Tc, W, L = 256, 4096, 12, 2
    alphas = [api.alpha_schedule("linear", 16)[l] for l in (3, 12)]
    kc = [inputs.normal_on("cuda", (B, Tc, 2, 64), layer=70 + l, stream="k") for l in range(L)]
    vc = [inputs.normal_on("cuda", (B, Tc, 2, 64), layer=70 + l, stream="v") for l in range(L)]
    qs = [inputs.normal_on("cuda", (B, 8, 64), layer=70 + l, stream="q") for l in range(L)]
    rng = np.random.default_rng(70)
    pos_np = rng.integers(Tc // 2, Tc, B).astype(np.int32)
    pos_np[:3] = [Tc // 2, Tc - 2, Tc - 1]
    pos = torch.from_numpy(pos_np).cuda()
    outs = [torch.empty_like(q) for q in qs]
    lses = [torch.empty((B, 8), dtype=torch.float32, device="cuda") for _ in range(L)]
    api.rope_table(Tc, "cuda")
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()

    def layers(s):
        for l in range(L):
            api.sfa_decode(qs[l], kc[l], vc[l], pos, alpha=alphas[l], W=W, out=outs[l], lse=lses[l], stream=s)

    side.wait_stream(main)
    with torch.cuda.stream(side):
        layers(side)
    main.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        layers(side)
    for o in outs:
        o.fill_(float("nan"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for l in range(L):
        for b in (0, 1, 2, 77, 128, 255):
            i = int(pos_np[b])
            q = np.zeros((1, Tc, 8, 64))
            q[0, i] = qs[l][b].double().cpu().numpy()
            k = kc[l][b:b + 1].double().cpu().numpy()
            v = vc[l][b:b + 1].double().cpu().numpy()
            o_ref, lse_ref = oracle.forward_rows(q, k, v, np.array([[0, i]], dtype=np.int32), W=W,
                                                 rungs=FIB, alpha=alphas[l])
            assert max_abs(np64(outs[l][b]), o_ref[0]) <= TOL["bf16"]["o"], (l, b)
            assert max_abs(np64(lses[l][b]), lse_ref[0]) <= TOL["bf16"]["lse"], (l, b)
