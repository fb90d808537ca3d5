"""The multi-layer forward (sfa_forward_layers): each layer must give exactly
what sfa_forward gives for that layer -- the attention launches are the same
kernels, and the next layer's keys are rotated (inside the previous layer's
launch) with the same roundings as the RoPE pass -- and must match the oracle
on sampled rows at the model shape."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, workloads
from oracle import oracle
from _helpers import TOL, draw, max_abs, np64, sample_rows, to_dev

pytestmark = pytest.mark.gpu


def _layers(B, T, L, dtype="bf16", first_layer=0):
    xs = [draw(B, T, dtype, layer=first_layer + l) for l in range(L)]
    return [to_dev(x) for x, _ in xs], [f for _, f in xs]


@pytest.mark.parametrize("B,T", [(2, 300), (4, 1024)])
def test_layers_equal_single_layer_calls(B, T):
    L = 5
    alphas = api.alpha_schedule("linear", 16)[:L]
    xd, _ = _layers(B, T, L)
    outs, lses = api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd],
                                        [x["v"] for x in xd], alphas=alphas, W=12)
    for l in range(L):
        o, lse = api.sfa_forward(xd[l]["q"], xd[l]["k"], xd[l]["v"], alpha=alphas[l], W=12)
        torch.cuda.synchronize()
        assert torch.equal(outs[l], o), l
        assert torch.equal(lses[l], lse), l


def test_layers_with_per_layer_windows_and_pow2_base():
    wl = workloads.POW2
    L = 4
    alphas, _ = wl.alphas()
    rungs = wl.rungs()
    B, T = 3, 600
    xd, _ = _layers(B, T, L)
    windows = [wl.window(l) for l in range(L)]
    outs, lses = api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd],
                                        [x["v"] for x in xd], alphas=alphas[:L], W=windows,
                                        rungs=rungs)
    for l in range(L):
        o, lse = api.sfa_forward(xd[l]["q"], xd[l]["k"], xd[l]["v"], alpha=alphas[l],
                                 W=windows[l], rungs=rungs)
        torch.cuda.synchronize()
        assert torch.equal(outs[l], o), l
        assert torch.equal(lses[l], lse), l


def test_layers_fp32_fall_back_to_single_calls():
    L = 3
    alphas = [1.0, 0.77, 1.31]
    xd, f = _layers(1, 200, L, dtype="f32")
    outs, lses = api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd],
                                        [x["v"] for x in xd], alphas=alphas, W=8)
    torch.cuda.synchronize()
    for l in range(L):
        o_ref, lse_ref = oracle.forward(f[l]["q"], f[l]["k"], f[l]["v"], W=8,
                                        rungs=api.FIBONACCI_BASE, alpha=alphas[l])
        assert max_abs(np64(outs[l]), o_ref) <= TOL["f32"]["o"]
        assert max_abs(np64(lses[l]), lse_ref) <= TOL["f32"]["lse"]


def test_model_shape_layers_sampled_against_oracle():
    """Two consecutive layers of the model-shape workload (B=32, T=1024,
    W=12, linear stagger) on sampled rows."""
    wl = workloads.MODEL_SHAPE
    alphas, _ = wl.alphas()
    first = 6
    L = 2
    xd, f = _layers(wl.B, wl.T, L, first_layer=first)
    outs, lses = api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd],
                                        [x["v"] for x in xd], alphas=alphas[first:first + L],
                                        W=12)
    torch.cuda.synchronize()
    for l in range(L):
        rows = sample_rows(wl.B, wl.T, 256, seed=first + l)
        o_ref, lse_ref = oracle.forward_rows(f[l]["q"], f[l]["k"], f[l]["v"], rows, W=12,
                                             rungs=wl.rungs(), alpha=alphas[first + l])
        og = np64(outs[l])[rows[:, 0], rows[:, 1]]
        lg = np64(lses[l])[rows[:, 0], rows[:, 1]]
        assert max_abs(og, o_ref) <= TOL["bf16"]["o"]
        assert max_abs(lg, lse_ref) <= TOL["bf16"]["lse"]
