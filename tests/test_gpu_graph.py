"""The training step of several layers (multi-layer forward, then each
layer's backward) captured in one CUDA graph and replayed: the library calls
allocate nothing and synchronise nothing, so they capture, and the replay
must reproduce the eager results -- exactly for O, LSE, dQ, dalpha and dtheta
(fixed summation orders), and up to the last bf16 bit for dK and dV (summed
by fp32 atomic reductions, whose order varies from run to run)."""
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, workloads
from _helpers import draw, to_dev

pytestmark = pytest.mark.gpu


def test_train_step_graph_replay_matches_eager():
    wl = workloads.TRAIN_STEP
    L, B, T = 3, 4, 512
    alphas = wl.alphas()[0][:L]
    xd = [to_dev(draw(B, T, "bf16", layer=l, with_dO=True)[0]) for l in range(L)]
    qs, ks, vs = [x["q"] for x in xd], [x["k"] for x in xd], [x["v"] for x in xd]
    outs = [torch.empty_like(q) for q in qs]
    lses = [torch.empty((B, T, 8), dtype=torch.float32, device="cuda") for _ in range(L)]
    grads = [[torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]),
              torch.empty(1, device="cuda"), torch.empty(1, device="cuda")] for x in xd]
    fwd_ws = torch.empty(api_ws_fwd(B, T, L), dtype=torch.uint8, device="cuda")
    bwd_ws = torch.empty(max(api.sfa_backward_workspace_size(B, T, alpha=a, W=12) for a in alphas),
                         dtype=torch.uint8, device="cuda")

    def step(stream):
        api.sfa_forward_layers(qs, ks, vs, alphas=alphas, W=12, outs=outs, lses=lses,
                               workspace=fwd_ws, stream=stream)
        for l in range(L):
            g = grads[l]
            api.sfa_backward(qs[l], ks[l], vs[l], outs[l], xd[l]["dO"], lses[l], alpha=alphas[l],
                             W=12, workspace=bwd_ws, out=g, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)                      # eager, also builds the RoPE table and kernel attributes
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [[t.clone() for t in [o, s] + g] for o, s, g in zip(outs, lses, grads)]
    for o in outs:
        o.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(side)
    for _ in range(2):
        for o, g in zip(outs, grads):
            o.zero_()
            for t in g:
                t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for l in range(L):
            got = [outs[l], lses[l]] + grads[l]
            names = ["o", "lse", "dq", "dk", "dv", "dalpha", "dtheta"]
            for name, a, b in zip(names, got, eager[l]):
                if name in ("dk", "dv"):
                    scale = float(b.float().abs().max())
                    err = float((a.float() - b.float()).abs().max())
                    assert err <= 1e-2 * max(scale, 1.0), (l, name, err, scale)
                else:
                    assert torch.equal(a, b), (l, name)


def api_ws_fwd(B, T, L):
    from fibonacci_spaced_sparse_gb300 import _lib
    import ctypes
    p = api.Params(B, T, W=12, alpha=1.0)
    win = (ctypes.c_int * L)(*([12] * L))
    return max(1, int(_lib.load().sfa_forward_layers_workspace_size(p.ref(), L, win)))
