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


def test_front_end_and_attention_graph_replay_matches_eager():
    """sfa_qkv_rope then sfa_forward(rope_theta = 0) for two layers, captured
    in one graph: the replay reproduces the eager outputs bit for bit."""
    from fibonacci_spaced_sparse_gb300 import inputs
    B, T, dm, L = 2, 384, 512, 2
    xw = [inputs.hidden_and_weight(B, T, dm, layer=30 + l) for l in range(L)]
    xs = [x.cuda() for x, _ in xw]
    ws = [w.cuda() for _, w in xw]
    bf = torch.bfloat16
    mids = [(torch.empty((B, T, 8, 64), dtype=bf, device="cuda"),
             torch.empty((B, T, 2, 64), dtype=bf, device="cuda"),
             torch.empty((B, T, 2, 64), dtype=bf, device="cuda")) for _ in range(L)]
    outs = [torch.empty((B, T, 8, 64), dtype=bf, device="cuda") for _ in range(L)]
    lses = [torch.empty((B, T, 8), dtype=torch.float32, device="cuda") for _ in range(L)]

    def step(stream):
        for l in range(L):
            qh, kh, v = api.sfa_qkv_rope(xs[l], ws[l], out=mids[l], stream=stream)
            api.sfa_forward(qh, kh, v, alpha=0.7 + 0.4 * l, W=12, rope_theta=0.0, out=outs[l],
                            lse=lses[l], stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [(o.clone(), s.clone(), m[0].clone()) for o, s, m in zip(outs, lses, mids)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(side)
    for o, m in zip(outs, mids):
        o.zero_()
        m[0].zero_()
    graph.replay()
    torch.cuda.synchronize()
    for l in range(L):
        assert torch.equal(outs[l], eager[l][0]) and torch.equal(lses[l], eager[l][1])
        assert torch.equal(mids[l][0], eager[l][2])
