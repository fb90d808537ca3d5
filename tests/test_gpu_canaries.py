"""Guard canaries: every output of the library (and the caller's workspace)
lives inside a larger buffer filled with a marker -- NaN for outputs, 0xA5
bytes for the workspace -- on ragged shapes.  After the call the guard bytes
before and after each output must be untouched (no write outside it), and
every element inside must have been written (a NaN left there fails the
comparison with the oracle)."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs
from oracle import oracle
from _helpers import DT, TOL, draw, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE
PAD = 4096  # elements of guard on each side (a multiple of 16 bytes for every dtype)


class Guarded:
    """A tensor of ``shape`` in the middle of a NaN-filled buffer."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.buf = torch.full((PAD + n + PAD,), float("nan"), dtype=dtype, device="cuda")
        self.t = self.buf[PAD:PAD + n].view(*shape)
        self.n = n

    def guards_intact(self):
        return bool(torch.isnan(self.buf[:PAD]).all()) and bool(torch.isnan(self.buf[PAD + self.n:]).all())


class GuardedBytes:
    """A byte workspace of ``nbytes`` in the middle of a 0xA5-filled buffer."""

    def __init__(self, nbytes):
        self.buf = torch.full((PAD + max(nbytes, 1) + PAD,), 0xA5, dtype=torch.uint8, device="cuda")
        self.t = self.buf[PAD:PAD + max(nbytes, 1)]
        self.n = max(nbytes, 1)

    def guards_intact(self):
        return bool((self.buf[:PAD] == 0xA5).all()) and bool((self.buf[PAD + self.n:] == 0xA5).all())


def _forward_ws_bytes(B, T, dtype, alpha, W):
    p = api.Params(B, T, W=W, alpha=alpha, rungs=FIB, dtype=DT[dtype])
    from fibonacci_spaced_sparse_gb300 import _lib
    return int(_lib.load().sfa_forward_workspace_size(p.ref()))


@pytest.mark.parametrize("dtype,B,T,W", [("bf16", 3, 97, 12), ("bf16", 2, 300, 30), ("f32", 2, 61, 8),
                                         ("bf16", 1, 1, 12)])
def test_forward_writes_exactly_its_outputs(dtype, B, T, W):
    x, f = draw(B, T, dtype, layer=41)
    xd = to_dev(x)
    o = Guarded((B, T, 8, 64), DT[dtype])
    lse = Guarded((B, T, 8), torch.float32)
    ws = GuardedBytes(_forward_ws_bytes(B, T, dtype, 1.23, W))
    api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=1.23, W=W, rungs=FIB, out=o.t, lse=lse.t,
                    workspace=ws.t)
    torch.cuda.synchronize()
    assert o.guards_intact() and lse.guards_intact() and ws.guards_intact()
    o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], W=W, rungs=FIB, alpha=1.23)
    assert max_abs(np64(o.t), o_ref) <= TOL[dtype]["o"]
    assert max_abs(np64(lse.t), lse_ref) <= TOL[dtype]["lse"]


def test_multi_layer_forward_writes_exactly_its_outputs():
    B, T, L = 2, 157, 3
    xs = [draw(B, T, "bf16", layer=50 + l) for l in range(L)]
    xd = [to_dev(x) for x, _ in xs]
    alphas = [0.7, 1.0, 1.41]
    outs = [Guarded((B, T, 8, 64), torch.bfloat16) for _ in range(L)]
    lses = [Guarded((B, T, 8), torch.float32) for _ in range(L)]
    api.sfa_forward_layers([x["q"] for x in xd], [x["k"] for x in xd], [x["v"] for x in xd],
                           alphas=alphas, W=12, outs=[g.t for g in outs], lses=[g.t for g in lses])
    torch.cuda.synchronize()
    for l in range(L):
        assert outs[l].guards_intact() and lses[l].guards_intact(), l
        f = xs[l][1]
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], W=12, rungs=FIB, alpha=alphas[l])
        assert max_abs(np64(outs[l].t), o_ref) <= TOL["bf16"]["o"], l
        assert max_abs(np64(lses[l].t), lse_ref) <= TOL["bf16"]["lse"], l


@pytest.mark.parametrize("dtype,B,T,W", [("bf16", 3, 97, 12), ("bf16", 1, 29, 17), ("f32", 2, 45, 6)])
def test_backward_writes_exactly_its_outputs(dtype, B, T, W):
    x, f = draw(B, T, dtype, layer=43, with_dO=True)
    xd = to_dev(x)
    o, lse = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=0.91, W=W, rungs=FIB)
    dq = Guarded((B, T, 8, 64), DT[dtype])
    dk = Guarded((B, T, 2, 64), DT[dtype])
    dv = Guarded((B, T, 2, 64), DT[dtype])
    da = Guarded((1,), torch.float32)
    dth = Guarded((1,), torch.float32)
    need = api.sfa_backward_workspace_size(B, T, alpha=0.91, W=W, dtype=DT[dtype])
    ws = GuardedBytes(need)
    api.sfa_backward(xd["q"], xd["k"], xd["v"], o, xd["dO"], lse, alpha=0.91, W=W, rungs=FIB,
                     workspace=ws.t, out=(dq.t, dk.t, dv.t, da.t, dth.t))
    torch.cuda.synchronize()
    for g in (dq, dk, dv, da, dth, ws):
        assert g.guards_intact()
    ref = oracle.backward(f["q"], f["k"], f["v"], f["dO"], W=W, rungs=FIB, alpha=0.91)
    for name, got, want in (("dq", dq.t, ref[0]), ("dk", dk.t, ref[1]), ("dv", dv.t, ref[2])):
        bound = TOL[dtype]["grad"] * max(1.0, float(np.abs(want).max()))
        assert max_abs(np64(got), want) <= bound, name
    assert np.isfinite(float(da.t.item())) and np.isfinite(float(dth.t.item()))


def test_decode_writes_exactly_its_outputs():
    B, Tc = 5, 300
    x, f = draw(B, Tc, "bf16", layer=44)
    pos = np.array([0, 13, 150, 298, 299], dtype=np.int32)
    qd = torch.stack([x["q"][b, p] for b, p in enumerate(pos)]).cuda()
    o = Guarded((B, 8, 64), torch.bfloat16)
    lse = Guarded((B, 8), torch.float32)
    api.sfa_decode(qd, x["k"].cuda(), x["v"].cuda(), torch.from_numpy(pos).cuda(), alpha=1.1, W=12,
                   rungs=FIB, out=o.t, lse=lse.t)
    torch.cuda.synchronize()
    assert o.guards_intact() and lse.guards_intact()
    rows = np.stack([np.arange(B, dtype=np.int32), pos], axis=1)
    o_ref, lse_ref = oracle.forward_rows(f["q"], f["k"], f["v"], rows, W=12, rungs=FIB, alpha=1.1)
    assert max_abs(np64(o.t), o_ref) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse.t), lse_ref) <= TOL["bf16"]["lse"]


def test_front_end_writes_exactly_its_outputs():
    B, T, dm = 2, 157, 192                      # 314 tokens: a ragged last 128-token tile
    x, w = inputs.hidden_and_weight(B, T, dm, layer=45)
    q = Guarded((B, T, 8, 64), torch.bfloat16)
    k = Guarded((B, T, 2, 64), torch.bfloat16)
    v = Guarded((B, T, 2, 64), torch.bfloat16)
    api.sfa_qkv_rope(x.cuda(), w.cuda(), out=(q.t, k.t, v.t))
    torch.cuda.synchronize()
    assert q.guards_intact() and k.guards_intact() and v.guards_intact()
    rq, rk, rv = oracle.qkv_rope(x.to(torch.float64).numpy(), w.to(torch.float64).numpy())
    for got, want in ((q.t, rq), (k.t, rk), (v.t, rv)):
        g = np64(got)
        assert np.isfinite(g).all()
        assert float(np.max(np.abs(g - want) - (2.0 ** -8 * np.abs(want) + 1e-3))) <= 0
