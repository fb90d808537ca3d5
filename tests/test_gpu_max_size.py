"""Parity at the largest sequence the library accepts: one sequence of 2^24
tokens (the longest T; positions are still exact in fp32 there).

The inputs are drawn on the GPU (``inputs.normal_on``) and the oracle runs on
three 4096-row slices of them, read back: the start, the middle and the end of
the sequence.  With RoPE every score depends on the positions only through
the distance i - j, so the oracle on a slice, at positions counted from the
slice's first row, gives the full sequence's result for every query whose
whole key list lies inside the slice (and that is past every rung's masking
threshold, or at the true start), and for every key row whose attending
queries are all such queries.  Those rows are compared element by element:
O and LSE of the forward, dQ, dK and dV of the backward, and the decode of
single queries over the whole 2^24-row cache."""
import gc

import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs
from oracle import oracle
from _helpers import TOL, max_abs, np64

pytestmark = pytest.mark.gpu

FIB = api.FIBONACCI_BASE
T_MAX = 1 << 24
SLICE = 4096
W = 12
ALPHA = 1.37
# the farthest key of a query is floor(fp32(alpha) * 987) + 1 = 1353 rows back
REACH = int(np.floor(np.float32(ALPHA) * np.float32(max(FIB)))) + 1
STARTS = (0, T_MAX // 2 - SLICE // 2, T_MAX - SLICE)


@pytest.fixture
def big_buffers():
    """Put the library's cached RoPE table and workspace back as they were,
    and free the device memory of the test, when the test ends."""
    rope, ws = dict(api._rope_cache), dict(api._ws_cache)
    yield
    api._rope_cache.clear()
    api._rope_cache.update(rope)
    api._ws_cache.clear()
    api._ws_cache.update(ws)
    gc.collect()
    torch.cuda.empty_cache()


def _draw(dtype, names):
    heads = {"q": 8, "k": 2, "v": 2, "dO": 8}
    return {n: inputs.normal_on("cuda", (1, T_MAX, heads[n], 64), dtype=dtype, layer=3, stream=n)
            for n in names}


def _host(t, s):
    return np64(t[:, s:s + SLICE])


def _query_rows(s):
    """Slice rows whose queries see their whole key list inside the slice."""
    return slice(0 if s == 0 else REACH, SLICE)


def _key_rows(s):
    """Slice rows whose attending queries (rows j .. j + REACH) are all exact."""
    return slice(0 if s == 0 else REACH, SLICE if s + SLICE == T_MAX else SLICE - REACH - 1)


def _close_grad(name, got, want, tol):
    err = max_abs(got, want)
    bound = tol * max(1.0, float(np.abs(want).max()))
    assert err <= bound, (name, err, bound)


def test_longest_sequence_bf16(big_buffers):
    x = _draw(torch.bfloat16, ("q", "k", "v", "dO"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = api.sfa_forward(x["q"], x["k"], x["v"], alpha=ALPHA, W=W, rungs=FIB, status=status)
    dq, dk, dv, da, dth = api.sfa_backward(x["q"], x["k"], x["v"], o, x["dO"], lse, alpha=ALPHA,
                                           W=W, rungs=FIB, status=status)
    # one new query at the start, the middle and the last position, over the
    # whole cache (B = 1 per call)
    positions = (5, T_MAX // 2, T_MAX - 1)
    dec = []
    for p in positions:
        od, ld = api.sfa_decode(x["q"][:, p].contiguous(), x["k"], x["v"],
                                torch.tensor([p], dtype=torch.int32, device="cuda"),
                                alpha=ALPHA, W=W, rungs=FIB, status=status)
        dec.append((p, od, ld))
    torch.cuda.synchronize()
    assert api.sfa_read_status(status) == 0
    tol = TOL["bf16"]
    for s in STARTS:
        h = {n: _host(t, s) for n, t in x.items()}
        o_ref, lse_ref = oracle.forward(h["q"], h["k"], h["v"], W=W, rungs=FIB, alpha=ALPHA)
        qr, kr = _query_rows(s), _key_rows(s)
        assert max_abs(_host(o, s)[:, qr], o_ref[:, qr]) <= tol["o"], s
        assert max_abs(_host(lse, s)[:, qr], lse_ref[:, qr]) <= tol["lse"], s
        for p, od, ld in dec:
            if s <= p < s + SLICE:
                assert qr.start <= p - s < qr.stop
                assert max_abs(np64(od)[0], o_ref[0, p - s]) <= tol["o"], p
                assert max_abs(np64(ld)[0], lse_ref[0, p - s]) <= tol["lse"], p
        ref = oracle.backward(h["q"], h["k"], h["v"], h["dO"], W=W, rungs=FIB, alpha=ALPHA)
        _close_grad("dq", _host(dq, s)[:, qr], ref[0][:, qr], tol["grad"])
        _close_grad("dk", _host(dk, s)[:, kr], ref[1][:, kr], tol["grad"])
        _close_grad("dv", _host(dv, s)[:, kr], ref[2][:, kr], tol["grad"])
    # over the whole sequence: finite everywhere, rows are convex combinations
    vmax = float(x["v"].abs().max())
    assert float(o.abs().max()) <= vmax * (1 + 1e-2)
    for t in (lse, dq, dk, dv, da, dth):
        assert bool(torch.isfinite(t).all())


def test_longest_sequence_fp32(big_buffers):
    x = _draw(torch.float32, ("q", "k", "v"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = api.sfa_forward(x["q"], x["k"], x["v"], alpha=ALPHA, W=W, rungs=FIB, status=status)
    torch.cuda.synchronize()
    assert api.sfa_read_status(status) == 0
    tol = TOL["f32"]
    for s in STARTS:
        h = {n: _host(t, s) for n, t in x.items()}
        o_ref, lse_ref = oracle.forward(h["q"], h["k"], h["v"], W=W, rungs=FIB, alpha=ALPHA)
        qr = _query_rows(s)
        assert max_abs(_host(o, s)[:, qr], o_ref[:, qr]) <= tol["o"], s
        assert max_abs(_host(lse, s)[:, qr], lse_ref[:, qr]) <= tol["lse"], s
    assert bool(torch.isfinite(o).all())
