"""The C ABI without a GPU: the library loads, exports every symbol that
include/sfa.h declares, and its host-side logic (schedules, rung preparation,
argument validation) behaves as documented.  No call here launches a kernel."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from fibonacci_spaced_sparse_gb300 import _lib, api
from oracle import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sfa.h")


@pytest.fixture(scope="module")
def lib():
    from fibonacci_spaced_sparse_gb300 import build
    build.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SFA_API\s+[^;{]*?\b(sfa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("sfa_forward", "sfa_backward", "sfa_backward_workspace_size", "sfa_strerror",
              "sfa_rope_table", "sfa_rung_plan", "sfa_alpha_schedule"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_no_stray_exports(lib):
    """Only the declared entry points are visible (hidden visibility)."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    ours = sorted({ln.split()[-1] for ln in out.splitlines() if " T sfa_" in ln})
    assert ours == declared_symbols()


def test_version_and_strerror(lib):
    assert lib.sfa_version() >> 16 == 1
    for code in range(5):
        assert lib.sfa_strerror(code)
    assert b"unknown" in lib.sfa_strerror(99)


def test_alpha_from_theta_matches_oracle(lib):
    for th in (-20.0, -3.5, -0.437, 0.0, 0.3, 1.0, 7.25):
        assert api.alpha_from_theta(th) == np.float32(oracle.alpha_from_theta(float(np.float32(th))))
    assert api.alpha_from_theta(0.0) == 1.0


@pytest.mark.parametrize("kind", ["fixed", "linear", "coprime", "learned"])
def test_schedules_match_oracle(lib, kind):
    thetas = [0.1 * l - 0.7 for l in range(16)]
    got = api.alpha_schedule(kind, 16, 7, thetas if kind == "learned" else None)
    ref = {"fixed": oracle.schedule_fixed(16), "linear": oracle.schedule_linear(16),
           "coprime": oracle.schedule_coprime(16, 7),
           "learned": oracle.schedule_learned([float(np.float32(t)) for t in thetas])}[kind]
    assert got == [float(np.float32(a)) for a in ref]


def test_schedule_rejects_bad_arguments(lib):
    out = (ctypes.c_float * 16)()
    fp = ctypes.cast(out, ctypes.POINTER(ctypes.c_float))
    assert lib.sfa_alpha_schedule(3, 16, 8, None, fp) == _lib.SFA_ERR_INVALID_ARG  # gcd(8,16) != 1
    assert lib.sfa_alpha_schedule(1, 16, 7, None, fp) == _lib.SFA_ERR_INVALID_ARG  # no thetas
    assert lib.sfa_alpha_schedule(2, 1, 7, None, fp) == _lib.SFA_ERR_INVALID_ARG  # L < 2
    assert lib.sfa_alpha_schedule(9, 16, 7, None, fp) == _lib.SFA_ERR_INVALID_ARG


def _plan_rule(alpha, W, T, base):
    """The documented rung rule: fp32 product, drop d <= W, leave out rungs
    with ceil(d) > T - 1 (masked for every query)."""
    out = []
    for k, f in enumerate(base):
        d = np.float32(np.float32(alpha) * np.float32(f))
        if not d > W:
            continue
        if math.ceil(d) > T - 1:
            continue
        n = math.floor(d)
        out.append((k, n, float(d - np.float32(n)), math.ceil(d)))
    return out


@pytest.mark.parametrize("alpha,W,T", [(1.0, 8, 256), (1.5, 12, 1024), (0.5, 12, 1024),
                                       (0.733333, 12, 4096), (1.2345, 6, 1024),
                                       (0.1000000005 * 10, 13, 1024), (1.0, 0, 10)])
def test_rung_plan_rule(lib, alpha, W, T):
    assert api.rung_plan(T=T, W=W, alpha=alpha) == _plan_rule(alpha, W, T, api.FIBONACCI_BASE)


def test_rung_plan_boundaries(lib):
    # alpha = 1.5, f = 8 gives d = 12 = W exactly: dropped
    assert all(r[0] != 4 for r in api.rung_plan(T=1024, W=12, alpha=1.5))
    # d just above W is kept even though floor(d) = W
    plan = api.rung_plan(T=64, W=8, alpha=1.0 + 2 ** -20, rungs=[8])
    assert len(plan) == 1 and plan[0][1] == 8 and 0 < plan[0][2] < 1e-4 and plan[0][3] == 9
    # integer distance: t = 0, ceil = floor
    assert api.rung_plan(T=64, W=8, alpha=1.0, rungs=[13]) == [(0, 13, 0.0, 13)]
    # pow2 base at T = 1024 with K = 10 rungs
    assert api.pow2_base(1024) == tuple(2 ** k for k in range(10))
    assert set(api.pow2_base(4096)) >= {1024, 2048}


def test_rung_plan_rounded(lib):
    """round_offsets: integer distances (t = 0), halves up, computed on the fp32
    product alpha * f_k; rounded distances inside the window are dropped."""
    plan = api.rung_plan(T=1024, W=3, alpha=0.5, round_offsets=True)
    # d = 1.5, 2.5, 4, 6.5, 10.5, ... -> 2, 3 (inside W = 3), 4, 7, 11, ...
    assert [(r[1], r[2], r[3]) for r in plan[:3]] == [(4, 0.0, 4), (7, 0.0, 7), (11, 0.0, 11)]
    assert all(r[2] == 0.0 and r[1] == r[3] for r in plan)
    # fp32(2.1) * 55 is just below 115.5: rounds down to 115, not up to 116
    assert np.float32(2.1) * np.float32(55) < np.float32(115.5)
    assert api.rung_plan(T=256, W=0, alpha=2.1, rungs=[55], round_offsets=True) == \
        [(0, 115, 0.0, 115)]
    # 10.96 rounds to 11 = W: dropped, though the interpolated rung is kept at W = 10
    assert api.rung_plan(T=64, W=11, alpha=1.37, rungs=[8], round_offsets=True) == []
    assert len(api.rung_plan(T=64, W=10, alpha=1.37, rungs=[8])) == 1
    p = api.Params(1, 16, W=2, alpha=1.0)
    p.struct.round_offsets = 2
    n = ctypes.c_int(0)
    assert lib.sfa_rung_plan(p.ref(), ctypes.byref(n), None, None, None, None) == \
        _lib.SFA_ERR_INVALID_ARG


def _params(**kw):
    d = dict(W=12, alpha=1.0)
    d.update(kw)
    B = d.pop("B", 2)
    T = d.pop("T", 64)
    return api.Params(B, T, **d)


def test_validation_codes(lib):
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails validation
    null = ctypes.c_void_p(0)
    fwd = lambda p, q=fake, o=fake, tab=fake: lib.sfa_forward(p.ref(), q, fake, fake, tab, o, null,
                                                              fake, 1 << 40, null, null)
    assert fwd(_params(Hq=4)) == _lib.SFA_ERR_UNSUPPORTED
    assert fwd(_params(D=128)) == _lib.SFA_ERR_UNSUPPORTED
    assert fwd(_params(W=-1)) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(alpha=float("nan"))) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(alpha=0.0)) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(rungs=[1.0, -2.0])) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(rungs=[1.0] * 33)) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(scale=-1.0)) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(), q=null) == _lib.SFA_ERR_INVALID_ARG
    assert fwd(_params(), q=ctypes.c_void_p(0x10008)) == _lib.SFA_ERR_INVALID_ARG  # misaligned
    assert fwd(_params(), tab=null) == _lib.SFA_ERR_INVALID_ARG    # rope on, no table
    p = _params(T=1 << 25)
    assert fwd(p) == _lib.SFA_ERR_UNSUPPORTED
    # B * T is capped at 2^28 tokens (the longest sequence, 2^24, times 16)
    assert fwd(_params(B=17, T=1 << 24)) == _lib.SFA_ERR_UNSUPPORTED
    assert fwd(_params(B=(1 << 28) + 1, T=1)) == _lib.SFA_ERR_UNSUPPORTED
    assert lib.sfa_forward_workspace_size(_params(B=17, T=1 << 24).ref()) == 0
    assert lib.sfa_forward_workspace_size(_params(B=16, T=1 << 24).ref()) == (1 << 28) * 2 * 64 * 2
    assert lib.sfa_forward(None, fake, fake, fake, fake, fake, null, fake, 0, null,
                           null) == _lib.SFA_ERR_INVALID_ARG
    # bf16 needs the rotated-key workspace: too small or misaligned is rejected
    p = _params()
    need = lib.sfa_forward_workspace_size(p.ref())
    assert need == 2 * 64 * 2 * 64 * 2
    ws_call = lambda ws, n: lib.sfa_forward(p.ref(), fake, fake, fake, fake, fake, null, ws, n,
                                            null, null)
    assert ws_call(fake, need - 1) == _lib.SFA_ERR_INVALID_ARG
    assert ws_call(ctypes.c_void_p(0x10010), need) == _lib.SFA_ERR_INVALID_ARG
    assert ws_call(null, need) == _lib.SFA_ERR_INVALID_ARG
    assert lib.sfa_forward_workspace_size(_params(dtype=__import__("torch").float32).ref()) == 0
    assert lib.sfa_forward_workspace_size(_params(rope_theta=0.0).ref()) == 0
    # nothing to do: B = 0 returns before looking at the pointers
    assert fwd(_params(B=0), q=null, o=null, tab=null) == _lib.SFA_OK
    # backward: workspace too small, missing lse
    p = _params()
    need = lib.sfa_backward_workspace_size(p.ref())
    assert need > 0
    bwd = lambda ws, nbytes, lse=fake: lib.sfa_backward(
        p.ref(), fake, fake, fake, fake, fake, lse, fake, fake, fake, fake, fake, fake, ws, nbytes,
        null, null)
    assert bwd(fake, need - 1) == _lib.SFA_ERR_INVALID_ARG
    assert bwd(ctypes.c_void_p(0x10010), need) == _lib.SFA_ERR_INVALID_ARG  # not 256-aligned
    assert bwd(fake, need, lse=null) == _lib.SFA_ERR_INVALID_ARG
    # rope table: bad sizes
    assert lib.sfa_rope_table(fake, 16, 63, 1e4, null) == _lib.SFA_ERR_INVALID_ARG
    assert lib.sfa_rope_table(fake, 16, 64, 0.0, null) == _lib.SFA_ERR_INVALID_ARG
    assert lib.sfa_rope_table_floats(1024, 64) == 1024 * 64
    assert lib.sfa_read_status(null, None, null) == _lib.SFA_ERR_INVALID_ARG


def test_workspace_size_formula(lib):
    p = _params(B=3, T=100)
    nkv = 3 * 100 * 2 * 64 * 4
    blocks = (3 * 100 * 2 + 7) // 8
    a256 = lambda x: (x + 255) // 256 * 256
    assert lib.sfa_backward_workspace_size(p.ref()) >= 2 * a256(nkv) + a256(blocks * 32 * 4)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def test_forward_layers_host_checks(lib):
    """Argument checks of the multi-layer forward (nothing is launched)."""
    p = api.Params(2, 64, W=12, alpha=1.0)
    one = api.Params(2, 64, W=12, alpha=1.0)
    L = 3
    win = (ctypes.c_int * L)(12, 12, 12)
    single = lib.sfa_forward_workspace_size(one.ref())
    assert lib.sfa_forward_layers_workspace_size(p.ref(), L, win) >= 2 * single
    assert lib.sfa_forward_layers_workspace_size(p.ref(), 0, win) == 0
    f32 = api.Params(2, 64, W=12, alpha=1.0, dtype=__import__("torch").float32)
    assert lib.sfa_forward_layers_workspace_size(f32.ref(), L, None) == 0
    null = ctypes.c_void_p(0)
    al = (ctypes.c_float * L)(1.0, 0.8, 1.2)
    ptrs = (ctypes.c_void_p * L)(16, 16, 16)
    assert lib.sfa_forward_layers(p.ref(), 0, al, win, ptrs, ptrs, ptrs, null, ptrs, None, null,
                                  0, null, null) == _lib.SFA_ERR_INVALID_ARG
    assert lib.sfa_forward_layers(p.ref(), L, None, win, ptrs, ptrs, ptrs, null, ptrs, None, null,
                                  0, null, null) == _lib.SFA_ERR_INVALID_ARG
    bad = (ctypes.c_float * L)(1.0, -0.5, 1.2)                      # alpha must be > 0
    assert lib.sfa_forward_layers(p.ref(), L, bad, win, ptrs, ptrs, ptrs, null, ptrs, None, null,
                                  0, null, null) == _lib.SFA_ERR_INVALID_ARG
    mis = (ctypes.c_void_p * L)(16, 24, 16)                          # misaligned layer 1
    assert lib.sfa_forward_layers(p.ref(), L, al, win, mis, ptrs, ptrs, null, ptrs, None, null,
                                  0, null, null) == _lib.SFA_ERR_INVALID_ARG


def test_decode_host_checks(lib):
    """Argument checks of the decode (nothing is launched)."""
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(256)
    p = api.Params(2, 64, W=12, alpha=1.0, rope_theta=0.0)
    assert lib.sfa_decode(p.ref(), fake, fake, fake, null, null, fake, None, null,
                          null) == _lib.SFA_ERR_INVALID_ARG           # no positions
    assert lib.sfa_decode(p.ref(), fake, fake, fake, ctypes.c_void_p(258), null, fake, None, null,
                          null) == _lib.SFA_ERR_INVALID_ARG           # misaligned positions
    empty = api.Params(2, 0, W=12, alpha=1.0, rope_theta=0.0)
    assert lib.sfa_decode(empty.ref(), fake, fake, fake, fake, null, fake, None, null,
                          null) == _lib.SFA_ERR_INVALID_ARG           # empty cache
    none = api.Params(0, 64, W=12, alpha=1.0, rope_theta=0.0)
    assert lib.sfa_decode(none.ref(), null, null, null, null, null, null, None, null,
                          null) == _lib.SFA_OK                        # nothing to do


def test_qkv_rope_validation(lib):
    """Host checks of sfa_qkv_rope (no launch): dtype, d_model, pointers."""
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails validation
    odd = ctypes.c_void_p(0x10008)
    tab = ctypes.c_void_p(0x20000)
    p = api.Params(2, 64, W=0, alpha=1.0)
    args = lambda dm, x=fake, t=tab: (p.ref(), dm, x, fake, t, fake, fake, fake, None, None)
    assert lib.sfa_qkv_rope(*args(100)) == _lib.SFA_ERR_INVALID_ARG      # not a multiple of 64
    assert lib.sfa_qkv_rope(*args(0)) == _lib.SFA_ERR_INVALID_ARG
    assert lib.sfa_qkv_rope(*args(32768)) == _lib.SFA_ERR_INVALID_ARG
    assert lib.sfa_qkv_rope(*args(512, x=odd)) == _lib.SFA_ERR_INVALID_ARG   # misaligned X
    assert lib.sfa_qkv_rope(*args(512, t=None)) == _lib.SFA_ERR_INVALID_ARG  # RoPE without a table
    p32 = api.Params(2, 64, W=0, alpha=1.0, dtype=__import__("torch").float32)
    assert lib.sfa_qkv_rope(p32.ref(), 512, fake, fake, tab, fake, fake, fake, None, None) == \
        _lib.SFA_ERR_UNSUPPORTED
    empty = api.Params(0, 64, W=0, alpha=1.0)
    assert lib.sfa_qkv_rope(empty.ref(), 512, None, None, None, None, None, None, None, None) == \
        _lib.SFA_OK
