"""The RoPE table (sfa_rope_table): (cos, sin) of pos * theta^(-2m/64) for
every position and pair, built on the GPU in double and stored as fp32,
against numpy's fp64 cos/sin rounded to fp32 -- at short lengths in full and
at the longest accepted length (2^24 positions) on sampled rows."""
import ctypes

import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import _lib

pytestmark = pytest.mark.gpu


def _table(T, D=64, theta=1e4):
    lib = _lib.load()
    n = int(lib.sfa_rope_table_floats(T, D))
    tab = torch.empty(n, dtype=torch.float32, device="cuda")
    st = lib.sfa_rope_table(ctypes.c_void_p(tab.data_ptr()), T, D, float(theta),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(st, "sfa_rope_table")
    torch.cuda.synchronize()
    return tab.view(T, D // 2, 2)


def _expected(pos, D=64, theta=1e4):
    m = np.arange(D // 2, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta ** (-2.0 * m / D)[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


@pytest.mark.parametrize("T,D,theta", [(1, 64, 1e4), (5000, 64, 1e4), (300, 32, 500.0)])
def test_table_matches_fp64_trigonometry(T, D, theta):
    got = _table(T, D, theta).cpu().numpy()
    want = _expected(np.arange(T), D, theta)
    # both sides round a double to fp32; they may differ by one fp32 ulp where
    # the two doubles straddle a rounding boundary
    assert np.max(np.abs(got.astype(np.float64) - want)) <= 2.0 ** -24


def test_table_at_the_longest_sequence():
    T = 1 << 24
    tab = _table(T)
    rng = np.random.default_rng(7)
    pos = np.unique(np.concatenate([np.arange(8), T - 1 - np.arange(8), rng.integers(0, T, 500)]))
    got = tab[torch.from_numpy(pos).cuda()].cpu().numpy()
    want = _expected(pos)
    assert np.max(np.abs(got.astype(np.float64) - want)) <= 2.0 ** -24
    # cos^2 + sin^2 = 1 to fp32 precision everywhere sampled
    r = got[..., 0].astype(np.float64) ** 2 + got[..., 1].astype(np.float64) ** 2
    assert np.max(np.abs(r - 1.0)) <= 4 * 2.0 ** -24
    del tab
    torch.cuda.empty_cache()
