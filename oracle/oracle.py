"""CPU oracle for depth-staggered Fibonacci sparse attention (fp64).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
(``__graft_entry__.smoke``) and by the CPU-baseline leg of ``bench.py``.  The
product path never imports it and it imports nothing from the product package.

The arithmetic lives in ``sfa_oracle.c`` (plain C, fp64, an explicit per-query
key list); this module compiles it with gcc, loads it with ctypes and adds the
oracle's own statement of the per-layer schedules and base-offset tables.

Every rule is from "Depth-Staggered Fibonacci Spacing for Sparse Attention:
Static Schedules Beat Learned Dilation and Extrapolate Where Dense Attention
Fails" (arXiv 2606.28560):
  * section 2, "Attended set": base offsets 1, 2, 3, 5, ..., 987 (K = 15);
  * section 2, "Per-layer scalar": alpha = 0.5 + sigmoid(theta); the fixed,
    learned, linear-stagger and coprime (S = 7) schedules over L = 16 layers;
  * section 2, "Control base": the reach-matched power-of-two base.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

# ------------------------------------------------------------------ build --


def build(force: bool = False) -> str:
    """Compile sfa_oracle.c into oracle/_build/liboracle.so (gcc, portable C)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("Hq", ctypes.c_int),
        ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("W", ctypes.c_int),
        ("K", ctypes.c_int), ("f", ctypes.POINTER(ctypes.c_double)),
        ("alpha", ctypes.c_double), ("d_fp32", ctypes.c_int),
        ("rope_theta", ctypes.c_double), ("scale", ctypes.c_double),
        ("nthreads", ctypes.c_int), ("round_offsets", ctypes.c_int),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        cp = ctypes.POINTER(_Cfg)
        lib.oracle_forward.argtypes = [cp, dp, dp, dp, dp, dp]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_forward_rows.argtypes = [cp, dp, dp, dp, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_int), dp, dp]
        lib.oracle_forward_rows.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [cp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_rope.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double, ctypes.c_int, dp, dp]
        lib.oracle_rope.restype = None
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _cfg(shape, W, rungs, alpha, d_fp32, rope_theta, scale, nthreads, round_offsets=False):
    B, T, Hq, D = shape[0], shape[1], shape[2], shape[3]
    f = _f64(rungs)
    cfg = _Cfg()
    cfg.B, cfg.T, cfg.Hq, cfg.D = B, T, Hq, D
    cfg.W, cfg.K = int(W), int(f.size)
    cfg.f = _ptr(f) if f.size else ctypes.POINTER(ctypes.c_double)()
    cfg.alpha = float(alpha)
    cfg.d_fp32 = 1 if d_fp32 else 0
    cfg.rope_theta = float(rope_theta)
    cfg.scale = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    cfg.nthreads = int(nthreads) if nthreads else default_threads()
    cfg.round_offsets = 1 if round_offsets else 0
    return cfg, f


# ------------------------------------------------------------- attention --


def forward(q, k, v, *, W: int, rungs: Sequence[float], alpha: float,
            rope_theta: float = 1e4, scale: float | None = None,
            d_fp32: bool = True, nthreads: int | None = None,
            round_offsets: bool = False):
    """O [B,T,Hq,D] and LSE [B,T,Hq] of the sparse attention, fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cfg, keep = _cfg(q.shape, W, rungs, alpha, d_fp32, rope_theta, scale, nthreads, round_offsets)
    cfg.Hkv = k.shape[2]
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:3], dtype=np.float64)
    st = _load().oracle_forward(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse))
    if st:
        raise RuntimeError(f"oracle_forward failed ({st})")
    del keep
    return o, lse


def forward_rows(q, k, v, rows, *, W: int, rungs: Sequence[float], alpha: float,
                 rope_theta: float = 1e4, scale: float | None = None,
                 d_fp32: bool = True, nthreads: int | None = None,
                 round_offsets: bool = False):
    """O and LSE of the sampled query rows ``rows`` (array of (b, i) pairs)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    cfg, keep = _cfg(q.shape, W, rungs, alpha, d_fp32, rope_theta, scale, nthreads, round_offsets)
    cfg.Hkv = k.shape[2]
    n = rows.shape[0]
    o = np.zeros((n, q.shape[2], q.shape[3]), dtype=np.float64)
    lse = np.zeros((n, q.shape[2]), dtype=np.float64)
    st = _load().oracle_forward_rows(
        ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), n,
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), _ptr(o), _ptr(lse))
    if st:
        raise RuntimeError(f"oracle_forward_rows failed ({st})")
    del keep
    return o, lse


def backward(q, k, v, dO, *, W: int, rungs: Sequence[float], alpha: float,
             rope_theta: float = 1e4, scale: float | None = None,
             d_fp32: bool = True, nthreads: int | None = None,
             round_offsets: bool = False):
    """(dq, dk, dv, dalpha, dtheta, dt) of L = sum(dO * O), fp64."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    cfg, keep = _cfg(q.shape, W, rungs, alpha, d_fp32, rope_theta, scale, nthreads, round_offsets)
    cfg.Hkv = k.shape[2]
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    da = ctypes.c_double(0.0)
    dth = ctypes.c_double(0.0)
    dt = np.zeros(max(1, len(keep)), dtype=np.float64)
    st = _load().oracle_backward(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(dO),
                                 _ptr(dq), _ptr(dk), _ptr(dv), ctypes.byref(da),
                                 ctypes.byref(dth), _ptr(dt))
    if st:
        raise RuntimeError(f"oracle_backward failed ({st})")
    return dq, dk, dv, da.value, dth.value, dt[:len(keep)]


def rope(x, rope_theta: float = 1e4, inverse: bool = False) -> np.ndarray:
    """x [B,T,H,D] rotated at its true positions (rotate-half pairing)."""
    x = _f64(x)
    y = np.zeros_like(x)
    B, T, H, D = x.shape
    _load().oracle_rope(B, T, H, D, float(rope_theta), 1 if inverse else 0, _ptr(x), _ptr(y))
    return y


def qkv_rope(x, w, *, Hq: int = 8, Hkv: int = 2, D: int = 64, rope_theta: float = 1e4):
    """The front end of a layer in fp64: [Q | K | V] = x w^T (section 3,
    "Model and training": d_model 512, 8 query and 2 key/value heads of
    dimension 64), then Q and K rotated at their true positions (section 2,
    "Attended set": RoPE before any key row is gathered).

    x [B, T, d_model]; w [(Hq + 2 Hkv) D, d_model], the rows of query head h
    first (h D .. h D + D - 1), then the key heads, then the value heads.
    Returns (qhat [B,T,Hq,D], khat [B,T,Hkv,D], v [B,T,Hkv,D])."""
    x, w = _f64(x), _f64(w)
    B, T, dm = x.shape
    if w.shape != ((Hq + 2 * Hkv) * D, dm):
        raise ValueError(f"w must be [{(Hq + 2 * Hkv) * D}, {dm}], got {w.shape}")
    y = x.reshape(B * T, dm) @ w.T
    q = np.ascontiguousarray(y[:, :Hq * D]).reshape(B, T, Hq, D)
    k = np.ascontiguousarray(y[:, Hq * D:(Hq + Hkv) * D]).reshape(B, T, Hkv, D)
    v = np.ascontiguousarray(y[:, (Hq + Hkv) * D:]).reshape(B, T, Hkv, D)
    if rope_theta > 0:
        q, k = rope(q, rope_theta), rope(k, rope_theta)
    return q, k, v


# ---------------------------------------------- schedules and base tables --

FIBONACCI_BASE = (1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610, 987)
"""Section 2, "Attended set": the base sequence, K = 15."""


def pow2_base(T: int) -> tuple:
    """Section 2, "Control base": the reach-matched power-of-two base, read as
    every 2^k below the sequence length (so a 4096-token sequence gains the
    offsets 1024 and 2048)."""
    out, x = [], 1
    while x < T:
        out.append(x)
        x *= 2
    return tuple(out)


def alpha_from_theta(theta: float) -> float:
    """Section 2, "Per-layer scalar": alpha = 0.5 + sigmoid(theta), in fp64."""
    return 0.5 + 1.0 / (1.0 + math.exp(-theta))


def schedule_fixed(L: int = 16) -> list:
    """alpha_l = 1 for every layer."""
    return [1.0] * L


def schedule_linear(L: int = 16) -> list:
    """alpha_l = 0.5 + l / (L - 1): a ramp from 0.5 at layer 0 to 1.5 at L - 1."""
    return [0.5 + l / (L - 1) for l in range(L)]


def schedule_coprime(L: int = 16, S: int = 7) -> list:
    """The linear ramp's values re-assigned to layers by l -> (S l) mod L:
    layer l takes the ramp value at index (S l) mod L."""
    ramp = schedule_linear(L)
    return [ramp[(S * l) % L] for l in range(L)]


def schedule_learned(thetas) -> list:
    """Per-layer free parameters theta_l mapped through alpha = 0.5 + sigmoid."""
    return [alpha_from_theta(float(t)) for t in thetas]
