"""Python binding of libsfa: the C ABI calls with the same names, over torch
tensors.  Argument marshalling only -- every step of the attention runs in the
library's CUDA kernels; torch supplies device memory and streams.

Method: "Depth-Staggered Fibonacci Spacing for Sparse Attention: Static
Schedules Beat Learned Dilation and Extrapolate Where Dense Attention Fails"
(arXiv 2606.28560), section 2 "Method".
"""
from __future__ import annotations

import ctypes
import math
from typing import Sequence

import torch

from . import _lib

FIBONACCI_BASE = (1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610, 987)
"""Section 2 "Attended set": the base offsets f_k, K = 15."""


def pow2_base(T: int) -> tuple:
    """Section 2 "Control base": the reach-matched power-of-two base, every
    2^k below the sequence length T (K = 10 at T = 1024)."""
    out, x = [], 1
    while x < T:
        out.append(x)
        x *= 2
    return tuple(out)


_DTYPES = {torch.float32: _lib.SFA_F32, torch.bfloat16: _lib.SFA_BF16}


def _vp(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device, stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


class Params:
    """An sfa_params struct plus the host rung array it points to."""

    def __init__(self, B, T, *, W, alpha, rungs=FIBONACCI_BASE, rope_theta=1e4, scale=0.0,
                 dtype=torch.bfloat16, Hq=8, Hkv=2, D=64, round_offsets=False):
        self._rungs = (ctypes.c_float * max(1, len(rungs)))(*[float(f) for f in rungs])
        p = _lib.SfaParams()
        p.B, p.T, p.Hq, p.Hkv, p.D = int(B), int(T), int(Hq), int(Hkv), int(D)
        p.W, p.K = int(W), len(rungs)
        p.rungs = ctypes.cast(self._rungs, ctypes.POINTER(ctypes.c_float))
        p.alpha = float(alpha)
        p.rope_theta = float(rope_theta)
        p.scale = float(scale)
        if dtype not in _DTYPES:
            raise TypeError(f"unsupported dtype {dtype}")
        p.dtype = _DTYPES[dtype]
        p.round_offsets = 1 if round_offsets else 0
        self.struct = p

    def ref(self):
        return ctypes.byref(self.struct)


# ------------------------------------------------------- host-side helpers --


def alpha_from_theta(theta: float) -> float:
    """alpha = 0.5 + sigmoid(theta) (section 2 "Per-layer scalar")."""
    return float(_lib.load().sfa_alpha_from_theta(float(theta)))


def alpha_schedule(kind: str, L: int = 16, S: int = 7, thetas: Sequence[float] | None = None) -> list:
    """Per-layer alphas of the fixed, learned, linear or coprime schedule."""
    lib = _lib.load()
    out = (ctypes.c_float * L)()
    th = (ctypes.c_float * L)(*[float(t) for t in thetas]) if thetas is not None else None
    st = lib.sfa_alpha_schedule(_lib.SCHEDULES[kind], int(L), int(S),
                                ctypes.cast(th, ctypes.POINTER(ctypes.c_float)) if th else None,
                                ctypes.cast(out, ctypes.POINTER(ctypes.c_float)))
    _lib.check(st, "sfa_alpha_schedule")
    return [float(x) for x in out]


def rung_plan(*, T: int, W: int, alpha: float, rungs=FIBONACCI_BASE, B: int = 1,
              round_offsets: bool = False):
    """The rungs the kernels use: list of (index, floor d, t, ceil d)."""
    lib = _lib.load()
    p = Params(B, T, W=W, alpha=alpha, rungs=rungs, round_offsets=round_offsets)
    K = max(1, len(rungs))
    n = ctypes.c_int(0)
    idx, fl, ce = (ctypes.c_int * K)(), (ctypes.c_int * K)(), (ctypes.c_int * K)()
    fr = (ctypes.c_float * K)()
    st = lib.sfa_rung_plan(p.ref(), ctypes.byref(n), idx, fl, fr, ce)
    _lib.check(st, "sfa_rung_plan")
    return [(idx[i], fl[i], float(fr[i]), ce[i]) for i in range(n.value)]


def launch_count() -> int:
    return int(_lib.load().sfa_launch_count())


# ------------------------------------------------------------- RoPE table --

_rope_cache: dict = {}


def rope_table(T: int, device, D: int = 64, rope_theta: float = 1e4, stream=None) -> torch.Tensor:
    """Device RoPE table [T, D/2, 2] (cos, sin), built once per (device, D,
    theta) and grown on demand; any table with >= T rows serves length T."""
    device = torch.device(device)
    key = (device.index if device.index is not None else torch.cuda.current_device(), D,
           float(rope_theta))
    tab = _rope_cache.get(key)
    if tab is None or tab.shape[0] < T:
        rows = max(T, 1024 if tab is None else 2 * tab.shape[0])
        lib = _lib.load()
        n = lib.sfa_rope_table_floats(int(rows), int(D))
        tab = torch.empty(n, dtype=torch.float32, device=device).view(rows, D // 2, 2)
        st = lib.sfa_rope_table(_vp(tab), int(rows), int(D), float(rope_theta), _stream(device, stream))
        _lib.check(st, "sfa_rope_table")
        # the table is shared by later calls on any stream: finish building it
        (stream if stream is not None else torch.cuda.current_stream(device)).synchronize()
        _rope_cache[key] = tab
    return tab


# -------------------------------------------------------- forward/backward --


def _check_qkv(q, k, v):
    for name, t, H in (("q", q, 8), ("k", k, 2), ("v", v, 2)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or t.shape[2] != H or t.shape[3] != 64:
            raise ValueError(f"{name} must be [B, T, {H}, 64], got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.dtype != q.dtype:
            raise ValueError("q, k, v must share a dtype")
    if k.shape[:2] != q.shape[:2] or v.shape[:2] != q.shape[:2]:
        raise ValueError("q, k, v must share B and T")


_ws_cache: dict = {}


def _workspace(device, nbytes: int) -> torch.Tensor:
    """A per-device scratch buffer of at least nbytes (grown on demand).  Calls
    on one device share it, so they must be ordered on one stream."""
    key = torch.device(device)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=key)
        _ws_cache[key] = buf
    return buf


def sfa_forward(q, k, v, *, alpha: float, W: int, rungs=FIBONACCI_BASE, rope_theta: float = 1e4,
                scale: float = 0.0, need_lse: bool = True, out=None, lse=None, status=None,
                workspace=None, stream=None, round_offsets: bool = False):
    """O (and LSE) of the sparse attention for one layer; see include/sfa.h."""
    _check_qkv(q, k, v)
    B, T = q.shape[0], q.shape[1]
    o = out if out is not None else torch.empty_like(q)
    if need_lse and lse is None:
        lse = torch.empty((B, T, 8), dtype=torch.float32, device=q.device)
    p = Params(B, T, W=W, alpha=alpha, rungs=rungs, rope_theta=rope_theta, scale=scale,
               dtype=q.dtype, round_offsets=round_offsets)
    lib = _lib.load()
    need = int(lib.sfa_forward_workspace_size(p.ref()))
    if workspace is None or workspace.numel() < need:
        workspace = _workspace(q.device, need) if need else None
    tab = rope_table(T, q.device, rope_theta=rope_theta, stream=stream) if rope_theta > 0 else None
    st = lib.sfa_forward(p.ref(), _vp(q), _vp(k), _vp(v), _vp(tab), _vp(o),
                         _vp(lse if need_lse else None), _vp(workspace),
                         ctypes.c_size_t(workspace.numel() if workspace is not None else 0),
                         _vp(status), _stream(q.device, stream))
    _lib.check(st, "sfa_forward")
    return o, (lse if need_lse else None)


def _ptrs(ts) -> ctypes.Array:
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() if t is not None else 0 for t in ts])


def sfa_forward_layers(qs, ks, vs, *, alphas, W, rungs=FIBONACCI_BASE, rope_theta: float = 1e4,
                       scale: float = 0.0, need_lse: bool = True, outs=None, lses=None,
                       status=None, workspace=None, stream=None, round_offsets: bool = False):
    """The forwards of L layers in one call (sfa_forward_layers in
    include/sfa.h): qs, ks, vs are lists of per-layer tensors, alphas the L
    per-layer scalars, W one window or a list of L windows."""
    L = len(qs)
    if not (len(ks) == len(vs) == len(alphas) == L) or L == 0:
        raise ValueError("qs, ks, vs and alphas must have one entry per layer")
    for q, k, v in zip(qs, ks, vs):
        _check_qkv(q, k, v)
        if q.shape != qs[0].shape or q.dtype != qs[0].dtype or q.device != qs[0].device:
            raise ValueError("all layers must share shape, dtype and device")
    B, T = qs[0].shape[0], qs[0].shape[1]
    dev = qs[0].device
    outs = outs if outs is not None else [torch.empty_like(q) for q in qs]
    if need_lse and lses is None:
        lses = [torch.empty((B, T, 8), dtype=torch.float32, device=dev) for _ in range(L)]
    windows = [int(W)] * L if isinstance(W, int) else [int(w) for w in W]
    p = Params(B, T, W=windows[0], alpha=alphas[0], rungs=rungs, rope_theta=rope_theta,
               scale=scale, dtype=qs[0].dtype, round_offsets=round_offsets)
    win = (ctypes.c_int * L)(*windows)
    al = (ctypes.c_float * L)(*[float(a) for a in alphas])
    lib = _lib.load()
    need = int(lib.sfa_forward_layers_workspace_size(p.ref(), L, win))
    if workspace is None or workspace.numel() < need:
        workspace = _workspace(dev, need) if need else None
    tab = rope_table(T, dev, rope_theta=rope_theta, stream=stream) if rope_theta > 0 else None
    lse_arr = _ptrs(lses) if need_lse else None
    st = lib.sfa_forward_layers(p.ref(), L, al, win, _ptrs(qs), _ptrs(ks), _ptrs(vs), _vp(tab),
                                _ptrs(outs), lse_arr, _vp(workspace),
                                ctypes.c_size_t(workspace.numel() if workspace is not None else 0),
                                _vp(status), _stream(dev, stream))
    _lib.check(st, "sfa_forward_layers")
    return outs, (lses if need_lse else None)


def sfa_decode(q, k_cache, v_cache, positions, *, alpha: float, W: int, rungs=FIBONACCI_BASE,
               rope_theta: float = 1e4, scale: float = 0.0, need_lse: bool = True, out=None,
               lse=None, status=None, stream=None, round_offsets: bool = False):
    """One new query per sequence over a key/value cache (sfa_decode in
    include/sfa.h): q [B, 8, 64], caches [B, Tc, 2, 64], positions int32 [B]
    on the device; returns O [B, 8, 64] and LSE [B, 8]."""
    if q.dim() != 3 or q.shape[1] != 8 or q.shape[2] != 64 or not q.is_contiguous():
        raise ValueError(f"q must be a contiguous [B, 8, 64] tensor, got {tuple(q.shape)}")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if (t.dim() != 4 or t.shape[0] != q.shape[0] or t.shape[2] != 2 or t.shape[3] != 64
                or not t.is_contiguous() or t.dtype != q.dtype or t.device != q.device):
            raise ValueError(f"{name} must be a contiguous [B, Tc, 2, 64] tensor like q")
    if (positions.dtype != torch.int32 or positions.shape != (q.shape[0],)
            or positions.device != q.device):
        raise ValueError("positions must be an int32 [B] tensor on q's device")
    B, Tc = q.shape[0], k_cache.shape[1]
    o = out if out is not None else torch.empty_like(q)
    if need_lse and lse is None:
        lse = torch.empty((B, 8), dtype=torch.float32, device=q.device)
    p = Params(B, Tc, W=W, alpha=alpha, rungs=rungs, rope_theta=rope_theta, scale=scale,
               dtype=q.dtype, round_offsets=round_offsets)
    tab = rope_table(Tc, q.device, rope_theta=rope_theta, stream=stream) if rope_theta > 0 else None
    st = _lib.load().sfa_decode(p.ref(), _vp(q), _vp(k_cache), _vp(v_cache), _vp(positions),
                                _vp(tab), _vp(o), _vp(lse if need_lse else None), _vp(status),
                                _stream(q.device, stream))
    _lib.check(st, "sfa_decode")
    return o, (lse if need_lse else None)


def sfa_selftest_wait_timeout(status, stream=None):
    """Runs the failure-path self-test (sfa_selftest_wait_timeout in
    include/sfa.h) on status's device: a bounded wait that nothing satisfies
    gives up and sets SFA_DEVSTAT_WAIT_TIMEOUT in the int32 word ``status``."""
    st = _lib.load().sfa_selftest_wait_timeout(_vp(status), _stream(status.device, stream))
    _lib.check(st, "sfa_selftest_wait_timeout")


def sfa_qkv_rope(x, w_qkv, *, rope_theta: float = 1e4, out=None, status=None, stream=None):
    """The fused front end (sfa_qkv_rope in include/sfa.h): x [B, T, d_model]
    and w_qkv [768, d_model] bf16 on the device; returns (qhat [B, T, 8, 64],
    khat [B, T, 2, 64], v [B, T, 2, 64]) with RoPE applied to qhat and khat,
    ready for sfa_forward(..., rope_theta=0)."""
    if x.dim() != 3 or x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError(f"x must be a contiguous bf16 [B, T, d_model] tensor, got {tuple(x.shape)}")
    B, T, dm = x.shape
    if (w_qkv.shape != (768, dm) or w_qkv.dtype != torch.bfloat16 or not w_qkv.is_contiguous()
            or w_qkv.device != x.device):
        raise ValueError(f"w_qkv must be a contiguous bf16 [768, {dm}] tensor on x's device")
    if out is None:
        out = (torch.empty((B, T, 8, 64), dtype=x.dtype, device=x.device),
               torch.empty((B, T, 2, 64), dtype=x.dtype, device=x.device),
               torch.empty((B, T, 2, 64), dtype=x.dtype, device=x.device))
    qh, kh, v = out
    p = Params(B, T, W=0, alpha=1.0, rope_theta=rope_theta, dtype=x.dtype)
    tab = rope_table(T, x.device, rope_theta=rope_theta, stream=stream) if rope_theta > 0 else None
    st = _lib.load().sfa_qkv_rope(p.ref(), int(dm), _vp(x), _vp(w_qkv), _vp(tab), _vp(qh), _vp(kh),
                                  _vp(v), _vp(status), _stream(x.device, stream))
    _lib.check(st, "sfa_qkv_rope")
    return qh, kh, v


def sfa_forward_noalloc(q, k, v, *, alpha: float, W: int, rungs=FIBONACCI_BASE,
                        rope_theta: float = 1e4, scale: float = 0.0, out, lse=None, rope=None,
                        status=None, stream=None):
    """sfa_forward without a workspace, for callers that cannot allocate device
    memory: the scratch lives in a fixed array inside the library.  The caller
    passes every buffer (``out``, ``lse`` and, when rope_theta > 0, a RoPE
    table ``rope`` from sfa_rope_table); nothing is allocated here."""
    _check_qkv(q, k, v)
    B, T = q.shape[0], q.shape[1]
    p = Params(B, T, W=W, alpha=alpha, rungs=rungs, rope_theta=rope_theta, scale=scale,
               dtype=q.dtype)
    st = _lib.load().sfa_forward_noalloc(p.ref(), _vp(q), _vp(k), _vp(v), _vp(rope), _vp(out),
                                         _vp(lse), _vp(status), _stream(q.device, stream))
    _lib.check(st, "sfa_forward_noalloc")
    return out, lse


def sfa_backward_workspace_size(B: int, T: int, *, alpha: float, W: int, rungs=FIBONACCI_BASE,
                                dtype=torch.bfloat16, round_offsets: bool = False) -> int:
    p = Params(B, T, W=W, alpha=alpha, rungs=rungs, dtype=dtype, round_offsets=round_offsets)
    return int(_lib.load().sfa_backward_workspace_size(p.ref()))


def sfa_backward(q, k, v, o, dO, lse, *, alpha: float, W: int, rungs=FIBONACCI_BASE,
                 rope_theta: float = 1e4, scale: float = 0.0, workspace=None, status=None,
                 stream=None, out=None, round_offsets: bool = False):
    """(dQ, dK, dV, dalpha, dtheta) of the sparse attention; dalpha/dtheta are
    one-element fp32 device tensors.  ``out`` may supply the five output
    tensors (then nothing is allocated here)."""
    _check_qkv(q, k, v)
    B, T = q.shape[0], q.shape[1]
    for name, t in (("o", o), ("dO", dO)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must match q")
    p = Params(B, T, W=W, alpha=alpha, rungs=rungs, rope_theta=rope_theta, scale=scale,
               dtype=q.dtype, round_offsets=round_offsets)
    lib = _lib.load()
    need = int(lib.sfa_backward_workspace_size(p.ref()))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is not None:
        dq, dk, dv, da, dth = out
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        da = torch.empty(1, dtype=torch.float32, device=q.device)
        dth = torch.empty(1, dtype=torch.float32, device=q.device)
    tab = rope_table(T, q.device, rope_theta=rope_theta, stream=stream) if rope_theta > 0 else None
    st = lib.sfa_backward(p.ref(), _vp(q), _vp(k), _vp(v), _vp(o), _vp(dO), _vp(lse), _vp(tab),
                          _vp(dq), _vp(dk), _vp(dv), _vp(da), _vp(dth), _vp(workspace),
                          ctypes.c_size_t(workspace.numel()), _vp(status),
                          _stream(q.device, stream))
    _lib.check(st, "sfa_backward")
    return dq, dk, dv, da, dth


def sfa_read_status(status: torch.Tensor, stream=None) -> int:
    """Synchronises and returns the device status word (0 = no error)."""
    w = ctypes.c_uint(0)
    st = _lib.load().sfa_read_status(_vp(status), ctypes.byref(w), _stream(status.device, stream))
    if st not in (_lib.SFA_OK, _lib.SFA_ERR_DEVICE_STATUS):
        _lib.check(st, "sfa_read_status")
    return int(w.value)


class SparseAttention(torch.autograd.Function):
    """Autograd wrapper: o = attention(q, k, v; alpha = 0.5 + sigmoid(theta)).

    theta is a 0-d tensor (the layer's only added parameter); its gradient is
    the library's dtheta."""

    @staticmethod
    def forward(ctx, q, k, v, theta, W, rungs=FIBONACCI_BASE, rope_theta=1e4):
        alpha = alpha_from_theta(float(theta))
        o, lse = sfa_forward(q, k, v, alpha=alpha, W=W, rungs=rungs, rope_theta=rope_theta)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.cfg = (alpha, W, tuple(rungs), rope_theta)
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse = ctx.saved_tensors
        alpha, W, rungs, rope_theta = ctx.cfg
        dq, dk, dv, _, dth = sfa_backward(q, k, v, o, dO.contiguous(), lse, alpha=alpha, W=W,
                                          rungs=rungs, rope_theta=rope_theta)
        return dq, dk, dv, dth.reshape(()), None, None, None
