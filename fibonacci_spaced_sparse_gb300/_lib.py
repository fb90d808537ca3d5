"""ctypes view of libsfa (the C ABI in include/sfa.h).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsfa.so")

SFA_OK = 0
SFA_ERR_INVALID_ARG = 1
SFA_ERR_UNSUPPORTED = 2
SFA_ERR_CUDA = 3
SFA_ERR_DEVICE_STATUS = 4
SFA_F32 = 0
SFA_BF16 = 1
SFA_MAX_RUNGS = 32

SCHEDULES = {"fixed": 0, "learned": 1, "linear": 2, "coprime": 3}


class SfaParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("W", ctypes.c_int), ("K", ctypes.c_int),
        ("rungs", ctypes.POINTER(ctypes.c_float)),
        ("alpha", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("scale", ctypes.c_float), ("dtype", ctypes.c_int),
        ("round_offsets", ctypes.c_int),
    ]


class SfaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


_lib = None

_VP = ctypes.c_void_p
_FP = ctypes.POINTER(ctypes.c_float)
_IP = ctypes.POINTER(ctypes.c_int)
_PP = ctypes.POINTER(SfaParams)

_SIGS = {
    "sfa_version": ([], ctypes.c_int),
    "sfa_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "sfa_launch_count": ([], ctypes.c_ulonglong),
    "sfa_alpha_from_theta": ([ctypes.c_float], ctypes.c_float),
    "sfa_alpha_schedule": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, _FP, _FP], ctypes.c_int),
    "sfa_rung_plan": ([_PP, _IP, _IP, _IP, _FP, _IP], ctypes.c_int),
    "sfa_rope_table_floats": ([ctypes.c_int, ctypes.c_int], ctypes.c_size_t),
    "sfa_rope_table": ([_VP, ctypes.c_int, ctypes.c_int, ctypes.c_float, _VP], ctypes.c_int),
    "sfa_forward_workspace_size": ([_PP], ctypes.c_size_t),
    "sfa_forward": ([_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP, _VP],
                    ctypes.c_int),
    "sfa_forward_layers_workspace_size": ([_PP, ctypes.c_int, _IP], ctypes.c_size_t),
    "sfa_forward_layers": ([_PP, ctypes.c_int, _FP, _IP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                            ctypes.c_size_t, _VP, _VP], ctypes.c_int),
    "sfa_forward_noalloc_scratch_bytes": ([], ctypes.c_size_t),
    "sfa_forward_noalloc": ([_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "sfa_decode": ([_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "sfa_selftest_wait_timeout": ([_VP, _VP], ctypes.c_int),
    "sfa_qkv_rope": ([_PP, ctypes.c_int, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "sfa_backward_workspace_size": ([_PP], ctypes.c_size_t),
    "sfa_backward": ([_PP] + [_VP] * 13 + [ctypes.c_size_t, _VP, _VP], ctypes.c_int),
    "sfa_read_status": ([_VP, ctypes.POINTER(ctypes.c_uint), _VP], ctypes.c_int),
}


def load():
    """The loaded library (ctypes.CDLL); raises if libsfa.so is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libsfa.so is not built ({LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def strerror(code: int) -> str:
    try:
        return load().sfa_strerror(int(code)).decode()
    except Exception:  # pragma: no cover - only when the library itself is absent
        return f"status {code}"


def check(code: int, where: str) -> None:
    if code != SFA_OK:
        raise SfaError(code, where)
