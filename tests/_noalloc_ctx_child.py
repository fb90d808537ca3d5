"""Child process of tests/test_zz_no_alloc.py: sfa_forward and
sfa_forward_noalloc inside CUDA contexts that the caller creates itself with
the driver API (as a plugin in a host application may), switching between
two of them.  Device memory comes from cuMemAlloc in the context current at
each call; torch is used on the CPU only (seeded inputs), so this process has
no other CUDA context.  Exits 0 when every pair of outputs is bit-identical
and the same inputs give the same outputs in both contexts."""
import ctypes
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from fibonacci_spaced_sparse_gb300 import _lib, api, inputs  # noqa: E402

cu = ctypes.CDLL("libcuda.so.1")
lib = _lib.load()


def ck(r, what):
    if r != 0:
        raise SystemExit(f"{what} failed with CUresult {r}")


def sfa(st, what):
    if st != _lib.SFA_OK:
        raise SystemExit(f"{what}: {_lib.strerror(st)}")


def alloc(nbytes, held):
    p = ctypes.c_uint64(0)
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
    held.append(p)
    return ctypes.c_void_p(p.value)


def upload(t, held):
    a = t.contiguous().view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.contiguous().numpy()
    d = alloc(a.nbytes, held)
    ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(d.value), a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)),
       "cuMemcpyHtoD")
    return d


def download(d, nbytes, dtype):
    a = np.empty(nbytes // np.dtype(dtype).itemsize, dtype=dtype)
    ck(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(d.value), ctypes.c_size_t(nbytes)),
       "cuMemcpyDtoH")
    return a


B, T, W = 2, 300, 12


def run_in(ctx, layer, alpha):
    """Both forwards of one seeded layer in context ctx; returns (O, LSE)."""
    ck(cu.cuCtxSetCurrent(ctx), "cuCtxSetCurrent")
    held = []
    x = inputs.qkv(B, T, dtype=torch.bfloat16, layer=layer)
    q, k, v = (upload(x[n], held) for n in ("q", "k", "v"))
    obytes, lbytes = B * T * 8 * 64 * 2, B * T * 8 * 4
    o1, o2, l1, l2 = alloc(obytes, held), alloc(obytes, held), alloc(lbytes, held), alloc(lbytes, held)
    tab = alloc(lib.sfa_rope_table_floats(T, 64) * 4, held)
    sfa(lib.sfa_rope_table(tab, T, 64, 1e4, None), "sfa_rope_table")
    p = api.Params(B, T, W=W, alpha=alpha)
    wsz = lib.sfa_forward_workspace_size(p.ref())
    ws = alloc(wsz, held)
    sfa(lib.sfa_forward(p.ref(), q, k, v, tab, o1, l1, ws, wsz, None, None), "sfa_forward")
    sfa(lib.sfa_forward_noalloc(p.ref(), q, k, v, tab, o2, l2, None, None), "sfa_forward_noalloc")
    ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    a_o, b_o = download(o1, obytes, np.int16), download(o2, obytes, np.int16)
    a_l, b_l = download(l1, lbytes, np.float32), download(l2, lbytes, np.float32)
    for h in held:
        ck(cu.cuMemFree_v2(h), "cuMemFree")
    if not (np.array_equal(a_o, b_o) and np.array_equal(a_l, b_l)):
        raise SystemExit(f"layer {layer}: sfa_forward_noalloc differs from sfa_forward")
    return a_o, a_l


def main():
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int(0)
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    ctxs = []
    for _ in range(2):
        c = ctypes.c_void_p(0)
        ck(cu.cuCtxCreate_v4(ctypes.byref(c), None, 0, dev), "cuCtxCreate")
        ctxs.append(c)
    first = run_in(ctxs[0], 3, 0.81)
    run_in(ctxs[1], 4, 1.37)
    again = run_in(ctxs[1], 3, 0.81)
    back = run_in(ctxs[0], 3, 0.81)
    for got in (again, back):
        if not (np.array_equal(first[0], got[0]) and np.array_equal(first[1], got[1])):
            raise SystemExit("the same layer gave different outputs in the two contexts")
    for c in ctxs:
        ck(cu.cuCtxDestroy_v2(c), "cuCtxDestroy")
    print("ok")


if __name__ == "__main__":
    main()
