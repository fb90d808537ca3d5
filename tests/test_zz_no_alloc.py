"""sfa_forward_noalloc, the forward for callers that cannot allocate device
memory (for example a plugin whose host application owns all device memory):
called through the C ABI, it must give what sfa_forward gives, call after
call, while the caller supplies only inputs and outputs.  This file is named
to be collected last."""
import ctypes

import pytest
import torch

from fibonacci_spaced_sparse_gb300 import _lib, api
from _helpers import TOL, draw, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(xd, out, lse, tab, *, alpha, W, dtype):
    B, T = xd["q"].shape[0], xd["q"].shape[1]
    p = api.Params(B, T, W=W, alpha=alpha, dtype=dtype)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    vp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)
    return _lib.load().sfa_forward_noalloc(p.ref(), vp(xd["q"]), vp(xd["k"]), vp(xd["v"]),
                                           vp(tab), vp(out), vp(lse), ctypes.c_void_p(0), stream)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_forward_twice(dtype):
    torch_dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    B, T, W = 4, 1000, 12
    tab = api.rope_table(T, "cuda")          # caller-owned table, built beforehand
    for call, (layer, alpha) in enumerate([(3, 0.81), (4, 1.37)]):
        x, _ = draw(B, T, dtype, layer=layer)
        xd = to_dev(x)
        ref_o, ref_l = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=W)
        out = torch.full_like(xd["q"], float("nan"))
        lse = torch.full((B, T, 8), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(xd, out, lse, tab, alpha=alpha, W=W, dtype=torch_dt)
        assert st == _lib.SFA_OK, _lib.strerror(st)
        torch.cuda.synchronize()
        assert max_abs(np64(out), np64(ref_o)) <= TOL[dtype]["o"], call
        assert max_abs(np64(lse), np64(ref_l)) <= TOL[dtype]["lse"], call


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _lib.load()
    limit = lib.sfa_forward_noalloc_scratch_bytes()
    assert limit == 8 << 20
    B, T = 33, 1024                          # 33 * 1024 * 2 * 64 * 2 bytes > 8 MiB
    p = api.Params(B, T, W=12, alpha=1.0)
    assert lib.sfa_forward_workspace_size(p.ref()) > limit
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: rejected before any launch
    n0 = api.launch_count()
    st = lib.sfa_forward_noalloc(p.ref(), fake, fake, fake, fake, fake, ctypes.c_void_p(0),
                                 ctypes.c_void_p(0), ctypes.c_void_p(0))
    assert st == _lib.SFA_ERR_UNSUPPORTED and api.launch_count() == n0


def test_noalloc_largest_accepted_shape():
    """B * T = 32768 with RoPE: the rotated keys fill the scratch exactly
    (32768 tokens x 2 heads x 64 x 2 bytes = 8 MiB), and the output is
    bit-identical to sfa_forward's (the same kernels, another workspace)."""
    lib = _lib.load()
    B, T, W, alpha = 32, 1024, 12, 1.13
    p = api.Params(B, T, W=W, alpha=alpha)
    assert lib.sfa_forward_workspace_size(p.ref()) == lib.sfa_forward_noalloc_scratch_bytes()
    x, _ = draw(B, T, "bf16", layer=5)
    xd = to_dev(x)
    tab = api.rope_table(T, "cuda")
    ref_o, ref_l = api.sfa_forward(xd["q"], xd["k"], xd["v"], alpha=alpha, W=W)
    out = torch.full_like(xd["q"], float("nan"))
    lse = torch.full((B, T, 8), float("nan"), dtype=torch.float32, device="cuda")
    st = _noalloc(xd, out, lse, tab, alpha=alpha, W=W, dtype=torch.bfloat16)
    assert st == _lib.SFA_OK, _lib.strerror(st)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_noalloc_in_contexts_the_caller_created():
    """A caller that creates its own CUDA contexts (cuCtxCreate) and switches
    between them: in each context both forwards agree bit for bit, and the
    scratch address and kernel set-up follow the context (a child process, so
    that no other context exists in it)."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "_noalloc_ctx_child.py")], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
