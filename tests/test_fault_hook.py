"""The host fault-injection hook (SFA_TEST_FAULT=launch, include/sfa.h):
every entry point that would launch work checks its arguments as usual and
then fails with SFA_ERR_CUDA before it touches the GPU, so a caller's error
path is exercised with no GPU and no device fault.  Runs in a child process,
because the library reads the variable once."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, json
from fibonacci_spaced_sparse_gb300 import _lib, api
lib = _lib.load()
fake = ctypes.c_void_p(0x100000)    # 16- and 256-byte aligned, never dereferenced
null = ctypes.c_void_p(0)
big = 1 << 40
out = {}
p = api.Params(2, 64, W=12, alpha=1.1)
out["forward"] = lib.sfa_forward(p.ref(), fake, fake, fake, fake, fake, fake, fake, big, null, null)
p32 = api.Params(2, 64, W=12, alpha=1.1, dtype=__import__("torch").float32)
out["forward_f32"] = lib.sfa_forward(p32.ref(), fake, fake, fake, fake, fake, fake, null, 0, null, null)
out["forward_bad_arg"] = lib.sfa_forward(p.ref(), null, fake, fake, fake, fake, fake, fake, big, null, null)
empty = api.Params(0, 64, W=12, alpha=1.1)
out["forward_empty"] = lib.sfa_forward(empty.ref(), null, null, null, null, null, null, null, 0, null, null)
L = 3
ptrs = (ctypes.c_void_p * L)(*([0x100000] * L))
alphas = (ctypes.c_float * L)(0.7, 1.0, 1.3)
out["forward_layers"] = lib.sfa_forward_layers(p.ref(), L, alphas, None, ptrs, ptrs, ptrs, fake, ptrs, None,
                                               fake, big, null, null)
out["backward"] = lib.sfa_backward(p.ref(), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                   fake, fake, fake, big, null, null)
out["backward_empty"] = lib.sfa_backward(empty.ref(), null, null, null, null, null, null, null, null, null,
                                         null, fake, fake, null, 0, null, null)
out["decode"] = lib.sfa_decode(p.ref(), fake, fake, fake, fake, fake, fake, fake, null, null)
out["qkv_rope"] = lib.sfa_qkv_rope(p.ref(), 512, fake, fake, fake, fake, fake, fake, null, null)
out["rope_table"] = lib.sfa_rope_table(fake, 64, 64, 1e4, null)
out["rope_table_empty"] = lib.sfa_rope_table(fake, 0, 64, 1e4, null)
out["selftest"] = lib.sfa_selftest_wait_timeout(fake, null)
out["read_status"] = lib.sfa_read_status(fake, None, null)
print(json.dumps(out))
"""


def test_every_launching_entry_point_reports_the_injected_fault():
    env = dict(os.environ, SFA_TEST_FAULT="launch", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    from fibonacci_spaced_sparse_gb300 import _lib
    cuda, ok, bad = _lib.SFA_ERR_CUDA, _lib.SFA_OK, _lib.SFA_ERR_INVALID_ARG
    for name in ("forward", "forward_f32", "forward_layers", "backward", "backward_empty", "decode",
                 "qkv_rope", "rope_table", "selftest", "read_status"):
        assert got[name] == cuda, (name, got[name])
    # argument checks still come first, and calls with nothing to launch succeed
    assert got["forward_bad_arg"] == bad
    assert got["forward_empty"] == ok
    assert got["rope_table_empty"] == ok


def test_hook_is_off_without_the_variable():
    """Without the variable the same argument errors are reported (and nothing
    here reaches a launch)."""
    env = {k: v for k, v in os.environ.items() if k != "SFA_TEST_FAULT"}
    env["PYTHONPATH"] = ROOT
    code = ("import ctypes; from fibonacci_spaced_sparse_gb300 import _lib, api; lib = _lib.load(); "
            "p = api.Params(2, 64, W=12, alpha=1.1); f = ctypes.c_void_p(0x100000); n = ctypes.c_void_p(0); "
            "print(lib.sfa_forward(p.ref(), n, f, f, f, f, f, f, 1 << 40, n, n))")
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    from fibonacci_spaced_sparse_gb300 import _lib
    assert int(r.stdout.strip().splitlines()[-1]) == _lib.SFA_ERR_INVALID_ARG
