"""The fused front end (sfa_qkv_rope): QKV projection on the tensor cores with
RoPE in the epilogue, against the fp64 oracle's projection and rotation of the
same bf16 inputs, element by element; then the pipeline front end ->
sfa_forward(rope_theta=0) against the oracle's attention."""
import numpy as np
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api, inputs
from oracle import oracle
from _helpers import TOL, max_abs, np64

pytestmark = pytest.mark.gpu


def _draw(B, T, dm, layer=0):
    x, w = inputs.hidden_and_weight(B, T, dm, layer=layer)
    return x, w, x.to(torch.float64).numpy(), w.to(torch.float64).numpy()


def _check(got, want):
    """bf16 outputs of an fp32-accumulated projection: within one bf16 step
    (2^-8 relative) of the fp64 value, plus 1e-3 for the accumulation order."""
    g = np64(got)
    err = np.abs(g - want) - (2.0 ** -8 * np.abs(want) + 1e-3)
    assert err.max() <= 0, float(np.max(np.abs(g - want)))


@pytest.mark.parametrize("B,T,dm", [(2, 300, 512), (1, 5, 64), (3, 97, 192), (1, 256, 1024), (2, 150, 320),
                                     (1, 40, 16384)])
@pytest.mark.parametrize("rope_theta", [1e4, 0.0])
def test_front_end_against_oracle(B, T, dm, rope_theta):
    x, w, xf, wf = _draw(B, T, dm, layer=B * 7 + dm)
    qh, kh, v = api.sfa_qkv_rope(x.cuda(), w.cuda(), rope_theta=rope_theta)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.qkv_rope(xf, wf, rope_theta=rope_theta)
    _check(qh, rq)
    _check(kh, rk)
    _check(v, rv)


def test_front_end_model_shape_sampled():
    """B = 32, T = 1024, d_model = 512 (the paper's model): rows sampled from
    every tile position, checked against the oracle row by row."""
    B, T, dm = 32, 1024, 512
    x, w, xf, wf = _draw(B, T, dm, layer=1)
    qh, kh, v = api.sfa_qkv_rope(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = sorted(set([(0, 0), (B - 1, T - 1), (5, 127), (5, 128)] +
                      [(int(rng.integers(B)), int(rng.integers(T))) for _ in range(60)]))
    for b, i in rows:
        # the oracle on the prefix of sequence b up to position i (true positions)
        rq, rk, rv = oracle.qkv_rope(xf[b:b + 1, :i + 1], wf)
        _check(qh[b, i], rq[0, i])
        _check(kh[b, i], rk[0, i])
        _check(v[b, i], rv[0, i])


def test_pipeline_front_end_then_attention():
    """x -> sfa_qkv_rope -> sfa_forward(rope_theta = 0) against the oracle
    attention (RoPE inside) on the oracle's projections of the same x and w.
    The tolerance adds to the bf16 bound of O the effect of the bf16 rounding
    of the projections on the GPU side: 3e-2."""
    B, T, dm = 2, 400, 512
    x, w, xf, wf = _draw(B, T, dm, layer=9)
    qh, kh, v = api.sfa_qkv_rope(x.cuda(), w.cuda())
    o, lse = api.sfa_forward(qh, kh, v, alpha=0.77, W=12, rope_theta=0.0)
    torch.cuda.synchronize()
    q, k, vv = oracle.qkv_rope(xf, wf, rope_theta=0.0)
    o_ref, lse_ref = oracle.forward(q, k, vv, W=12, rungs=api.FIBONACCI_BASE, alpha=0.77,
                                    rope_theta=1e4)
    assert max_abs(np64(o), o_ref) <= 3e-2
    assert max_abs(np64(lse), lse_ref) <= 3e-2
    # on the GPU's own bf16 projections, the attention meets the usual bound
    o2, l2 = oracle.forward(np64(qh), np64(kh), np64(v), W=12, rungs=api.FIBONACCI_BASE,
                            alpha=0.77, rope_theta=0.0)
    assert max_abs(np64(o), o2) <= TOL["bf16"]["o"]
    assert max_abs(np64(lse), l2) <= TOL["bf16"]["lse"]


def test_front_end_status_word_clean_and_empty_input():
    x, w, _, _ = _draw(1, 64, 128, layer=2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.sfa_qkv_rope(x.cuda(), w.cuda(), status=status)
    assert api.sfa_read_status(status) == 0
    e = torch.empty((2, 0, 128), dtype=torch.bfloat16, device="cuda")
    n0 = api.launch_count()
    qh, kh, v = api.sfa_qkv_rope(e, w.cuda())
    assert qh.shape == (2, 0, 8, 64) and kh.shape == (2, 0, 2, 64)
    assert api.launch_count() == n0
