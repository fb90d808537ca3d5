"""The usage example of the design notes runs as written (bf16 forward,
backward, a schedule, the autograd wrapper) and gives finite results of the
documented shapes."""
import pytest
import torch

from fibonacci_spaced_sparse_gb300 import api

pytestmark = pytest.mark.gpu


def test_documented_usage_runs():
    torch.manual_seed(0)
    q = torch.randn(2, 256, 8, 64, device="cuda").bfloat16()
    k = torch.randn(2, 256, 2, 64, device="cuda").bfloat16()
    v = torch.randn(2, 256, 2, 64, device="cuda").bfloat16()
    o, lse = api.sfa_forward(q, k, v, alpha=0.9, W=12)
    dq, dk, dv, dalpha, dtheta = api.sfa_backward(q, k, v, o, torch.randn_like(o), lse,
                                                  alpha=0.9, W=12)
    alphas = api.alpha_schedule("linear", 16)
    assert len(alphas) == 16 and abs(alphas[0] - 0.5) < 1e-6 and abs(alphas[-1] - 1.5) < 1e-6
    theta = torch.zeros((), device="cuda", requires_grad=True)
    qg, kg, vg = (t.clone().requires_grad_(True) for t in (q, k, v))
    o2 = api.SparseAttention.apply(qg, kg, vg, theta, 12)
    o2.float().square().mean().backward()
    torch.cuda.synchronize()
    assert o.shape == (2, 256, 8, 64) and lse.shape == (2, 256, 8)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    for t in (o, lse, dq, dk, dv, o2, qg.grad, kg.grad, vg.grad):
        assert torch.isfinite(t.float()).all()
    assert torch.isfinite(theta.grad) and theta.grad.item() != 0.0
    # alpha = 1 at theta = 0: the wrapper's forward is sfa_forward at alpha = 1
    o1, _ = api.sfa_forward(q, k, v, alpha=1.0, W=12)
    assert torch.equal(o2.detach(), o1)
