"""The synthetic workloads the attention is measured and checked on.

Shapes follow the paper's model (section 3 "Model and training" of
"Depth-Staggered Fibonacci Spacing for Sparse Attention", arXiv 2606.28560):
8 query heads, 2 key/value heads, head dimension 64, training length 1024,
16 layers, windows W in {6, 8, 10, 12}; the length-extrapolation study runs at
4x the training length (section 4.5).  Every layer is an independent draw of
Q/K/V ~ N(0, 1) (fibonacci_spaced_sparse_gb300.inputs) with that layer's alpha.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import api


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    W: tuple            # window per layer group (one entry, or one per sweep point)
    schedule: str       # "fixed", "linear", "coprime" or "learned"
    base: str           # "fibonacci" or "pow2"
    layers: int
    dtype: str          # "f32" or "bf16"
    theta_sigma: float = 0.0   # std of theta_l for the learned schedule
    backward: bool = False

    def rungs(self):
        return api.FIBONACCI_BASE if self.base == "fibonacci" else api.pow2_base(self.T)

    def alphas(self, seed: int = 42):
        from . import inputs
        if self.schedule == "learned":
            th = inputs.thetas(self.layers, self.theta_sigma, seed=seed)
            return api.alpha_schedule("learned", self.layers, 7, th), th
        if self.schedule == "fixed" and self.layers == 1:
            return [1.0], None
        return api.alpha_schedule(self.schedule, self.layers, 7), None

    def window(self, layer: int) -> int:
        return self.W[layer % len(self.W)]

    @property
    def tokens(self) -> int:
        return self.B * self.T


TINY_F32 = Workload("tiny fp32 forward, alpha=1", 1, 256, (8,), "fixed", "fibonacci", 1, "f32")
MODEL_SHAPE = Workload("model-shape forward, linear stagger", 32, 1024, (12,), "linear",
                       "fibonacci", 16, "bf16")
EXTRAPOLATION = Workload("length-extrapolation forward, coprime stagger", 8, 4096, (12,),
                         "coprime", "fibonacci", 16, "bf16")
POW2 = Workload("power-of-two base forward, learned-style alpha", 32, 1024, (6, 8, 10, 12),
                "learned", "pow2", 16, "bf16", theta_sigma=0.3)
TRAIN_STEP = Workload("training step forward+backward", 32, 1024, (12,), "learned",
                      "fibonacci", 16, "bf16", theta_sigma=0.5, backward=True)
LONG_FORWARD = Workload("long forward", 2, 16384, (12,), "learned", "fibonacci", 16, "bf16",
                        theta_sigma=0.5)

DECODE = Workload("single-token decode over a 4096-row cache, linear stagger", 256, 4096, (12,),
                  "linear", "fibonacci", 16, "bf16")

ALL = (TINY_F32, MODEL_SHAPE, EXTRAPOLATION, POW2, TRAIN_STEP, LONG_FORWARD)
