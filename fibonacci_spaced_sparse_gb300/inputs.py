"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module only draws random numbers: it holds none of the attention
arithmetic.  Every tensor is drawn on the CPU from a ``torch.Generator`` seeded
from (seed, layer, stream), as N(0, 1) in fp32 and then rounded to the
requested dtype, so the GPU path and the oracle can be fed the identical bytes.
Seed 42 is the training seed of the paper's recipe (section 3 "Model and
training" of arXiv 2606.28560); the shapes are the paper's attention shape
(8 query heads, 2 key/value heads, head dimension 64).
"""
from __future__ import annotations

import torch

_STREAMS = {"q": 0, "k": 1, "v": 2, "dO": 3, "theta": 4, "x": 5, "w": 6}


def _gen(seed: int, layer: int, stream: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((int(seed) * 1_000_003 + int(layer) * 7_919 + _STREAMS[stream]) % (2 ** 62))
    return g


def normal(shape, *, dtype=torch.bfloat16, seed: int = 42, layer: int = 0,
           stream: str = "q") -> torch.Tensor:
    """N(0, 1) draws of ``shape`` rounded to ``dtype`` (CPU tensor)."""
    x = torch.randn(tuple(shape), generator=_gen(seed, layer, stream), dtype=torch.float32)
    return x.to(dtype)


def normal_on(device, shape, *, dtype=torch.bfloat16, seed: int = 42, layer: int = 0,
              stream: str = "q", chunk: int = 1 << 26) -> torch.Tensor:
    """N(0, 1) draws of ``shape`` made on ``device`` by a generator of that
    device seeded as above, rounded to ``dtype``: for tensors too large to
    draw on the host.  Drawn ``chunk`` elements at a time (in order), so the
    fp32 intermediate stays small; the same arguments give the same tensor on
    the same device type and PyTorch version, and a test reads back the rows
    it hands to the oracle."""
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(layer) * 7_919 + _STREAMS[stream]) % (2 ** 62))
    out = torch.empty(tuple(shape), dtype=dtype, device=device)
    flat = out.view(-1)
    for c in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - c)
        flat[c:c + n] = torch.randn((n,), generator=g, device=device, dtype=torch.float32).to(dtype)
    return out


def qkv(B: int, T: int, Hq: int = 8, Hkv: int = 2, D: int = 64, *,
        dtype=torch.bfloat16, seed: int = 42, layer: int = 0, with_dO: bool = False):
    """Q [B,T,Hq,D], K and V [B,T,Hkv,D] (and dO [B,T,Hq,D]) as CPU tensors."""
    out = {
        "q": normal((B, T, Hq, D), dtype=dtype, seed=seed, layer=layer, stream="q"),
        "k": normal((B, T, Hkv, D), dtype=dtype, seed=seed, layer=layer, stream="k"),
        "v": normal((B, T, Hkv, D), dtype=dtype, seed=seed, layer=layer, stream="v"),
    }
    if with_dO:
        out["dO"] = normal((B, T, Hq, D), dtype=dtype, seed=seed, layer=layer, stream="dO")
    return out


def thetas(L: int, sigma: float, *, seed: int = 42) -> list:
    """Per-layer theta_l ~ N(0, sigma) (sigma is a standard deviation), fp64."""
    g = _gen(seed, 0, "theta")
    x = torch.randn((L,), generator=g, dtype=torch.float64) * float(sigma)
    return [float(t) for t in x]


def hidden_and_weight(B: int, T: int, d_model: int = 512, rows: int = 768, *,
                      dtype=torch.bfloat16, seed: int = 42, layer: int = 0):
    """Inputs of the QKV front end: hidden states X [B,T,d_model] ~ N(0, 1) and
    a projection weight [rows, d_model] ~ N(0, 1/d_model) (so that the
    projections are of unit scale), both rounded to ``dtype``."""
    x = normal((B, T, d_model), dtype=dtype, seed=seed, layer=layer, stream="x")
    g = _gen(seed, layer, "w")
    w = torch.randn((rows, d_model), generator=g, dtype=torch.float32) / float(d_model) ** 0.5
    return x, w.to(dtype)
