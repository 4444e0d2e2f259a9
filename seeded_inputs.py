"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module only draws random numbers and names shapes.  It holds none of the
method's arithmetic (no scales, no rounding, no packing), so the oracle and the
CUDA path can both be fed from it without sharing any step of the computation.

Recipes (the ternary-weight pages publish no data set; these stand in):
  * weights: W ~ N(0, 1) fp32, shape [N][K] (out x in, like nn.Linear.weight);
  * activations: x ~ N(0, 1) fp32, shape [M][K], drawn after W from the same
    torch CPU generator seeded with ``seed``;
  * outliers: each activation element independently, with probability 0.01,
    is multiplied by 20 (Bernoulli draws from the same generator);
  * RMSNorm gain: g = 1 + 0.1 * N(0, 1) per channel, eps = 1e-6;
  * large tensors are drawn on the GPU with a seeded torch CUDA generator, one
    tensor at a time (seed = base + 1000 * layer + index of the matrix).
"""
from __future__ import annotations

import numpy as np
import torch

RMS_EPS = 1e-6

# Decoder-layer matrix shapes (N = out features, K = in features).
# 2B: hidden 2560, ffn 6912, 20 heads / 5 KV heads, head_dim 128.
# 8B: hidden 4096, ffn 14336, 32 / 8 heads.  70B: hidden 8192, ffn 28672, 64 / 8 heads.
MODELS = {
    "2B": dict(hidden=2560, ffn=6912, heads=20, kv_heads=5, head_dim=128),
    "8B": dict(hidden=4096, ffn=14336, heads=32, kv_heads=8, head_dim=128),
    "70B": dict(hidden=8192, ffn=28672, heads=64, kv_heads=8, head_dim=128),
}


def layer_shapes(model: str) -> dict:
    """Per-layer GEMV shapes {name: (N, K)} of a decoder layer."""
    c = MODELS[model]
    h, f, kv = c["hidden"], c["ffn"], c["kv_heads"] * c["head_dim"]
    q = c["heads"] * c["head_dim"]
    return {"q": (q, h), "k": (kv, h), "v": (kv, h), "o": (h, q),
            "gate": (f, h), "up": (f, h), "down": (h, f)}


def fused_layer_shapes(model: str) -> dict:
    """The same layer with q|k|v and gate|up concatenated along N (one launch each)."""
    s = layer_shapes(model)
    h = s["q"][1]
    return {"qkv": (s["q"][0] + s["k"][0] + s["v"][0], h), "o": s["o"],
            "gateup": (s["gate"][0] + s["up"][0], h), "down": s["down"]}


def cpu_generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def weights(N: int, K: int, seed: int = 0, gen: torch.Generator | None = None) -> np.ndarray:
    g = gen if gen is not None else cpu_generator(seed)
    return torch.randn(N, K, generator=g, dtype=torch.float32).numpy()


def activations(M: int, K: int, seed: int = 0, gen: torch.Generator | None = None,
                outliers: bool = False) -> np.ndarray:
    g = gen if gen is not None else cpu_generator(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    if outliers:
        mask = torch.rand(M, K, generator=g, dtype=torch.float32) < 0.01
        x = torch.where(mask, x * 20.0, x)
    return x.numpy()


def gemv_case(M: int, N: int, K: int, seed: int = 0, outliers: bool = False):
    """W [N][K] first, then x [M][K], from one CPU generator (the small-config recipe)."""
    g = cpu_generator(seed)
    W = weights(N, K, gen=g)
    x = activations(M, K, gen=g, outliers=outliers)
    return W, x


def rms_gain(K: int, seed: int = 0) -> np.ndarray:
    g = cpu_generator(seed + 7777)
    return (1.0 + 0.1 * torch.randn(K, generator=g, dtype=torch.float32)).numpy()


def device_normal(shape, seed: int, device="cuda") -> torch.Tensor:
    """N(0,1) fp32 drawn on the GPU by torch's seeded CUDA generator."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def device_outliers(shape, seed: int, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    mask = torch.rand(*shape, generator=g, device=device, dtype=torch.float32) < 0.01
    return torch.where(mask, x * 20.0, x)
