"""Seeded synthetic inputs shaped like the workloads the TurboQuant pages measure.

This module draws random data and nothing else: it holds none of the method's
arithmetic (no rotation, codebook, quantization or estimator), so both the CUDA
path and the CPU oracle may consume what it produces.  Every generator takes a
``device`` so that large inputs can be drawn directly in HBM; a test draws once
and copies the same bytes to both sides.

Generators:

* ``gaussian`` -- i.i.d. N(0, 1) rows (the tiny correctness case).
* ``anisotropic_factors`` / ``anisotropic`` -- a stand-in for real LLM key and
  value caches (Llama / Gemma / Mistral, whose weights are not available): for
  each KV head a rank-64 Gaussian factor W ~ N(0, 1/64)^{64 x d}, rows
  X = Z W + 0.1 E with Z, E standard normal, and 4 outlier channels (a random
  choice per head) multiplied by 10.  Keys and values use separate seeds; queries
  are drawn from the same per-head law as that head's keys.
* ``cone`` -- unit vectors concentrated around a random mean direction mu:
  x = normalise(mu + sigma * N(0, I)), sigma = 0.5 (a stand-in for GloVe d=200).
"""

from __future__ import annotations

import torch

RANK = 64
NOISE = 0.1
OUTLIERS = 4
OUTLIER_SCALE = 10.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(n: int, d: int, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(n, d, generator=g, device=device, dtype=torch.float32).to(dtype)


def anisotropic_factors(H: int, d: int, seed: int, device="cpu"):
    """Per-head factor W [H, 64, d] (fp32) and outlier channel indices [H, 4] (int64)."""
    g = _gen(seed, device)
    W = torch.randn(H, RANK, d, generator=g, device=device) / (RANK ** 0.5)
    out = torch.stack([torch.randperm(d, generator=g, device=device)[:OUTLIERS] for _ in range(H)])
    return W, out


def anisotropic(B: int, H: int, N: int, d: int, factors, seed: int, device="cpu",
                dtype=torch.bfloat16) -> torch.Tensor:
    """Rows [B, H, N, d] of the anisotropic law for each head h (cast with round-to-nearest-even)."""
    W, out = factors
    g = _gen(seed, device)
    X = torch.empty(B, H, N, d, device=device, dtype=dtype)
    for b in range(B):
        for h in range(H):
            Z = torch.randn(N, RANK, generator=g, device=device)
            E = torch.randn(N, d, generator=g, device=device)
            x = torch.addmm(NOISE * E, Z, W[h])
            x[:, out[h]] *= OUTLIER_SCALE
            X[b, h] = x.to(dtype)
    return X


def cone(n: int, d: int, seed: int, mu_seed: int, device="cpu", sigma: float = 0.5) -> torch.Tensor:
    """n unit vectors x = normalise(mu + sigma * N(0, I)); mu is a random unit vector from mu_seed."""
    gm = _gen(mu_seed, device)
    mu = torch.randn(d, generator=gm, device=device)
    mu = mu / mu.norm()
    g = _gen(seed, device)
    x = mu[None, :] + sigma * torch.randn(n, d, generator=g, device=device)
    return x / x.norm(dim=1, keepdim=True)
