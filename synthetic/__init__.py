"""Seeded synthetic inputs for the KV-cache decode-attention workloads.

This module is the only code the CPU oracle and the CUDA library's callers
share: it draws random numbers and shapes them, and holds none of the
method's arithmetic (no quantisation, no softmax, no ring logic).

Recipes (the shapes and distributions of the workloads the pages describe;
the pages' own model/eval data are not available, so these stand in):

* K, V, q ~ N(0, 1) f32 (the R-SWA and tiny GQA cases);
* "outlier channels": per (sequence, KV head, channel) a standard deviation
  sigma = exp(U[ln 0.1, ln 10]) (log-uniform in [0.1, 10], the RoPE-band-like
  channel structure the per-32-channel K scales are meant for); K, V =
  sigma * N(0, 1);
* ragged lengths L_b ~ U{1 .. 16384};
* dead GQA groups: 2 of 8 KV heads per layer, drawn without replacement.

NumPy draws (PCG64) serve the sizes the oracle handles; torch draws on the
target device serve the full-size benchmark caches (generated in HBM, then
sampled back to the host where a test needs oracle values for them).
"""

from __future__ import annotations

import numpy as np

SIGMA_LO, SIGMA_HI = 0.1, 10.0


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal(shape, seed: int) -> np.ndarray:
    """f32 N(0,1) of the given shape."""
    return rng(seed).standard_normal(shape, dtype=np.float32)


def channel_sigma(shape, seed: int) -> np.ndarray:
    """f32 log-uniform standard deviations in [0.1, 10] of the given shape."""
    u = rng(seed).uniform(np.log(SIGMA_LO), np.log(SIGMA_HI), size=shape)
    return np.exp(u).astype(np.float32)


def outlier_rows(n_rows: int, n_kv: int, hd: int, sigma: np.ndarray, seed: int) -> np.ndarray:
    """[n_rows, n_kv, hd] f32 rows with per-(head, channel) std sigma [n_kv, hd]."""
    z = normal((n_rows, n_kv, hd), seed)
    return (z * sigma[None, :, :]).astype(np.float32)


def ragged_lengths(n_seq: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """int64 lengths uniform in [lo, hi]."""
    return rng(seed).integers(lo, hi + 1, size=n_seq, dtype=np.int64)


def dead_mask(n_kv: int, n_dead: int, seed: int) -> np.ndarray:
    """uint8 alive mask [n_kv] with n_dead heads set to 0."""
    alive = np.ones(n_kv, np.uint8)
    alive[rng(seed).choice(n_kv, size=n_dead, replace=False)] = 0
    return alive


# ---- device-side draws for full-size caches ------------------------------

def torch_normal(shape, seed: int, device, generator=None):
    """f32 N(0,1) drawn with torch's generator on `device` (seeded)."""
    import torch

    g = generator if generator is not None else torch.Generator(device=device).manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def torch_channel_sigma(shape, seed: int, device):
    import torch

    g = torch.Generator(device=device).manual_seed(seed)
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float64)
    lo, hi = np.log(SIGMA_LO), np.log(SIGMA_HI)
    return torch.exp(lo + (hi - lo) * u).to(torch.float32)
