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


# ---- the benchmark workloads' per-sequence recipes -----------------------
# (seeds and shapes only; the library's workload builders and the oracle's
# CPU baseline both draw a workload's rows from these, on the device or on
# the host: torch's CPU and CUDA generators give different draws of the same
# distribution)

SEED_OFFSETS = {"k": 101, "v": 202, "sk": 303, "sv": 404, "q": 505}


def gqa_seq_rows(seed: int, b: int, L: int, n_kv: int, hd: int, outliers: bool, device="cuda"):
    """(K, V) rows [L, n_kv, hd] f32 of sequence b of a GQA workload: N(0,1),
    times the per-(head, channel) log-uniform sigma with outlier channels."""
    base = seed * 1_000_003 + b * 9973
    k = torch_normal((L, n_kv, hd), base + SEED_OFFSETS["k"], device)
    v = torch_normal((L, n_kv, hd), base + SEED_OFFSETS["v"], device)
    if outliers:
        k *= torch_channel_sigma((n_kv, hd), base + SEED_OFFSETS["sk"], device)
        v *= torch_channel_sigma((n_kv, hd), base + SEED_OFFSETS["sv"], device)
    return k, v


def gqa_query(seed: int, step: int, n_seq: int, n_q: int, hd: int, device="cuda"):
    """The queries [n_seq, n_q, hd] of decode step `step` of a GQA workload."""
    return torch_normal((n_seq, n_q, hd), seed * 7919 + SEED_OFFSETS["q"] + step, device)


RAGGED_MODE_NAMES = ("f32", "q8", "q8k", "q8v")


def ragged_batch(n_seq: int = 256):
    """The ragged serving batch: 256 lengths U{1..16384} (seed 7; n_seq < 256
    keeps the first n_seq), 32 query / 8 KV heads, head_dim 128, and one layer
    per storage mode (f32, q8, q8k, q8v) with 2 of its 8 KV heads dead and its
    own row seed.  Returns (lengths, [(mode name, alive mask, row seed)])."""
    lengths = ragged_lengths(256, 1, 16384, 7)[:n_seq]
    layers = [(name, dead_mask(8, 2, 7 * 100 + li), 70 + li) for li, name in enumerate(RAGGED_MODE_NAMES)]
    return lengths, layers


# The fixed-length GQA workloads: storage mode, sequences, query / KV heads,
# head_dim, rows per sequence, row seed, outlier channels, and whether the
# benchmark builds the cache one row at a time (else in bulk appends).
GQA_WORKLOADS = {
    "tiny_f32": dict(mode="f32", n_seq=1, n_q=4, n_kv=2, hd=64, rows=256, seed=0, outliers=False,
                     stepwise=False),
    "q8_gqa": dict(mode="q8", n_seq=32, n_q=32, n_kv=8, hd=128, rows=4096, seed=2, outliers=True,
                   stepwise=True),
    "long_q8": dict(mode="q8", n_seq=4, n_q=64, n_kv=4, hd=128, rows=131072, seed=4, outliers=True,
                    stepwise=False),
}
