"""Seeded synthetic decode workloads, built in HBM through the library's own calls.

Each builder draws its inputs with torch's seeded generator on the device
(the recipes of ``synthetic``), builds the cache with ``kv_append`` /
``rswa_record_prefill`` / ``rswa_ring_write``, and keeps what a checker needs
to regenerate any sequence's rows on the host.

Workloads (shapes of the pages' use: cortiq decode over a q8_2f cache,
franken_ocr R-SWA decode):
  tiny_f32      1 seq, 4 Q / 2 KV heads, hd 64, 256 rows, f32, N(0,1), seed 0
  q8_gqa        32 seqs x 4096 rows, 32 Q / 8 KV heads, hd 128, q8_2f, outlier
                channels, built one row at a time (freeze at 64), seed 2
  rswa_steady   16 streams, 10 heads, hd 128, prefix 32640 rows N(0,1), ring
                W = 128 after 500 decode steps, seed 3
  long_q8       4 seqs x 131072 rows, 64 Q / 4 KV heads, hd 128, q8_2f, outlier
                channels, bulk-appended, seed 4
  ragged        256 seqs, L ~ U{1..16384}, 32 Q / 8 KV heads, hd 128, four
                layers (f32, q8, q8k, q8v), 2 of 8 KV heads dead per layer,
                outlier channels, seed 7
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

import synthetic

from . import api

SEED_OFFSETS = {"k": 101, "v": 202, "sk": 303, "sv": 404, "q": 505}


@dataclass
class GqaWorkload:
    name: str
    mode: int
    n_seq: int
    n_q: int
    n_kv: int
    hd: int
    lengths: np.ndarray
    alive: np.ndarray
    seed: int
    layer: api.LayerKvCache
    scale: float
    outliers: bool
    extra: dict = field(default_factory=dict)

    @property
    def hpk(self) -> int:
        return self.n_q // self.n_kv

    def rows(self, b: int, device="cuda"):
        """(K, V) rows [L_b, n_kv, hd] f32 of sequence b, regenerated exactly."""
        return seq_rows(self.seed, b, int(self.lengths[b]), self.n_kv, self.hd, self.outliers, device)

    def query(self, step: int, device="cuda"):
        return synthetic.torch_normal((self.n_seq, self.n_q, self.hd),
                                      self.seed * 7919 + SEED_OFFSETS["q"] + step, device)

    def new_rows(self, step: int, device="cuda"):
        """One appended row per sequence for decode step `step`: [n_seq, n_kv, hd]."""
        g = torch.Generator(device=device).manual_seed(self.seed * 104729 + step)
        k = torch.randn(self.n_seq, self.n_kv, self.hd, generator=g, device=device)
        v = torch.randn(self.n_seq, self.n_kv, self.hd, generator=g, device=device)
        return k, v


def seq_rows(seed: int, b: int, L: int, n_kv: int, hd: int, outliers: bool, device="cuda"):
    base = seed * 1_000_003 + b * 9973
    k = synthetic.torch_normal((L, n_kv, hd), base + SEED_OFFSETS["k"], device)
    v = synthetic.torch_normal((L, n_kv, hd), base + SEED_OFFSETS["v"], device)
    if outliers:
        k *= synthetic.torch_channel_sigma((n_kv, hd), base + SEED_OFFSETS["sk"], device)
        v *= synthetic.torch_channel_sigma((n_kv, hd), base + SEED_OFFSETS["sv"], device)
    return k, v


def _build_gqa(name, mode, n_seq, n_q, n_kv, hd, lengths, alive, seed, outliers, stepwise,
               extra_cap=0, device="cuda", batch_rows=1 << 22):
    lengths = np.asarray(lengths, np.int64)
    layer = api.LayerKvCache(n_seq, n_kv, hd, mode, lengths + extra_cap, alive=alive, device=device)
    wl = GqaWorkload(name, mode, n_seq, n_q, n_kv, hd, lengths, np.asarray(alive, np.uint8), seed,
                     layer, 1.0 / math.sqrt(hd), outliers)
    if stepwise:
        # every sequence has the same length here: one call per row position
        L = int(lengths.max())
        rows = [seq_rows(seed, b, int(lengths[b]), n_kv, hd, outliers, device) for b in range(n_seq)]
        K = torch.stack([r[0] for r in rows], 1).contiguous()  # [L, n_seq, n_kv, hd]
        V = torch.stack([r[1] for r in rows], 1).contiguous()
        del rows
        for t in range(L):
            api.kv_append(layer, K[t], V[t])
        del K, V
    else:
        # bulk appends, a group of sequences at a time (bounded input memory)
        b0 = 0
        while b0 < n_seq:
            b1, acc = b0, 0
            while b1 < n_seq and (b1 == b0 or acc + lengths[b1] * n_kv * hd <= batch_rows * hd):
                acc += lengths[b1] * n_kv * hd
                b1 += 1
            nn = np.zeros(n_seq, np.int32)
            nn[b0:b1] = lengths[b0:b1]
            parts = [seq_rows(seed, b, int(lengths[b]), n_kv, hd, outliers, device) for b in range(b0, b1)]
            K = torch.cat([p[0] for p in parts]).contiguous()
            V = torch.cat([p[1] for p in parts]).contiguous()
            api.kv_append(layer, K, V, nn)
            del parts, K, V
            b0 = b1
    torch.cuda.synchronize()
    return wl


def tiny_f32(device="cuda"):
    return _build_gqa("tiny_f32", api.F32, 1, 4, 2, 64, [256], np.ones(2, np.uint8), 0,
                      outliers=False, stepwise=False, extra_cap=64, device=device)


def q8_gqa(device="cuda", extra_cap=512):
    return _build_gqa("q8_gqa", api.Q8, 32, 32, 8, 128, [4096] * 32, np.ones(8, np.uint8), 2,
                      outliers=True, stepwise=True, extra_cap=extra_cap, device=device)


def long_q8(device="cuda", extra_cap=512):
    return _build_gqa("long_q8", api.Q8, 4, 64, 4, 128, [131072] * 4, np.ones(4, np.uint8), 4,
                      outliers=True, stepwise=False, extra_cap=extra_cap, device=device)


RAGGED_MODES = (api.F32, api.Q8, api.Q8K, api.Q8V)


def ragged(device="cuda", extra_cap=64, modes=RAGGED_MODES):
    lengths = synthetic.ragged_lengths(256, 1, 16384, 7)
    out = []
    for li, mode in enumerate(modes):
        alive = synthetic.dead_mask(8, 2, 7 * 100 + li)
        out.append(_build_gqa("ragged_%s" % ["f32", "q8", "q8k", "q8v"][mode], mode, 256, 32, 8, 128,
                              lengths, alive, 70 + li, outliers=True, stepwise=False,
                              extra_cap=extra_cap, device=device))
    return out


@dataclass
class RswaWorkload:
    cache: api.RingCache
    seed: int
    prefill: int
    steps: int
    H: int = 10
    hd: int = 128

    def prefill_rows(self, s: int, device="cuda"):
        base = self.seed * 1_000_003 + s * 9973
        k = synthetic.torch_normal((self.H, self.prefill, self.hd), base + 1, device)
        v = synthetic.torch_normal((self.H, self.prefill, self.hd), base + 2, device)
        return k, v

    def step_rows(self, t: int, device="cuda"):
        g = torch.Generator(device=device).manual_seed(self.seed * 104729 + t)
        B = self.cache.B
        k = torch.randn(B, self.H, self.hd, generator=g, device=device)
        v = torch.randn(B, self.H, self.hd, generator=g, device=device)
        return k, v

    def query(self, t: int, device="cuda"):
        return synthetic.torch_normal((self.cache.B, self.H, self.hd), self.seed * 7919 + t, device)


def rswa_steady(device="cuda", B=16, prefill=32640, steps=500, seed=3, int8=False):
    cache = api.RingCache(B, prefill, 10, 128, 128, device=device, int8=int8)
    wl = RswaWorkload(cache, seed, prefill, steps)
    for s in range(B):
        k, v = wl.prefill_rows(s, device)
        api.rswa_record_prefill(cache, s, k, v)
        del k, v
    for t in range(steps):
        k, v = wl.step_rows(t, device)
        api.rswa_ring_write(cache, k, v)
    torch.cuda.synchronize()
    return wl


# ---------------------------------------------------------------- byte counts

def kv_bytes_per_row(mode: int, hd: int) -> int:
    """Stored bytes per cached row per live KV head (K and V with their scales)."""
    qk = mode in (api.Q8, api.Q8K)
    qv = mode in (api.Q8, api.Q8V)
    kb = hd + 4 * (hd // 32) if qk else 4 * hd
    vb = hd + 4 if qv else 4 * hd
    return kb + vb


def decode_bytes(mode, n_live, hd, n_q, lengths, with_imp, n_seq) -> int:
    """Algorithmic bytes of one decode call: every live row's K/V (+ scales) once,
    the query and output, the fields of the quantised components, and imp
    read + write when it is requested."""
    rows = int(np.sum(lengths)) * n_live
    b = rows * kv_bytes_per_row(mode, hd)
    b += 2 * n_seq * n_q * hd * 4
    nf = (1 if mode in (api.Q8, api.Q8K) else 0) + (1 if mode in (api.Q8, api.Q8V) else 0)
    b += nf * n_seq * n_live * hd * 4
    if with_imp:
        b += 8 * int(np.sum(lengths))
    return b


def append_bytes(mode, n_live, hd, n_seq) -> int:
    """Algorithmic bytes of appending one row per sequence: f32 K, V in for the
    live heads, stored codes/scales (or f32 rows) out, fields read."""
    b = n_seq * n_live * (8 * hd + kv_bytes_per_row(mode, hd))
    nf = (1 if mode in (api.Q8, api.Q8K) else 0) + (1 if mode in (api.Q8, api.Q8V) else 0)
    return b + nf * n_seq * n_live * hd * 4


def rswa_bytes(B, H, hd, lengths) -> int:
    return int(np.sum(lengths)) * H * hd * 8 + 2 * B * H * hd * 4


def rswa_i8_bytes(B, H, hd, lengths) -> int:
    """Algorithmic bytes of one int8-mirror decode: every row's K and V codes and
    their two row scales, plus the f32 query and output."""
    return int(np.sum(lengths)) * H * (2 * hd + 8) + 2 * B * H * hd * 4
