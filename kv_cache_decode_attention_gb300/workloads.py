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
        return synthetic.gqa_query(self.seed, step, self.n_seq, self.n_q, self.hd, device)

    def new_rows(self, step: int, device="cuda"):
        """One appended row per sequence for decode step `step`: [n_seq, n_kv, hd]."""
        g = torch.Generator(device=device).manual_seed(self.seed * 104729 + step)
        k = torch.randn(self.n_seq, self.n_kv, self.hd, generator=g, device=device)
        v = torch.randn(self.n_seq, self.n_kv, self.hd, generator=g, device=device)
        return k, v


def seq_rows(seed: int, b: int, L: int, n_kv: int, hd: int, outliers: bool, device="cuda"):
    return synthetic.gqa_seq_rows(seed, b, L, n_kv, hd, outliers, device)


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


def _fixed(name, device, extra_cap):
    w = synthetic.GQA_WORKLOADS[name]
    return _build_gqa(name, api.MODE_NAMES[w["mode"]], w["n_seq"], w["n_q"], w["n_kv"], w["hd"],
                      [w["rows"]] * w["n_seq"], np.ones(w["n_kv"], np.uint8), w["seed"],
                      outliers=w["outliers"], stepwise=w["stepwise"], extra_cap=extra_cap, device=device)


def tiny_f32(device="cuda", extra_cap=64):
    return _fixed("tiny_f32", device, extra_cap)


def q8_gqa(device="cuda", extra_cap=512):
    return _fixed("q8_gqa", device, extra_cap)


def long_q8(device="cuda", extra_cap=512):
    return _fixed("long_q8", device, extra_cap)


RAGGED_MODES = (api.F32, api.Q8, api.Q8K, api.Q8V)


def ragged(device="cuda", extra_cap=64, modes=RAGGED_MODES, n_seq=256):
    """The ragged serving batch: one layer per storage mode over the same 256
    sequence lengths (n_seq < 256 keeps the first n_seq of them, a smaller
    batch of the same length mix)."""
    lengths, specs = synthetic.ragged_batch(n_seq)
    out = []
    for mode in modes:
        name, alive, seed = specs[mode]
        out.append(_build_gqa("ragged_%s" % name, mode, n_seq, 32, 8, 128,
                              lengths, alive, seed, outliers=True, stepwise=False,
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
