#!/usr/bin/env python
"""Decode-attention benchmark on GB300: KV GB/s (fraction of the HBM roofline)
and decode queries/s.

Default workload: the ragged serving batch -- 256 sequences with lengths
U{1..16384} (seed 7), 32 query / 8 KV heads, head_dim 128, one layer per
storage mode (f32, q8_2f, q8k, q8v), 2 of 8 KV heads dead per layer, outlier
channels.  One step = the whole hot path for one decode token through the
four layers: kv_append of one new K/V row per sequence (quantised against
the frozen fields) + decode_attention over every cached row with the
attention-mass (imp) accumulation.  The timed region holds exactly --steps
steps between a barrier + device synchronisation on each side; --warmup
steps run untimed first.  The layers hold ~34 GB, far above L2.  The line
reports the step's KV GB/s, each mode's decode (without imp, timed alone)
against the HBM roofline, the same with imp, the end-to-end rate through the
public API with host buffers, and the CPU oracle on one and on all host cores.

Other workloads (--workload): q8_gqa (32 sequences x 4096 rows, the cache
built one row at a time, two or more cache replicas rotated so each step
streams HBM), long_q8 (4 sequences x 131072 rows, 64 query / 4 KV heads),
tiny_f32, verify_q8 (4 drafts verified per step), and the R-SWA decode of
franken_ocr's rswa module (16 streams x 10 heads, a 32640-row reference block
+ a full 128-slot ring): rswa reads the f32 regions, rswa_i8 the int8 mirror;
one step = the ring write of one token per stream (mirror included) + the
decode of every stream; rswa_verify / rswa_i8_verify verify 4 drafts.  The
q8_2f GQA lines also carry the decode against the tensor-core peak
(roofline_tensor), the second roof at 16 heads per group.

Under torchrun each rank times its own replica on its own GPU (independent
sequences: weak scaling, no data-path collective); rank 0 prints one JSON line
with the whole-job value.  `--impl reference` times the CPU oracle instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention KV GB/s (fraction of GB300 HBM peak) and queries/sec, 1 GPU"
# the q8_2f decode's contraction: int8 codes are exact in f16; the query and the
# softmax weights are each split into two f16 terms (hi + lo), so the products
# keep ~22 bits of the f32 operand; mma.sync m16n8k16, f32 accumulate
Q8_ARITHMETIC = ("int8 codes exact in f16, query and weights split into two f16 terms each, "
                 "mma.sync, f32 accumulate")
L2_BYTES = 129 * 1024 * 1024
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode call
# without imp -- the split kernel plus its merge -- from one ncu capture of
# this benchmark's own decode calls (the capture's command and figures are
# kept with the profiles), valid while the sources the call compiles from hash
# to the captured version, null otherwise.  The capture may run a smaller case
# of the same workload (fewer steps, or the first sequences of the ragged
# batch); a run reports it scaled by its algorithmic bytes over the capture's
# (both are rows x bytes per row plus a small fixed part).
CSRC_COMMON = ("kvd_internal.cuh", "kvd_decode.cu")
CSRC_CUDA_CORE = CSRC_COMMON + ("kvd_decode_kernels.cuh", "kvd_split_f32.cu", "kvd_split_q8k.cu",
                                "kvd_split_q8v.cu")
CSRC_TC = CSRC_COMMON + ("kvd_decode_kernels.cuh", "kvd_split_mma.cuh", "kvd_split_h16.cuh", "kvd_split_q8.cu")
TRAFFIC = {
    # q8_gqa (--steps 20 --warmup 5): the first two calls of the roofline loop
    "q8_gqa": {"files": CSRC_TC, "sources_sha256": "9af7d0aafcc69837b27d6875bd2f3de87a29105e02b53d479939617aa50d907e",
               "bytes": 300552576, "algorithmic_bytes": 291954176},
    # long_q8 (--steps 5 --warmup 3): the first two calls of the roofline loop
    "long_q8": {"files": CSRC_TC, "sources_sha256": "9af7d0aafcc69837b27d6875bd2f3de87a29105e02b53d479939617aa50d907e",
                "bytes": 609561088, "algorithmic_bytes": 579149888},
    # the first 16 sequences of the ragged batch, 3 + 3 steps in, mean of 10 calls
    "ragged_f32": {"files": CSRC_CUDA_CORE, "sources_sha256": "f4a882943a7a7c529c7b9734d27e061751fe904afe4ad531d73855d01ab93e16",
                   "bytes": 944721178, "algorithmic_bytes": 939376640},
    "ragged_q8": {"files": CSRC_TC, "sources_sha256": "9af7d0aafcc69837b27d6875bd2f3de87a29105e02b53d479939617aa50d907e",
                  "bytes": 259236506, "algorithmic_bytes": 253672640},
    "ragged_q8k": {"files": CSRC_CUDA_CORE, "sources_sha256": "f4a882943a7a7c529c7b9734d27e061751fe904afe4ad531d73855d01ab93e16",
                   "bytes": 606727347, "algorithmic_bytes": 602025728},
    "ragged_q8v": {"files": CSRC_CUDA_CORE, "sources_sha256": "f4a882943a7a7c529c7b9734d27e061751fe904afe4ad531d73855d01ab93e16",
                   "bytes": 595746355, "algorithmic_bytes": 591023552},
}


def kernel_sources_sha256(files=None) -> str:
    """sha256 over the named csrc files (every .cu / .cuh when None)."""
    import hashlib

    csrc = os.path.join(ROOT, "kv_cache_decode_attention_gb300", "csrc")
    names = sorted(files) if files else sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh")))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(workload: str, bytes_per_launch=None):
    t = TRAFFIC.get(workload)
    if not t or t["bytes"] is None or t["sources_sha256"] != kernel_sources_sha256(t["files"]):
        return None
    if bytes_per_launch is None:
        return t["bytes"]
    return int(round(t["bytes"] * bytes_per_launch / t["algorithmic_bytes"]))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense 16-bit tensor peak in TFLOP/s (the measured bf16 burst figure; f16
    runs at the same rate), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured (bf16 burst; f16 at the same rate)"
    return 1900.0, "fallback"


def decode_flops(n_live, hd, hpk, lengths, n_seq) -> int:
    """The decode's algorithmic floating-point work: two contractions (q.K and
    P.V) of 2 flops per multiply-add, hpk heads x hd channels per cached row
    per live group."""
    return int(4 * hpk * hd * n_live * int(np.sum(np.asarray(lengths[:n_seq], dtype=np.int64))))


# ------------------------------------------------------------ byte counts
# The metric's algorithmic bytes: what a decode must move at least, whatever
# the kernel (scratch partials are implementation cost and not counted).

F32_MODE, Q8_MODE, Q8K_MODE, Q8V_MODE = 0, 1, 2, 3
MODE_NAMES = ("f32", "q8", "q8k", "q8v")


def kv_bytes_per_row(mode: int, hd: int) -> int:
    """Stored bytes per cached row per live KV head (K and V with their scales)."""
    qk = mode in (Q8_MODE, Q8K_MODE)
    qv = mode in (Q8_MODE, Q8V_MODE)
    kb = hd + 4 * (hd // 32) if qk else 4 * hd
    vb = hd + 4 if qv else 4 * hd
    return kb + vb


def n_fields(mode: int) -> int:
    return (1 if mode in (Q8_MODE, Q8K_MODE) else 0) + (1 if mode in (Q8_MODE, Q8V_MODE) else 0)


def decode_bytes(mode, n_live, hd, n_q, lengths, with_imp, n_seq) -> int:
    """One decode call: every live row's K/V (+ scales) once, the query and
    output, the fields of the quantised components, and imp read + write when
    it is requested."""
    rows = int(np.sum(lengths)) * n_live
    b = rows * kv_bytes_per_row(mode, hd)
    b += 2 * n_seq * n_q * hd * 4
    b += n_fields(mode) * n_seq * n_live * hd * 4
    if with_imp:
        b += 8 * int(np.sum(lengths))
    return b


def append_bytes(mode, n_live, hd, n_seq) -> int:
    """Appending one row per sequence: f32 K, V in for the live heads, stored
    codes/scales (or f32 rows) out, fields read."""
    b = n_seq * n_live * (8 * hd + kv_bytes_per_row(mode, hd))
    return b + n_fields(mode) * n_seq * n_live * hd * 4


def rswa_bytes(B, H, hd, lengths) -> int:
    return int(np.sum(lengths)) * H * hd * 8 + 2 * B * H * hd * 4


def rswa_i8_bytes(B, H, hd, lengths) -> int:
    """One int8-mirror decode: every row's K and V codes and their two row
    scales, plus the f32 query and output."""
    return int(np.sum(lengths)) * H * (2 * hd + 8) + 2 * B * H * hd * 4


def host_cpu() -> dict:
    """The host's core count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


class GqaOracleSample:
    """Sampled sequences of one GQA layer rebuilt in the CPU oracle from the
    workload's seeded recipe -- rows drawn on the host (the device's draws come
    from another generator: same distribution, other numbers) and appended one
    row at a time -- with one decode query per sequence.  run() decodes every
    sampled sequence (all query heads, every row, imp on) through the oracle's
    multi-sequence driver."""

    def __init__(self, mode, n_q, n_kv, hd, lengths, alive, seed, outliers, picks):
        import oracle
        import synthetic

        self.mode, self.n_q, self.picks = mode, n_q, list(picks)
        q_all = synthetic.gqa_query(seed, 0, len(lengths), n_q, hd, "cpu").numpy()
        self.caches, self.qs = [], []
        for b in self.picks:
            L = int(lengths[b])
            k, v = synthetic.gqa_seq_rows(seed, b, L, n_kv, hd, outliers, "cpu")
            oc = oracle.OracleSeqCache(mode, n_kv, hd, max(L, 1), alive=alive)
            oc.append_rows(k.numpy(), v.numpy())
            self.caches.append(oc)
            self.qs.append(q_all[b])
        self.scale = np.float32(1.0 / math.sqrt(hd))
        self.rows = [int(lengths[b]) for b in self.picks]
        self.bytes = decode_bytes(mode, int(np.sum(alive)), hd, n_q, self.rows, True, len(self.picks))

    def run(self, threads: int) -> int:
        import oracle

        imps = [np.zeros(c.cap) for c in self.caches]
        _, used = oracle.decode_many(self.caches, self.qs, self.n_q, self.scale, imps, threads)
        return used


def time_oracle(samples, threads: int, min_seconds: float = 0.0, reps: int | None = None):
    """Decode every sample (one call per sample per repetition) until
    min_seconds have passed or `reps` repetitions ran: (GB/s, seconds per
    repetition, threads used)."""
    nbytes = sum(s.bytes for s in samples)
    n, used, t0 = 0, 1, time.perf_counter()
    while True:
        for smp in samples:
            used = max(used, smp.run(threads))
        n += 1
        el = time.perf_counter() - t0
        if (reps is not None and n >= reps) or (reps is None and el >= min_seconds):
            break
    return nbytes / (el / n) / 1e9, el / n, used


def time_threaded(samples, threads: int, min_seconds: float):
    """Run every sample's decode() once per repetition, the samples shared among
    `threads` Python threads (each decode is one call into the C oracle, which
    releases the interpreter lock), until min_seconds have passed: (GB/s,
    seconds per repetition, threads)."""
    from concurrent.futures import ThreadPoolExecutor

    nbytes = sum(s.bytes for s in samples)
    n, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            list(ex.map(lambda smp: smp.decode(), samples))
            n += 1
            el = time.perf_counter() - t0
            if el >= min_seconds:
                break
    return nbytes / (el / n) / 1e9, el / n, min(threads, len(samples))


def cpu_baseline_gqa(single, multi, seconds: float, what_single: str, what_multi: str) -> dict:
    """The oracle on one host core (the `single` samples) and on every core
    (the `multi` samples, its (sequence, head) pairs shared among threads)."""
    v1, _, _ = time_oracle(single, 1, seconds / 2)
    vn, _, used = time_oracle(multi, 0, seconds / 2)
    info = host_cpu()
    return {"value": round(vn, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": "%s, %.1f s" % (what_multi, seconds / 2),
            "single_core": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                            "sample": "%s, %.1f s" % (what_single, seconds / 2)},
            "nproc": info["nproc"], "cpu_model": info["cpu_model"]}


def gqa_samples(name: str, n_multi: int):
    """(single-core samples, all-core samples, descriptions) of a fixed-length
    GQA workload: one sequence, and the first n_multi sequences."""
    import synthetic

    w = synthetic.GQA_WORKLOADS[name]
    mode = MODE_NAMES.index(w["mode"])
    lengths = [w["rows"]] * w["n_seq"]
    alive = np.ones(w["n_kv"], np.uint8)
    n_multi = min(n_multi, w["n_seq"])
    multi = GqaOracleSample(mode, w["n_q"], w["n_kv"], w["hd"], lengths, alive, w["seed"], w["outliers"],
                            range(n_multi))
    single = GqaOracleSample(mode, w["n_q"], w["n_kv"], w["hd"], lengths, alive, w["seed"], w["outliers"],
                             [0])
    what = "%%d of %d sequences (all %d query heads x %d rows, imp on), f64" % (w["n_seq"], w["n_q"], w["rows"])
    return [single], [multi], what % 1, what % n_multi


def ragged_samples(n_multi: int, n_seq: int = 256):
    """(single-core samples, all-core samples, descriptions) of the ragged
    batch: per layer (f32, q8, q8k, q8v) the sequence nearest the mean length,
    and n_multi sequences spaced evenly through the batch."""
    import synthetic

    lengths, specs = synthetic.ragged_batch(n_seq)
    step = max(1, len(lengths) // n_multi)
    picks = list(range(0, len(lengths), step))[:n_multi]
    one = int(np.argmin(np.abs(lengths - lengths.mean())))
    single, multi = [], []
    for mode, (_, alive, seed) in enumerate(specs):
        multi.append(GqaOracleSample(mode, 32, 8, 128, lengths, alive, seed, True, picks))
        single.append(GqaOracleSample(mode, 32, 8, 128, lengths, alive, seed, True, [one]))
    rows = int(np.sum(lengths[picks]))
    return (single, multi,
            "1 sequence (%d rows) of each of the 4 layers, all 32 query heads, imp on, f64" % lengths[one],
            "%d of %d sequences (%d rows) of each of the 4 layers, all 32 query heads, imp on, f64"
            % (len(picks), len(lengths), rows))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period_ms = index, period_ms
        self.samples, self.proc, self.thread = [], None, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + CLOCK_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self):
        return time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not inside:  # a short timed region: take the samples nearest to it
            inside = [p for (t, p) in sorted(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[:3]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][2]), "samples": len(inside), "reasons": reasons}


# --------------------------------------------------------------- reference

class RswaOracleSample:
    """One stream of an R-SWA workload rebuilt on the host from the workload's
    generators (its reference rows and the ring rows of its 500 writes), ready
    for the CPU oracle's decode (f32 regions, or their int8 mirror)."""

    @classmethod
    def many(cls, wl, int8: bool, streams, verify_k: int = 0):
        """Samples of several streams, their ring writes replayed together."""
        import oracle

        c = wl.cache
        rings = {s: (np.zeros((c.H, c.W, c.head_dim), np.float32), np.zeros((c.H, c.W, c.head_dim), np.float32),
                     np.zeros(2, np.int32)) for s in streams}
        for t in range(wl.steps):
            k, v = wl.step_rows(t)
            k, v = k.cpu().numpy(), v.cpu().numpy()
            for s, (rk, rv, cur) in rings.items():
                oracle.rswa_write(rk, rv, k[s], v[s], True, cur)
        return [cls(wl, int8, s, verify_k, rings[s]) for s in streams]

    def __init__(self, wl, int8: bool, s: int = 0, verify_k: int = 0, ring=None):
        import oracle

        c = wl.cache
        self.int8, self.H, self.hd, self.verify_k = int8, c.H, c.head_dim, verify_k
        pk, pv = wl.prefill_rows(s)
        self.ref_k, self.ref_v = pk.cpu().numpy(), pv.cpu().numpy()
        if ring is None:
            self.ring_k = np.zeros((c.H, c.W, c.head_dim), np.float32)
            self.ring_v = np.zeros_like(self.ring_k)
            cur = np.zeros(2, np.int32)
            for t in range(wl.steps):
                k, v = wl.step_rows(t)
                oracle.rswa_write(self.ring_k, self.ring_v, k[s].cpu().numpy(), v[s].cpu().numpy(), True, cur)
        else:
            self.ring_k, self.ring_v, cur = ring
        self.prefill, self.ring_len = wl.prefill, int(cur[0])
        self.cursors = cur
        self.q = wl.query(10_000)[s].cpu().numpy()
        if verify_k:
            import synthetic

            shp = (verify_k, c.H, c.head_dim)
            self.vq, self.vk, self.vv = (synthetic.normal(shp, 90_000 + i) for i in range(3))
        if int8:
            self.mir = [oracle.rswa_mirror(x) for x in (self.ref_k, self.ref_v, self.ring_k, self.ring_v)]
        self.rows = self.prefill + self.ring_len
        self.bytes = (rswa_i8_bytes if int8 else rswa_bytes)(1, c.H, c.head_dim, [self.rows])
        if verify_k:
            self.bytes += 2 * verify_k * c.H * c.head_dim * 4 + 2 * (verify_k - 1) * c.H * c.head_dim * 4

    def decode(self):
        import oracle

        scale = np.float32(1.0 / math.sqrt(self.hd))
        if self.verify_k:
            return oracle.rswa_verify(self.vq, self.vk, self.vv, self.ref_k, self.ref_v, self.prefill, self.ring_k,
                                      self.ring_v, self.cursors, scale, int8=self.int8)
        if self.int8:
            (rk, rks), (rv, rvs), (gk, gks), (gv, gvs) = self.mir
            return oracle.rswa_decode_i8(self.q, rk, rks, rv, rvs, self.prefill, gk, gks, gv, gvs,
                                         self.ring_len, scale)
        return oracle.rswa_decode(self.q, self.ref_k, self.ref_v, self.prefill, self.ring_k, self.ring_v,
                                  self.ring_len, scale)

    def gbs(self, min_seconds: float, max_reps: int | None = None):
        reps, t0 = 0, time.perf_counter()
        while True:
            self.decode()
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or (max_reps is not None and reps >= max_reps):
                break
        per = el / reps
        return self.bytes / per / 1e9, per

    def describe(self, wl):
        return "1 of %d streams (all %d heads, %d rows%s), %s, f64 softmax" % (
            wl.cache.B, self.H, self.rows, ", %d draft queries" % self.verify_k if self.verify_k else "",
            "int8 mirror" if self.int8 else "f32 regions")


class VerifyOracleSample:
    """Sequence 0 of q8_gqa rebuilt in the oracle from its seeded recipe on the
    host, with K draft rows appended; run() verifies the K draft queries
    (oracle decode_verify, causal among the drafts)."""

    def __init__(self, K: int, b: int = 0):
        import oracle
        import synthetic

        w = synthetic.GQA_WORKLOADS["q8_gqa"]
        self.K, self.n_q, self.picks = K, w["n_q"], [b]
        k, v = synthetic.gqa_seq_rows(w["seed"], b, w["rows"], w["n_kv"], w["hd"], True, "cpu")
        self.oc = oracle.OracleSeqCache(Q8_MODE, w["n_kv"], w["hd"], w["rows"] + K)
        self.oc.append_rows(k.numpy(), v.numpy())
        self.oc.append_rows(synthetic.normal((K, w["n_kv"], w["hd"]), 91_000),
                            synthetic.normal((K, w["n_kv"], w["hd"]), 91_001))
        self.q = synthetic.normal((K, w["n_q"], w["hd"]), 91_002)
        self.scale = np.float32(1.0 / math.sqrt(w["hd"]))
        self.bytes = decode_bytes(Q8_MODE, w["n_kv"], w["hd"], w["n_q"], [w["rows"] + K], False, 1)
        self.what = "1 of %d sequences (%d drafts x %d query heads x %d rows), f64" % (
            w["n_seq"], K, w["n_q"], w["rows"] + K)

    def decode(self):
        return self.oc.decode_verify(self.q, self.n_q, self.K, self.scale)

    def run(self, threads: int) -> int:
        self.decode()
        return 1


def run_reference(args, rank):
    """--impl reference: the CPU oracle as it stands, on the host cores, each
    step a bounded sample of the workload decoded through the oracle's
    multi-sequence driver on every core; rank 0 only.  The GQA workloads are
    rebuilt from their seeded recipes on the host (the library under test is
    neither loaded nor built); the R-SWA ones read their rows from the device
    workload."""
    if rank != 0:
        return
    if args.workload in ("ragged", "q8_gqa", "long_q8", "tiny_f32", "verify_q8"):
        if args.workload == "ragged":
            _, multi, _, what = ragged_samples(args.cpu_sample_seqs)
            name = "ragged"
        elif args.workload == "verify_q8":
            multi = [VerifyOracleSample(VERIFY_DRAFTS)]
            what, name = multi[0].what, "verify_q8_gqa"
        else:
            _, multi, _, what = gqa_samples(args.workload, args.cpu_sample_seqs)
            name = args.workload
        time_oracle(multi, 0, reps=max(1, args.warmup))
        gbs, per, used = time_oracle(multi, 0, reps=args.steps)
        sample = what
        queries = sum(len(m.picks) for m in multi)
    else:
        import torch

        from kv_cache_decode_attention_gb300 import workloads as W

        if not torch.cuda.is_available():
            print(json.dumps({"impl": "reference", "unavailable": "needs the GPU box to build the workload"}))
            return
        int8, verify = args.workload.startswith("rswa_i8"), args.workload.endswith("_verify")
        wl = W.rswa_steady(B=args.rswa_streams, int8=int8)
        smp = RswaOracleSample(wl, int8, verify_k=VERIFY_DRAFTS if verify else 0)
        smp.gbs(0.0, max_reps=max(1, args.warmup))
        gbs, per = smp.gbs(0.0, max_reps=args.steps)
        sample, name, used, queries = smp.describe(wl), args.workload + "_steady", 1, 1
    info = host_cpu()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": sample, "nproc": info["nproc"], "cpu_model": info["cpu_model"]},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "queries_per_s": round(queries / per, 4),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

RSWA_WORKLOADS = ("rswa", "rswa_i8", "rswa_verify", "rswa_i8_verify")
VERIFY_DRAFTS = 4  # draft tokens per speculative step in the verify workloads


def packed_inputs(torch, parts_per_step):
    """Each step's input tensors packed into one pinned host buffer, and one device
    staging buffer with views of the same shapes: one host-to-device copy per step."""
    shapes = [t.shape for t in parts_per_step[0]]
    sizes = [t.numel() for t in parts_per_step[0]]
    pinned = [torch.cat([t.reshape(-1).cpu() for t in parts]).pin_memory() for parts in parts_per_step]
    stage = torch.empty(sum(sizes), device=parts_per_step[0][0].device)
    views, o = [], 0
    for shp, n in zip(shapes, sizes):
        views.append(stage[o:o + n].view(shp))
        o += n
    return pinned, stage, views


def e2e_pipelined(torch, pinned, stages, steps, launch):
    """End-to-end steps through the public API with host buffers, pipelined: step j's
    inputs go host -> device on a copy stream into staging buffer j % 2 while step
    j - 1 computes, its kernels wait for that copy, its output goes device -> host on
    a second copy stream once they finish, and the host waits once, at the end.
    stages: two (buffer, views) pairs; launch(j, views) enqueues step j on the
    current stream and returns (output tensor, pinned host tensor to copy it to).
    Events keep a staging buffer from being refilled before the step reading it has
    run, and an output from being rewritten before its copy out has.  Returns the
    seconds from the first copy to the last result on the host."""
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    Event = torch.cuda.Event
    freed = [None, None]   # staging buffer b no longer read (its step's kernels done)
    copied = {}            # output tensor -> its last copy out
    torch.cuda.synchronize()
    a0 = time.perf_counter()
    for j in range(steps):
        buf, views = stages[j % 2]
        ev_in = Event()
        with torch.cuda.stream(cin):
            if freed[j % 2] is not None:
                cin.wait_event(freed[j % 2])
            buf.copy_(pinned[j % len(pinned)], non_blocking=True)
            ev_in.record(cin)
        comp.wait_event(ev_in)
        out, host = launch(j, views, lambda t: copied.get(t.data_ptr()))
        done = Event()
        done.record(comp)
        freed[j % 2] = done
        ev_out = Event()
        with torch.cuda.stream(cout):
            cout.wait_event(done)
            host.copy_(out, non_blocking=True)
            ev_out.record(cout)
        copied[out.data_ptr()] = ev_out
    torch.cuda.synchronize()
    return time.perf_counter() - a0


def restage(torch, stage, views):
    """A second device staging buffer with views of the same shapes."""
    buf = torch.empty_like(stage)
    out, o = [], 0
    for v in views:
        out.append(buf[o:o + v.numel()].view(v.shape))
        o += v.numel()
    return buf, out


def wait_copied(torch, ev):
    """Make the current stream wait for an output's last copy out (None: none yet)."""
    if ev is not None:
        torch.cuda.current_stream().wait_event(ev)


def run_gpu_rswa(args, rank, world):
    """The R-SWA workloads: 16 streams in steady state (reference 32640 rows +
    a full ring), one step = rswa ring write of one token per stream + decode
    of every stream (f32 regions or the int8 mirror)."""
    import torch

    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300 import replicas
    from kv_cache_decode_attention_gb300 import workloads as W

    int8 = args.workload.startswith("rswa_i8")
    verify = args.workload.endswith("_verify")
    K = VERIFY_DRAFTS
    dev = torch.device("cuda", replicas.rank_info().local_rank)
    torch.cuda.set_device(dev)
    wl = W.rswa_steady(B=args.rswa_streams, int8=int8)
    c = wl.cache
    if verify:
        # speculative step: verify K drafts per stream (read-only), then write the
        # accepted token; qs hold the drafts' queries, news their K / V rows
        def decode(q, cache, out=None):
            return kvd.rswa_verify(q, dks[cur_i[0] % 8], dvs[cur_i[0] % 8], cache, int8=int8, out=out)
    else:
        decode = kvd.rswa_decode_i8 if int8 else kvd.rswa_decode
    B, H, hd = c.B, c.H, c.head_dim
    lengths = c.prefill_len + c.ring_len  # steady state: constant over the steps
    dec_bytes = (rswa_i8_bytes if int8 else rswa_bytes)(B, H, hd, lengths)
    # ring write: read k, v; write the f32 rows (+ codes and scales with the mirror)
    wr_bytes = B * H * hd * 4 * 4 + (B * H * (2 * hd + 8) if int8 else 0)
    if verify:
        import synthetic

        qs = [synthetic.torch_normal((B, K, H, hd), 70_000 + i, dev) for i in range(8)]
        dks = [synthetic.torch_normal((B, K, H, hd), 71_000 + i, dev) for i in range(8)]
        dvs = [synthetic.torch_normal((B, K, H, hd), 72_000 + i, dev) for i in range(8)]
        out = torch.empty(B, K, H * hd, device=dev)
        # the drafts are read once per step; the verify writes K outputs per stream
        dec_bytes += 2 * B * K * H * hd * 4 + 2 * B * (K - 1) * H * hd * 4
    else:
        qs = [wl.query(i, dev) for i in range(8)]
        out = torch.empty(B, H * hd, device=dev)
    news = [wl.step_rows(wl.steps + i, dev) for i in range(8)]
    stream = torch.cuda.current_stream()
    cur_i = [0]

    def step(i, with_events=None):
        k, v = news[i % 8]
        cur_i[0] = i
        if not verify:
            kvd.rswa_ring_write(c, k, v)
        if with_events is not None:
            with_events[0].record(stream)
        decode(qs[i % 8], c, out=out)
        if with_events is not None:
            with_events[1].record(stream)
        if verify:
            kvd.rswa_ring_write(c, k, v)  # the accepted token

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    with sampler:
        time.sleep(0.3)
        replicas.barrier()
        torch.cuda.synchronize()
        c0 = time.time()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.profiler.start()
        t0.record(stream)
        for j in range(args.steps):
            step(args.warmup + j)
        t1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        replicas.barrier()
        c1 = time.time()
        time.sleep(0.1)
    elapsed_ms = replicas.max_over_ranks(t0.elapsed_time(t1))
    ms_per_step = elapsed_ms / args.steps
    gbs = replicas.whole_job_rate((dec_bytes + wr_bytes) * args.steps, elapsed_ms * 1e-3, world) / 1e9
    # the decode's share of a step: the same steps again with events around it
    # (kept out of the timed steps above)
    for j in range(len(ev)):
        step(args.warmup + args.steps + j, ev[j])
    torch.cuda.synchronize()
    dec_ms = [a.elapsed_time(b) for a, b in ev]

    nrep = max(20, args.steps)
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nrep)]
    torch.cuda.profiler.start()
    for j in range(nrep):
        cur_i[0] = j
        dev_ev[j][0].record(stream)
        decode(qs[j % 8], c, out=out)
        dev_ev[j][1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    k_ms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
    peak, peak_kind = peaks()
    achieved = dec_bytes / (k_ms * 1e-3) / 1e9

    # end to end: pipelined (the headline), then synchronising on every step
    pinned, stage, (dq, dk, dv) = packed_inputs(torch, [(qs[i], news[i][0], news[i][1]) for i in range(8)])
    stages = [(stage, (dq, dk, dv)), restage(torch, stage, (dq, dk, dv))]
    pin_outs = [torch.empty(out.shape).pin_memory() for _ in range(2)]

    def e2e_step(j, views, last_copy):
        wait_copied(torch, last_copy(out))
        cur_i[0] = j
        if not verify:
            kvd.rswa_ring_write(c, views[1], views[2])
        decode(views[0], c, out=out)
        if verify:
            kvd.rswa_ring_write(c, views[1], views[2])
        return out, pin_outs[j % 2]

    secs = e2e_pipelined(torch, pinned, stages, args.steps, e2e_step)
    e2e = {"value": round((dec_bytes + wr_bytes) * args.steps / secs / 1e9 * world, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int((dq.numel() + dk.numel() + dv.numel()) * 4),
           "d2h_bytes_per_step": int(pin_outs[0].numel() * 4),
           "mode": "pipelined: inputs copied in on a copy stream while the previous step computes, "
                   "outputs copied out on another, one host synchronisation at the end"}
    torch.cuda.synchronize()
    a0 = time.perf_counter()
    for j in range(args.steps):
        stage.copy_(pinned[j % 8], non_blocking=True)
        cur_i[0] = j
        if not verify:
            kvd.rswa_ring_write(c, dk, dv)
        decode(dq, c, out=out)
        if verify:
            kvd.rswa_ring_write(c, dk, dv)
        pin_outs[0].copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    a1 = time.perf_counter()
    e2e_sync = {"value": round((dec_bytes + wr_bytes) * args.steps / (a1 - a0) / 1e9 * world, 2),
                "unit": "GB/s", "mode": "the host waits for every step's result before the next step"}
    if c.device_error():
        raise SystemExit("device error word set")
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        info = host_cpu()
        n_par = max(1, min(B, info["nproc"] or 1, args.cpu_sample_seqs))
        smps = RswaOracleSample.many(wl, int8, list(range(n_par)), verify_k=K if verify else 0)
        v1, _ = smps[0].gbs(args.cpu_seconds / 2)
        vn, _, used = time_threaded(smps, n_par, args.cpu_seconds / 2)
        cpu = {"value": round(vn, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": "%d streams at once, one per thread: %s, %.1f s" % (
                   n_par, smps[0].describe(wl), args.cpu_seconds / 2),
               "single_core": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                               "sample": smps[0].describe(wl) + ", %.1f s" % (args.cpu_seconds / 2)},
               "nproc": info["nproc"], "cpu_model": info["cpu_model"]}
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8" if int8 else "f32", "data": "synthetic",
        "config": {"workload": args.workload + "_steady", "streams": B, "heads": H, "head_dim": hd,
                   "reference_rows": int(wl.prefill), "ring_rows": int(c.W),
                   "step": ("rswa verify of %d drafts/stream (read-only) + ring write of the accepted token" % K
                            if verify else "rswa ring write 1 token/stream + decode of every stream"),
                   "arithmetic": ("int8 query and K codes exact in f16, mma.sync, f32 accumulate, per-row "
                                  "K scales applied to the scores (reference block); f32 CUDA-core dots "
                                  "elsewhere" if int8 and verify else
                                  "int8 codes widened to f32, CUDA-core dots" if int8 else
                                  "f32 CUDA-core dots"),
                   "l2": "inputs larger than L2 (%.2f GB read per decode)" % (dec_bytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "single"},
        "fraction_of_peak": round(gbs / world / peak, 4),
        "queries_per_s": round(B * world / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm",
                     "kernel": ("rswa verify (stream tables + tensor-core split + tail fused with the run merge)"
                                if int8
                                else "rswa verify (split + tail + merge)") if verify
                     else "rswa decode (split + merge)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": measured_traffic(args.workload),
                     "peak_kind": peak_kind, "ms_per_launch": round(k_ms, 5),
                     "bytes_per_launch": int(dec_bytes)},
        "decode_ms_in_step": round(statistics.mean(dec_ms), 5),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_sync": e2e_sync,
        "gpu_launches": args.steps * (4 if verify else 3),
        "clocks": sampler.summary(c0, c1),
    }
    if verify:
        line["queries_per_s"] = round(B * K * world / (ms_per_step * 1e-3), 1)
    print(json.dumps(line), flush=True)


def run_gpu_verify(args, rank, world):
    """q8_gqa speculative step: append VERIFY_DRAFTS draft rows per sequence, verify
    them in one query-batched call (causal among the drafts), reject them all
    (kv_truncate_last) so the cache length stays steady."""
    import torch

    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300 import replicas
    from kv_cache_decode_attention_gb300 import workloads as W
    import synthetic

    K = VERIFY_DRAFTS
    dev = torch.device("cuda", replicas.rank_info().local_rank)
    torch.cuda.set_device(dev)
    probe = W.q8_gqa(extra_cap=64)
    n_live = int(probe.alive.sum())
    bytes_each = decode_bytes(probe.mode, n_live, probe.hd, probe.n_q, probe.lengths + K, False, probe.n_seq)
    R = max(1, min(8, math.ceil(4 * L2_BYTES / bytes_each)))
    wls = [probe] + [W.q8_gqa(extra_cap=64) for _ in range(R - 1)]
    n_seq, n_q, n_kv, hd = probe.n_seq, probe.n_q, probe.n_kv, probe.hd
    qs = [synthetic.torch_normal((n_seq, K, n_q, hd), 80_000 + i, dev) for i in range(8)]
    drafts = [(synthetic.torch_normal((n_seq * K, n_kv, hd), 81_000 + i, dev),
               synthetic.torch_normal((n_seq * K, n_kv, hd), 82_000 + i, dev)) for i in range(8)]
    nn = np.full(n_seq, K, np.int32)
    out = torch.empty(n_seq, K, n_q, hd, device=dev)
    import ctypes as C

    from kv_cache_decode_attention_gb300 import _abi

    nb = C.c_int64(0)
    _abi.call("kvd_verify_workspace_bytes", C.byref(probe.layer.L), n_q, K, C.byref(nb))
    ws = torch.empty(int(nb.value), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, with_events=None):
        w = wls[i % R]
        kvd.kv_append(w.layer, drafts[i % 8][0], drafts[i % 8][1], nn)
        if with_events is not None:
            with_events[0].record(stream)
        kvd.decode_attention_verify(qs[i % 8], w.layer, K, out=out, scale=w.scale, workspace=ws)
        if with_events is not None:
            with_events[1].record(stream)
        kvd.kv_truncate_last(w.layer, K)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    with sampler:
        time.sleep(0.3)
        replicas.barrier()
        torch.cuda.synchronize()
        c0 = time.time()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.profiler.start()
        t0.record(stream)
        for j in range(args.steps):
            step(args.warmup + j)
        t1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        replicas.barrier()
        c1 = time.time()
        time.sleep(0.1)
    elapsed_ms = replicas.max_over_ranks(t0.elapsed_time(t1))
    ms_per_step = elapsed_ms / args.steps
    # per step: K appended rows per sequence, the verify's read of every cached row
    # (the drafts included), its K queries and outputs
    step_bytes = K * append_bytes(probe.mode, n_live, hd, n_seq) + bytes_each + 2 * n_seq * (K - 1) * n_q * hd * 4
    gbs = replicas.whole_job_rate(step_bytes * args.steps, elapsed_ms * 1e-3, world) / 1e9
    # the verify call timed inside the same steps run again with events around
    # it (kept out of the timed steps above)
    for j in range(len(ev)):
        step(args.warmup + args.steps + j, ev[j])
    torch.cuda.synchronize()
    ver_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    achieved = (bytes_each + 2 * n_seq * (K - 1) * n_q * hd * 4) / (ver_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    # end to end: the step's queries and drafts copied in (one pinned buffer),
    # the K outputs copied out, every step
    pinned, stage, (dq, ddk, ddv) = packed_inputs(torch, [(qs[i], drafts[i][0], drafts[i][1]) for i in range(8)])
    stages = [(stage, (dq, ddk, ddv)), restage(torch, stage, (dq, ddk, ddv))]
    pin_outs = [torch.empty(out.shape).pin_memory() for _ in range(2)]

    def e2e_step(j, views, last_copy):
        w = wls[j % R]
        wait_copied(torch, last_copy(out))
        kvd.kv_append(w.layer, views[1], views[2], nn)
        kvd.decode_attention_verify(views[0], w.layer, K, out=out, scale=w.scale, workspace=ws)
        kvd.kv_truncate_last(w.layer, K)
        return out, pin_outs[j % 2]

    secs = e2e_pipelined(torch, pinned, stages, args.steps, e2e_step)
    e2e = {"value": round(step_bytes * args.steps / secs / 1e9 * world, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(stage.numel() * 4), "d2h_bytes_per_step": int(pin_outs[0].numel() * 4),
           "mode": "pipelined: inputs copied in on a copy stream while the previous step computes, "
                   "outputs copied out on another, one host synchronisation at the end"}
    torch.cuda.synchronize()
    a0 = time.perf_counter()
    for j in range(args.steps):
        w = wls[j % R]
        stage.copy_(pinned[j % 8], non_blocking=True)
        kvd.kv_append(w.layer, ddk, ddv, nn)
        kvd.decode_attention_verify(dq, w.layer, K, out=out, scale=w.scale, workspace=ws)
        kvd.kv_truncate_last(w.layer, K)
        pin_outs[0].copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    a1 = time.perf_counter()
    e2e_sync = {"value": round(step_bytes * args.steps / (a1 - a0) / 1e9 * world, 2), "unit": "GB/s",
                "mode": "the host waits for every step's result before the next step"}
    for w in wls:
        if w.layer.device_error():
            raise SystemExit("device error word set")
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        info = host_cpu()
        n_par = max(1, min(n_seq, info["nproc"] or 1, args.cpu_sample_seqs))
        smps = [VerifyOracleSample(K, b) for b in range(n_par)]
        v1, _, _ = time_oracle(smps[:1], 1, args.cpu_seconds / 2)
        vn, _, used = time_threaded(smps, n_par, args.cpu_seconds / 2)
        cpu = {"value": round(vn, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": "%d sequences at once, one per thread: %s, %.1f s" % (
                   n_par, smps[0].what, args.cpu_seconds / 2),
               "single_core": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                               "sample": smps[0].what + ", %.1f s" % (args.cpu_seconds / 2)},
               "nproc": info["nproc"], "cpu_model": info["cpu_model"]}
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "verify_q8_gqa", "mode": "q8_2f", "n_seq": n_seq,
                   "cached_rows": int(probe.lengths[0]), "drafts": K, "n_q": n_q, "n_kv": n_kv, "head_dim": hd,
                   "step": "kv_append %d drafts/seq + decode_attention_verify + kv_truncate_last %d" % (K, K),
                   "arithmetic": Q8_ARITHMETIC,
                   "replicas": R, "l2": "inputs larger than L2 (%d rotated cache replicas)" % R,
                   "parallelism": "replicas" if world > 1 else "single"},
        "fraction_of_peak": round(gbs / world / peak, 4),
        "queries_per_s": round(n_seq * K * world / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "decode_attention_verify (split + merge)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "peak_kind": peak_kind,
                     "ms_per_launch": round(ver_ms, 5), "bytes_per_launch": int(bytes_each)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_sync": e2e_sync,
        "gpu_launches": args.steps * 4,
        "clocks": sampler.summary(c0, c1),
    }
    print(json.dumps(line), flush=True)


def run_gpu_ragged(args, rank, world):
    """The ragged serving batch: 256 sequences, lengths U{1..16384}, one layer
    per storage mode (f32, q8, q8k, q8v), 2 of 8 KV heads dead per layer.  One
    step = for every layer, kv_append of one row per sequence + decode_attention
    with imp (a decode token through the four layers).  The layers together hold
    ~34 GB, far above L2, so every step streams HBM."""
    import torch

    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300 import replicas
    from kv_cache_decode_attention_gb300 import workloads as W

    dev = torch.device("cuda", replicas.rank_info().local_rank)
    torch.cuda.set_device(dev)
    n_ev = min(args.steps, 10)
    sync_steps = min(args.steps, 20)
    spare = args.warmup + 2 * args.steps + n_ev + sync_steps + 16
    layers = W.ragged(extra_cap=spare, n_seq=args.ragged_seqs, device=dev)
    w0 = layers[0]
    n_seq, n_q, n_kv, hd = w0.n_seq, w0.n_q, w0.n_kv, w0.hd
    n_live = [int(w.alive.sum()) for w in layers]
    imps = [torch.zeros(w.layer.imp_len, device=dev) for w in layers]
    out_all = torch.empty(len(layers), n_seq, n_q, hd, device=dev)
    outs = [out_all[i] for i in range(len(layers))]
    ws = torch.empty(max(w.layer.workspace_bytes(n_q, True) for w in layers), dtype=torch.uint8, device=dev)
    qs = [[w.query(i, dev) for i in range(8)] for w in layers]
    news = [[w.new_rows(i, dev) for i in range(8)] for w in layers]
    stream = torch.cuda.current_stream()
    lens = np.array([w0.layer.seq_len(b) for b in range(n_seq)], np.int64)  # the same in every layer

    def step(i, ev=None):
        for li, w in enumerate(layers):
            k, v = news[li][i % 8]
            kvd.kv_append(w.layer, k, v)
            if ev is not None:
                ev[li][0].record(stream)
            kvd.decode_attention(qs[li][i % 8], w.layer, out=outs[li], imp=imps[li], scale=w.scale,
                                 workspace=ws)
            if ev is not None:
                ev[li][1].record(stream)

    def step_bytes(lens_after):
        return sum(append_bytes(w.mode, n_live[li], hd, n_seq) +
                   decode_bytes(w.mode, n_live[li], hd, n_q, lens_after, True, n_seq)
                   for li, w in enumerate(layers))

    for i in range(args.warmup):
        step(i)
    lens += args.warmup
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    with sampler:
        time.sleep(0.3)
        replicas.barrier()
        torch.cuda.synchronize()
        c0 = time.time()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.profiler.start()
        t0.record(stream)
        for j in range(args.steps):
            step(args.warmup + j)
        t1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        replicas.barrier()
        c1 = time.time()
        time.sleep(0.1)
    bytes_total = 0
    for j in range(args.steps):
        lens += 1
        bytes_total += step_bytes(lens)
    n_done = args.warmup + args.steps
    elapsed_ms = replicas.max_over_ranks(t0.elapsed_time(t1))
    ms_per_step = elapsed_ms / args.steps
    gbs = replicas.whole_job_rate(bytes_total, elapsed_ms * 1e-3, world) / 1e9

    # each layer's decode with imp, timed inside steps run again with events
    # around it (kept out of the timed steps above)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in layers]
           for _ in range(n_ev)]
    imp_bytes = [0] * len(layers)
    for j in range(n_ev):
        step(n_done + j, evs[j])
        lens += 1
        for li, w in enumerate(layers):
            imp_bytes[li] += decode_bytes(w.mode, n_live[li], hd, n_q, lens, True, n_seq)
    n_done += n_ev
    torch.cuda.synchronize()
    imp_ms = [statistics.mean(evs[j][li][0].elapsed_time(evs[j][li][1]) for j in range(n_ev))
              for li in range(len(layers))]
    imp_bytes = [b / n_ev for b in imp_bytes]

    # ---- per mode: the decode call without imp timed alone (CUDA events on the
    #      launching stream), each layer's calls back to back
    peak, peak_kind = peaks()
    nrep = max(10, min(args.steps, 40))
    per_mode = {}
    k_bytes, k_ms = [], []
    kernels = {F32_MODE: "split_layer_kernel<128,4,f32> + merge_layer_kernel",
               Q8_MODE: "split_warp_kernel (mma.sync) + merge_heads_kernel",
               Q8K_MODE: "split_layer_kernel<128,4,q8k> + merge_layer_kernel",
               Q8V_MODE: "split_layer_kernel<128,4,q8v> + merge_layer_kernel"}
    torch.cuda.profiler.start()  # second profiled range: the per-mode decode calls
    for li, w in enumerate(layers):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nrep)]
        for j in range(nrep):
            ev[j][0].record(stream)
            kvd.decode_attention(qs[li][j % 8], w.layer, out=outs[li], imp=None, scale=w.scale, workspace=ws)
            ev[j][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        nb = decode_bytes(w.mode, n_live[li], hd, n_q, lens, False, n_seq)
        k_bytes.append(nb)
        k_ms.append(ms)
        name = MODE_NAMES[w.mode]
        achieved = nb / (ms * 1e-3) / 1e9
        per_mode[name] = {
            "bound": "hbm", "kernel": kernels[w.mode], "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": measured_traffic("ragged_" + name, nb), "peak_kind": peak_kind,
            "ms_per_launch": round(ms, 5), "bytes_per_launch": int(nb),
            "imp_on": {"ms_per_launch": round(imp_ms[li], 5), "bytes_per_launch": int(imp_bytes[li]),
                       "achieved": round(imp_bytes[li] / (imp_ms[li] * 1e-3) / 1e9, 1),
                       "frac": round(imp_bytes[li] / (imp_ms[li] * 1e-3) / 1e9 / peak, 4)},
        }
    torch.cuda.profiler.stop()
    achieved = sum(k_bytes) / (sum(k_ms) * 1e-3) / 1e9
    tr = [per_mode[MODE_NAMES[w.mode]]["traffic"] for w in layers]

    # ---- end to end through the public API with host buffers: every step's 4
    #      queries and 4 x (k, v) new rows copied in from one pinned buffer, the
    #      4 layers' outputs copied out (pipelined; then synchronising per step)
    parts = [tuple(t for li in range(len(layers)) for t in (qs[li][i], news[li][i][0], news[li][i][1]))
             for i in range(8)]
    pinned, stage, views = packed_inputs(torch, parts)
    stages = [(stage, views), restage(torch, stage, views)]
    pin_outs = [torch.empty(out_all.shape).pin_memory() for _ in range(2)]

    def e2e_step(j, vw, last_copy):
        wait_copied(torch, last_copy(out_all))
        for li, w in enumerate(layers):
            kvd.kv_append(w.layer, vw[3 * li + 1], vw[3 * li + 2])
            kvd.decode_attention(vw[3 * li], w.layer, out=outs[li], imp=imps[li], scale=w.scale, workspace=ws)
        return out_all, pin_outs[j % 2]

    lens_b = lens.copy()
    secs = e2e_pipelined(torch, pinned, stages, args.steps, e2e_step)
    eb = 0
    for j in range(args.steps):
        lens += 1
        eb += step_bytes(lens)
    e2e = {"value": round(eb / secs / 1e9 * world, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(stage.numel() * 4), "d2h_bytes_per_step": int(out_all.numel() * 4),
           "mode": "pipelined: inputs copied in on a copy stream while the previous step computes, "
                   "outputs copied out on another, one host synchronisation at the end"}
    torch.cuda.synchronize()
    eb = 0
    a0 = time.perf_counter()
    for j in range(sync_steps):
        stage.copy_(pinned[j % 8], non_blocking=True)
        for li, w in enumerate(layers):
            kvd.kv_append(w.layer, views[3 * li + 1], views[3 * li + 2])
            kvd.decode_attention(views[3 * li], w.layer, out=outs[li], imp=imps[li], scale=w.scale,
                                 workspace=ws)
        pin_outs[0].copy_(out_all, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    a1 = time.perf_counter()
    for j in range(sync_steps):
        lens += 1
        eb += step_bytes(lens)
    e2e_sync = {"value": round(eb / (a1 - a0) / 1e9 * world, 2), "unit": "GB/s",
                "mode": "the host waits for every step's result before the next step"}
    del lens_b
    for w in layers:
        err = w.layer.device_error()
        if err:
            raise SystemExit("device error word set: %d" % err)
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        del layers, qs, news, imps, out_all, outs, ws, pinned, stage, views, stages
        torch.cuda.empty_cache()
        single, multi, w1, wn = ragged_samples(args.cpu_sample_seqs, args.ragged_seqs)
        cpu = cpu_baseline_gqa(single, multi, args.cpu_seconds, w1, wn)
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "ragged", "n_seq": n_seq, "lengths": "U{1..16384}, seed 7 (mean %.0f at the start)"
                   % float(np.mean(synthetic_lengths(n_seq))),
                   "n_q": n_q, "n_kv": n_kv, "head_dim": hd,
                   "layers": "f32, q8 (q8_2f), q8k, q8v; 2 of 8 KV heads dead per layer",
                   "step": "per layer: kv_append 1 row/seq + decode_attention with imp",
                   "arithmetic": "f32 CUDA-core dots (f32, q8k, q8v layers); q8 layer: " + Q8_ARITHMETIC,
                   "l2": "inputs larger than L2 (%.1f GB read per step)" % (bytes_total / args.steps / 1e9),
                   "parallelism": "replicas" if world > 1 else "single"},
        "fraction_of_peak": round(gbs / world / peak, 4),
        "queries_per_s": round(n_seq * world / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "decode_attention over the four layers (imp off; per mode below)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": int(sum(tr)) if all(t is not None for t in tr) else None,
                     "peak_kind": peak_kind, "ms_per_launch": round(sum(k_ms), 5),
                     "bytes_per_launch": int(sum(k_bytes))},
        "per_mode": per_mode,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_sync": e2e_sync,
        "gpu_launches": args.steps * 16,
        "clocks": sampler.summary(c0, c1),
    }
    print(json.dumps(line), flush=True)


def synthetic_lengths(n_seq):
    import synthetic

    return synthetic.ragged_batch(n_seq)[0]


def build_workload(name: str, replicas: int):
    from kv_cache_decode_attention_gb300 import workloads as W

    # spare rows for the appends of the timed, event and end-to-end steps (long_q8
    # runs one replica, so every step lands on it)
    builders = {"q8_gqa": lambda: W.q8_gqa(extra_cap=512), "long_q8": lambda: W.long_q8(extra_cap=1536),
                "tiny_f32": lambda: W.tiny_f32(extra_cap=64)}
    if name not in builders:
        raise SystemExit("unknown workload %s" % name)
    return [builders[name]() for _ in range(replicas)]


def run_gpu(args, rank, world):
    import torch

    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300 import workloads as W

    from kv_cache_decode_attention_gb300 import replicas

    dev = torch.device("cuda", replicas.rank_info().local_rank)
    torch.cuda.set_device(dev)

    probe = build_workload(args.workload, 1)
    wl0 = probe[0]
    n_live = int(wl0.alive.sum())
    ws_bytes_each = decode_bytes(wl0.mode, n_live, wl0.hd, wl0.n_q, wl0.lengths, True, wl0.n_seq)
    R = max(1, min(8, math.ceil(4 * L2_BYTES / ws_bytes_each)))
    wls = probe + build_workload(args.workload, R - 1)
    n_steps = args.warmup + args.steps
    extra = int(wl0.layer.capacity[0] - wl0.lengths[0])
    if math.ceil(2 * n_steps / R) > extra:
        raise SystemExit("too many steps for the cache capacity (%d rows spare)" % extra)

    # per-replica buffers, all resident before timing
    imps = [torch.zeros(w.layer.imp_len, device=dev) for w in wls]
    outs = [torch.empty(w.n_seq, w.n_q, w.hd, device=dev) for w in wls]
    ws = torch.empty(max(w.layer.workspace_bytes(w.n_q, True) for w in wls), dtype=torch.uint8, device=dev)
    qs = [wl0.query(i, dev) for i in range(8)]
    news = [wl0.new_rows(i, dev) for i in range(8)]
    stream = torch.cuda.current_stream()

    def step(i, with_events=None):
        w = wls[i % R]
        k, v = news[i % 8]
        kvd.kv_append(w.layer, k, v)
        if with_events is not None:
            with_events[0].record(stream)
        kvd.decode_attention(qs[i % 8], w.layer, out=outs[i % R], imp=imps[i % R], scale=w.scale,
                             workspace=ws)
        if with_events is not None:
            with_events[1].record(stream)

    def lengths_now():
        return [np.array([w.layer.seq_len(b) for b in range(w.n_seq)], np.int64) for w in wls]

    # ---- warm-up
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # ---- timed region
    bytes_total = 0
    n_ev = min(args.steps, 10)  # steps run again with events around the decode, after the timing
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_ev)]
    lens_before = lengths_now()
    sampler = ClockSampler(dev.index)
    with sampler:
        time.sleep(0.3)
        replicas.barrier()
        torch.cuda.synchronize()
        c0 = time.time()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.profiler.start()  # profilers started with capture off record only this range
        t0.record(stream)
        for j in range(args.steps):
            step(args.warmup + j)
        t1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        replicas.barrier()
        c1 = time.time()
        time.sleep(0.1)
    elapsed_ms = t0.elapsed_time(t1)
    # algorithmic bytes of exactly the timed steps (lengths known on the host)
    lens = [l.copy() for l in lens_before]
    for j in range(args.steps):
        r = (args.warmup + j) % R
        w = wls[r]
        bytes_total += append_bytes(w.mode, n_live, w.hd, w.n_seq)
        lens[r] += 1
        bytes_total += decode_bytes(w.mode, n_live, w.hd, w.n_q, lens[r], True, w.n_seq)
    # the decode's share of a step, from steps run again with events around it
    # (kept out of the timed steps above)
    for j in range(n_ev):
        step(n_steps + j, ev[j])
    torch.cuda.synchronize()
    dec_ms = [a.elapsed_time(b) for a, b in ev]
    n_steps += n_ev
    elapsed_ms = replicas.max_over_ranks(elapsed_ms)  # every rank ran its own replica
    ms_per_step = elapsed_ms / args.steps
    gbs = replicas.whole_job_rate(bytes_total, elapsed_ms * 1e-3, world) / 1e9

    # ---- dominant kernel: the decode call without imp, timed alone (same
    #      workload and launch configuration, CUDA events on the launching stream)
    nrep = max(20, args.steps)
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nrep)]
    torch.cuda.profiler.start()  # second profiled range: the decode calls of the roofline
    for j in range(nrep):
        w = wls[j % R]
        dev_ev[j][0].record(stream)
        kvd.decode_attention(qs[j % 8], w.layer, out=outs[j % R], imp=None, scale=w.scale, workspace=ws)
        dev_ev[j][1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    k_ms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
    lens_now = lengths_now()
    kbytes = statistics.mean(
        decode_bytes(wls[j % R].mode, n_live, wl0.hd, wl0.n_q, lens_now[j % R], False, wl0.n_seq)
        for j in range(nrep))
    # the same calls with imp on (the score round trip and the imp pass), timed alone
    for j in range(nrep):
        w = wls[j % R]
        dev_ev[j][0].record(stream)
        kvd.decode_attention(qs[j % 8], w.layer, out=outs[j % R], imp=imps[j % R], scale=w.scale, workspace=ws)
        dev_ev[j][1].record(stream)
    torch.cuda.synchronize()
    imp_ms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
    imp_bytes = statistics.mean(
        decode_bytes(wls[j % R].mode, n_live, wl0.hd, wl0.n_q, lens_now[j % R], True, wl0.n_seq)
        for j in range(nrep))
    # decode_attention_static (no workspace: the library's scratch array, the
    # CUDA-core split kernel) on the same calls, where its partials fit
    static_ms = None
    try:
        for j in range(nrep):
            w = wls[j % R]
            dev_ev[j][0].record(stream)
            kvd.decode_attention_static(qs[j % 8], w.layer, out=outs[j % R], scale=w.scale)
            dev_ev[j][1].record(stream)
        torch.cuda.synchronize()
        static_ms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
    except kvd.KvdError:
        torch.cuda.synchronize()
    peak, peak_kind = peaks()
    achieved = kbytes / (k_ms * 1e-3) / 1e9
    tpeak, tpeak_kind = tensor_peak()
    kflops = statistics.mean(
        decode_flops(n_live, wl0.hd, wl0.n_q // wl0.n_kv, lens_now[j % R], wl0.n_seq) for j in range(nrep))
    kflops = int(kflops)

    # ---- end to end through the public API with host buffers: pipelined (the
    #      headline), then the same steps synchronising on every step's result
    pinned, stage, (dq, dk, dv) = packed_inputs(torch, [(qs[i], news[i][0], news[i][1]) for i in range(8)])
    stages = [(stage, (dq, dk, dv)), restage(torch, stage, (dq, dk, dv))]
    pin_outs = [torch.empty(wl0.n_seq, wl0.n_q, wl0.hd).pin_memory() for _ in range(2)]
    e2e_steps = args.steps
    sync_steps = min(e2e_steps, 50)  # the synchronised leg: a shorter sample of the same steps
    if math.ceil(2 * (n_steps + e2e_steps + sync_steps) / R) > extra:
        e2e_steps = sync_steps = 0
    e2e = e2e_sync = None

    def e2e_bytes(first, count, lens_b):
        eb = 0
        lens_e = [l.copy() for l in lens_b]
        for j in range(count):
            r = (first + j) % R
            w = wls[r]
            lens_e[r] += 1
            eb += append_bytes(w.mode, n_live, w.hd, w.n_seq)
            eb += decode_bytes(w.mode, n_live, w.hd, w.n_q, lens_e[r], True, w.n_seq)
        return eb

    def e2e_step(j, views, last_copy):
        i = n_steps + j
        w, o = wls[i % R], outs[i % R]
        wait_copied(torch, last_copy(o))  # o's previous copy out has left before it is rewritten
        kvd.kv_append(w.layer, views[1], views[2])
        kvd.decode_attention(views[0], w.layer, out=o, imp=imps[i % R], scale=w.scale, workspace=ws)
        return o, pin_outs[j % 2]

    if e2e_steps:
        lens_b = lengths_now()
        secs = e2e_pipelined(torch, pinned, stages, e2e_steps, e2e_step)
        e2e = {"value": round(e2e_bytes(n_steps, e2e_steps, lens_b) / secs / 1e9 * world, 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(dq.numel() * 4 + dk.numel() * 4 + dv.numel() * 4),
               "d2h_bytes_per_step": int(pin_outs[0].numel() * 4),
               "mode": "pipelined: inputs copied in on a copy stream while the previous step computes, "
                       "outputs copied out on another, one host synchronisation at the end"}
        first = n_steps + e2e_steps
        torch.cuda.synchronize()
        lens_b = lengths_now()
        a0 = time.perf_counter()
        for j in range(sync_steps):
            i = first + j
            w = wls[i % R]
            stage.copy_(pinned[i % 8], non_blocking=True)
            kvd.kv_append(w.layer, dk, dv)
            kvd.decode_attention(dq, w.layer, out=outs[i % R], imp=imps[i % R], scale=w.scale, workspace=ws)
            pin_outs[0].copy_(outs[i % R], non_blocking=True)
            torch.cuda.current_stream().synchronize()
        a1 = time.perf_counter()
        e2e_sync = {"value": round(e2e_bytes(first, sync_steps, lens_b) / (a1 - a0) / 1e9 * world, 2),
                    "unit": "GB/s", "mode": "the host waits for every step's result before the next step"}
    for w in wls:
        err = w.layer.device_error()
        if err:
            raise SystemExit("device error word set: %d" % err)

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        single, multi, w1, wn = gqa_samples(wl0.name, args.cpu_sample_seqs)
        cpu = cpu_baseline_gqa(single, multi, args.cpu_seconds, w1, wn)
    clocks = sampler.summary(c0, c1)
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl0.name, "mode": "q8_2f", "n_seq": wl0.n_seq,
                   "cached_rows": int(wl0.lengths[0]), "n_q": wl0.n_q, "n_kv": wl0.n_kv,
                   "head_dim": wl0.hd, "step": "kv_append 1 row/seq + decode_attention with imp",
                   "arithmetic": Q8_ARITHMETIC,
                   "replicas": R, "l2": "inputs larger than L2 (%d rotated cache replicas)" % R,
                   "parallelism": "replicas" if world > 1 else "single"},
        "fraction_of_peak": round(gbs / world / peak, 4),
        "queries_per_s": round(wl0.n_seq * world / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "decode_attention (split + merge, imp off)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": measured_traffic(wl0.name, kbytes),
                     "peak_kind": peak_kind, "ms_per_launch": round(k_ms, 5),
                     "bytes_per_launch": int(kbytes),
                     "imp_on": {"ms_per_launch": round(imp_ms, 5), "bytes_per_launch": int(imp_bytes),
                                "achieved": round(imp_bytes / (imp_ms * 1e-3) / 1e9, 1),
                                "frac": round(imp_bytes / (imp_ms * 1e-3) / 1e9 / peak, 4)},
                     "static": None if static_ms is None else
                     {"kernel": "decode_attention_static (CUDA-core split + merge, no workspace)",
                      "ms_per_launch": round(static_ms, 5), "bytes_per_launch": int(kbytes),
                      "achieved": round(kbytes / (static_ms * 1e-3) / 1e9, 1),
                      "frac": round(kbytes / (static_ms * 1e-3) / 1e9 / peak, 4)}},
        # the second roof: the same decode call against the tensor peak (the
        # q8_2f kernels run each contraction twice, one f16 term each)
        "roofline_tensor": {"bound": "tensor", "achieved": round(kflops / (k_ms * 1e-3) / 1e12, 2),
                            "peak": tpeak, "unit": "TFLOP/s",
                            "frac": round(kflops / (k_ms * 1e-3) / 1e12 / tpeak, 4), "peak_kind": tpeak_kind,
                            "flops_per_launch": kflops, "executed_flops_per_launch": 2 * kflops}
        if wl0.mode == Q8_MODE else None,
        "decode_ms_in_step": round(statistics.mean(dec_ms), 5),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_sync": e2e_sync,
        "gpu_launches": args.steps * 4,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="ragged",
                    choices=["ragged", "q8_gqa", "long_q8", "tiny_f32", "verify_q8", *RSWA_WORKLOADS])
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of oracle decoding for the CPU baseline (half on one core, half on all)")
    ap.add_argument("--cpu-sample-seqs", type=int, default=16,
                    help="sequences (streams) in the all-core CPU baseline sample")
    ap.add_argument("--ragged-seqs", type=int, default=256,
                    help="sequences of the ragged batch (256 = the measured configuration; fewer keeps "
                         "the first ones, for small profiler captures)")
    ap.add_argument("--rswa-streams", type=int, default=16,
                    help="streams of the R-SWA workloads (16 = the measured configuration)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    from kv_cache_decode_attention_gb300.replicas import rank_info

    info = rank_info()
    world, rank = info.world, info.rank
    if world > 1 and args.impl != "reference":
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(info.local_rank)
        dist.init_process_group("nccl")
    from __graft_entry__ import build

    if args.impl == "reference":
        if rank == 0:
            from oracle.oracle import build_oracle

            build_oracle()
            if args.workload in RSWA_WORKLOADS:
                build()
        run_reference(args, rank)
        return
    build()
    if args.workload == "ragged":
        run_gpu_ragged(args, rank, world)
    elif args.workload in RSWA_WORKLOADS:
        run_gpu_rswa(args, rank, world)
    elif args.workload == "verify_q8":
        run_gpu_verify(args, rank, world)
    else:
        run_gpu(args, rank, world)


if __name__ == "__main__":
    main()
