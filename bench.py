#!/usr/bin/env python
"""Decode-attention benchmark on GB300: KV GB/s (fraction of the HBM roofline)
and decode queries/s.

Default workload: q8_2f GQA decode, 32 sequences x 4096 cached rows, 32 query
/ 8 KV heads, head_dim 128, the cache built one row at a time through
kv_append (freeze and requantisation at row 64).  One step = the whole hot
path for one decode token: kv_append of one new K/V row per sequence
(quantised against the frozen fields) + decode_attention over every cached
row with the attention-mass (imp) accumulation.  The timed region holds
exactly --steps steps between a barrier + device synchronisation on each side;
--warmup steps run untimed first.  Two cache replicas alternate step by step
so that every step streams HBM, not L2 (2 x 289 MB > 129 MB of L2).

Other workloads (--workload): long_q8 (4 sequences x 131072 rows, 64 query /
4 KV heads), tiny_f32, and the R-SWA decode of franken_ocr's rswa module
(16 streams x 10 heads, a 32640-row reference block + a full 128-slot ring):
rswa reads the f32 regions, rswa_i8 the int8 mirror; one step = the ring
write of one token per stream (mirror included) + the decode of every stream.

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
L2_BYTES = 129 * 1024 * 1024
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode call
# without imp -- the split kernel plus the run merge -- from one ncu capture of
# this benchmark's roofline loop (command and figures in
# profiles/decode_q8_gqa_traffic.md), valid while the kernel sources hash to
# the captured version; reported as null otherwise.  The capture ran 25 steps
# (cache rows 4096 + 25); a run of another length reports it scaled by its
# algorithmic bytes over the capture's (both are rows x bytes per row plus a
# small fixed part).
TRAFFIC = {
    "q8_gqa": {"sources_sha256": "813bda5fa871babc27a6d8f99409a7ac294be15c3a90ad55523a3c5f51eb5034",
               "bytes": 300582016, "algorithmic_bytes": 291600896},
}


def kernel_sources_sha256() -> str:
    import hashlib

    csrc = os.path.join(ROOT, "kv_cache_decode_attention_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(workload: str, bytes_per_launch=None):
    t = TRAFFIC.get(workload)
    if not t or t["bytes"] is None or t["sources_sha256"] != kernel_sources_sha256():
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

def oracle_sample_gbs(wl, n_seq_sample: int, min_seconds: float, max_reps: int | None = None):
    """Time the CPU oracle (single thread) decoding `n_seq_sample` sequences of
    the workload (every query head, every cached row, f64 two-pass softmax)."""
    import oracle
    import torch

    from kv_cache_decode_attention_gb300 import workloads as W

    caches, qs = [], []
    q_all = wl.query(10_000).cpu().numpy()
    for b in range(n_seq_sample):
        k, v = wl.rows(b)
        k, v = k.cpu().numpy(), v.cpu().numpy()
        oc = oracle.OracleSeqCache(wl.mode, wl.n_kv, wl.hd, int(wl.lengths[b]), alive=wl.alive)
        oc.append_rows(k, v)
        caches.append(oc)
        qs.append(q_all[b])
        del k, v
        torch.cuda.empty_cache()
    n_live = int(wl.alive.sum())
    bytes_per = W.decode_bytes(wl.mode, n_live, wl.hd, wl.n_q, wl.lengths[:n_seq_sample], True,
                               n_seq_sample)
    reps, t0 = 0, time.perf_counter()
    while True:
        for b, oc in enumerate(caches):
            imp = np.zeros(oc.cap)
            oc.decode(qs[b], wl.n_q, np.float32(wl.scale), imp)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or (max_reps is not None and reps >= max_reps):
            break
    per_rep = el / reps
    return bytes_per / per_rep / 1e9, per_rep, bytes_per


class RswaOracleSample:
    """One stream of an R-SWA workload rebuilt on the host from the workload's
    generators (its reference rows and the ring rows of its 500 writes), ready
    for the CPU oracle's decode (f32 regions, or their int8 mirror)."""

    def __init__(self, wl, int8: bool, s: int = 0, verify_k: int = 0):
        import oracle

        c = wl.cache
        self.int8, self.H, self.hd, self.verify_k = int8, c.H, c.head_dim, verify_k
        pk, pv = wl.prefill_rows(s)
        self.ref_k, self.ref_v = pk.cpu().numpy(), pv.cpu().numpy()
        self.ring_k = np.zeros((c.H, c.W, c.head_dim), np.float32)
        self.ring_v = np.zeros_like(self.ring_k)
        cur = np.zeros(2, np.int32)
        for t in range(wl.steps):
            k, v = wl.step_rows(t)
            oracle.rswa_write(self.ring_k, self.ring_v, k[s].cpu().numpy(), v[s].cpu().numpy(), True, cur)
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
        from kv_cache_decode_attention_gb300 import workloads as W

        self.bytes = (W.rswa_i8_bytes if int8 else W.rswa_bytes)(1, c.H, c.head_dim, [self.rows])
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


def run_reference(args, rank):
    """--impl reference: the CPU oracle as it stands, on the host cores, each
    step a bounded sample (one sequence, every head and cached row) of the
    workload; rank 0 only."""
    if rank != 0:
        return
    import torch

    from kv_cache_decode_attention_gb300 import workloads as W

    if not torch.cuda.is_available():
        print(json.dumps({"impl": "reference", "unavailable": "needs the GPU box to build the workload"}))
        return
    if args.workload in RSWA_WORKLOADS:
        int8, verify = args.workload.startswith("rswa_i8"), args.workload.endswith("_verify")
        wl = W.rswa_steady(B=args.rswa_streams, int8=int8)
        smp = RswaOracleSample(wl, int8, verify_k=VERIFY_DRAFTS if verify else 0)
        smp.gbs(0.0, max_reps=max(1, args.warmup))
        gbs, per = smp.gbs(0.0, max_reps=args.steps)
        sample, name = smp.describe(wl), args.workload + "_steady"
    elif args.workload == "verify_q8":
        import oracle
        import synthetic

        K = VERIFY_DRAFTS
        wl = W.q8_gqa(extra_cap=64)
        k, v = wl.rows(0)
        oc = oracle.OracleSeqCache(wl.mode, wl.n_kv, wl.hd, int(wl.lengths[0]) + K, alive=wl.alive)
        oc.append_rows(k.cpu().numpy(), v.cpu().numpy())
        oc.append_rows(synthetic.normal((K, wl.n_kv, wl.hd), 91_000), synthetic.normal((K, wl.n_kv, wl.hd), 91_001))
        q0 = synthetic.normal((K, wl.n_q, wl.hd), 91_002)
        one = W.decode_bytes(wl.mode, int(wl.alive.sum()), wl.hd, wl.n_q, wl.lengths[:1] + K, False, 1)
        for _ in range(max(1, args.warmup)):
            oc.decode_verify(q0, wl.n_q, K, np.float32(wl.scale))
        a0 = time.perf_counter()
        for _ in range(args.steps):
            oc.decode_verify(q0, wl.n_q, K, np.float32(wl.scale))
        per = (time.perf_counter() - a0) / args.steps
        gbs = one / per / 1e9
        sample = "1 of %d sequences (%d drafts x %d query heads x %d rows), f64" % (
            wl.n_seq, K, wl.n_q, int(wl.lengths[0]) + K)
        name = "verify_q8_gqa"
    else:
        wl = build_workload(args.workload, replicas=1)[0]
        # warm-up and timed steps: one oracle decode of the sampled sequence each
        gbs_w, _, _ = oracle_sample_gbs(wl, 1, 0.0, max_reps=max(1, args.warmup))
        gbs, per, nbytes = oracle_sample_gbs(wl, 1, 0.0, max_reps=args.steps)
        sample = "1 of %d sequences (all %d query heads, %d rows), f64 two-pass softmax" % (
            wl.n_seq, wl.n_q, int(wl.lengths[0]))
        name = wl.name
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "queries_per_s": round(1.0 / per, 4),
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
    dec_bytes = (W.rswa_i8_bytes if int8 else W.rswa_bytes)(B, H, hd, lengths)
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
        smp = RswaOracleSample(wl, int8, verify_k=K if verify else 0)
        v, per = smp.gbs(args.cpu_seconds)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": smp.describe(wl) + ", %.1f s" % args.cpu_seconds}
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8" if int8 else "f32", "data": "synthetic",
        "config": {"workload": args.workload + "_steady", "streams": B, "heads": H, "head_dim": hd,
                   "reference_rows": int(wl.prefill), "ring_rows": int(c.W),
                   "step": ("rswa verify of %d drafts/stream (read-only) + ring write of the accepted token" % K
                            if verify else "rswa ring write 1 token/stream + decode of every stream"),
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
    bytes_each = W.decode_bytes(probe.mode, n_live, probe.hd, probe.n_q, probe.lengths + K, False, probe.n_seq)
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
    step_bytes = K * W.append_bytes(probe.mode, n_live, hd, n_seq) + bytes_each + 2 * n_seq * (K - 1) * n_q * hd * 4
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
        import oracle

        k, v = probe.rows(0)
        oc = oracle.OracleSeqCache(probe.mode, n_kv, hd, int(probe.lengths[0]) + K, alive=probe.alive)
        oc.append_rows(k.cpu().numpy(), v.cpu().numpy())
        dk = drafts[0][0].cpu().numpy().reshape(n_seq, K, n_kv, hd)[0]
        dv = drafts[0][1].cpu().numpy().reshape(n_seq, K, n_kv, hd)[0]
        oc.append_rows(dk, dv)
        q0 = qs[0][0].cpu().numpy()
        reps, a0 = 0, time.perf_counter()
        while time.perf_counter() - a0 < args.cpu_seconds:
            oc.decode_verify(q0, n_q, K, np.float32(probe.scale))
            reps += 1
        per = (time.perf_counter() - a0) / reps
        one = W.decode_bytes(probe.mode, n_live, hd, n_q, probe.lengths[:1] + K, False, 1)
        cpu = {"value": round(one / per / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "1 of %d sequences (%d drafts x %d query heads x %d rows), f64, %.1f s" % (
                   n_seq, K, n_q, int(probe.lengths[0]) + K, args.cpu_seconds)}
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "verify_q8_gqa", "mode": "q8_2f", "n_seq": n_seq,
                   "cached_rows": int(probe.lengths[0]), "drafts": K, "n_q": n_q, "n_kv": n_kv, "head_dim": hd,
                   "step": "kv_append %d drafts/seq + decode_attention_verify + kv_truncate_last %d" % (K, K),
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


def build_workload(name: str, replicas: int):
    from kv_cache_decode_attention_gb300 import workloads as W

    builders = {"q8_gqa": W.q8_gqa, "long_q8": W.long_q8, "tiny_f32": W.tiny_f32}
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
    ws_bytes_each = W.decode_bytes(wl0.mode, n_live, wl0.hd, wl0.n_q, wl0.lengths, True, wl0.n_seq)
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
        bytes_total += W.append_bytes(w.mode, n_live, w.hd, w.n_seq)
        lens[r] += 1
        bytes_total += W.decode_bytes(w.mode, n_live, w.hd, w.n_q, lens[r], True, w.n_seq)
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
        W.decode_bytes(wls[j % R].mode, n_live, wl0.hd, wl0.n_q, lens_now[j % R], False, wl0.n_seq)
        for j in range(nrep))
    peak, peak_kind = peaks()
    achieved = kbytes / (k_ms * 1e-3) / 1e9

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
            eb += W.append_bytes(w.mode, n_live, w.hd, w.n_seq)
            eb += W.decode_bytes(w.mode, n_live, w.hd, w.n_q, lens_e[r], True, w.n_seq)
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
    if not args.no_cpu_baseline and world >= 1:
        v, per, nb = oracle_sample_gbs(wl0, 1, args.cpu_seconds)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "1 of %d sequences (all %d query heads x %d rows) decoded in f64, "
                         "%.1f s" % (wl0.n_seq, wl0.n_q, int(wl0.lengths[0]), args.cpu_seconds)}
    clocks = sampler.summary(c0, c1)
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl0.name, "mode": "q8_2f", "n_seq": wl0.n_seq,
                   "cached_rows": int(wl0.lengths[0]), "n_q": wl0.n_q, "n_kv": wl0.n_kv,
                   "head_dim": wl0.hd, "step": "kv_append 1 row/seq + decode_attention with imp",
                   "replicas": R, "l2": "inputs larger than L2 (%d rotated cache replicas)" % R,
                   "parallelism": "replicas" if world > 1 else "single"},
        "fraction_of_peak": round(gbs / world / peak, 4),
        "queries_per_s": round(wl0.n_seq * world / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "decode_attention (split + merge, imp off)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": measured_traffic(wl0.name, kbytes),
                     "peak_kind": peak_kind, "ms_per_launch": round(k_ms, 5),
                     "bytes_per_launch": int(kbytes)},
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
    ap.add_argument("--workload", default="q8_gqa",
                    choices=["q8_gqa", "long_q8", "tiny_f32", "verify_q8", *RSWA_WORKLOADS])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
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
            build()
        run_reference(args, rank)
        return
    build()
    if args.workload in RSWA_WORKLOADS:
        run_gpu_rswa(args, rank, world)
    elif args.workload == "verify_q8":
        run_gpu_verify(args, rank, world)
    else:
        run_gpu(args, rank, world)


if __name__ == "__main__":
    main()
