"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by
element, on seeded inputs that span several tiles, several chunks and ragged
tails, plus the edge cases (empty and one-row sequences, exactly 64 rows, dead
groups, every storage mode, head_dim 64 and 128, 1..16 query heads per group).
"""

import math

import numpy as np
import pytest

import oracle
import synthetic
from helpers import (OUT_TOL, assert_imp_close, assert_storage_bitexact, gpu_append_bulk,
                     gpu_append_stepwise, oracle_caches, out_error, seq_rows)

pytestmark = pytest.mark.gpu

MODES = {"f32": oracle.F32, "q8": oracle.Q8, "q8k": oracle.Q8K, "q8v": oracle.Q8V}


@pytest.fixture(scope="module")
def torch():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


@pytest.fixture(scope="module")
def kvd(torch):
    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300.build import build

    build()
    return kvd


def _layer(kvd, mode, lengths, n_kv, hd, alive, cap_extra=0):
    cap = [max(int(L) + cap_extra, 1) for L in lengths]
    return kvd.LayerKvCache(len(lengths), n_kv, hd, mode, cap, alive=alive)


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("hd", [128, 64])
@pytest.mark.parametrize("how", ["stepwise", "bulk"])
def test_append_and_freeze_bitexact(torch, kvd, mode, hd, how):
    lengths = [0, 1, 63, 64, 65, 130, 300]
    n_kv, alive = 4, np.array([1, 0, 1, 1], np.uint8)
    ks, vs = seq_rows(lengths, n_kv, hd, seed=5)
    layer = _layer(kvd, MODES[mode], lengths, n_kv, hd, alive, cap_extra=7)
    # canary: unwritten storage holds NaN bit patterns, never read as data
    for b in layer.bufs[:6]:
        if b is not None:
            b.fill_(0xFF)
    if how == "stepwise":
        gpu_append_stepwise(layer, ks, vs, torch)
    else:
        gpu_append_bulk(layer, ks, vs, torch, pieces=(0.3, 0.75, 1.0))
    torch.cuda.synchronize()
    ocs = oracle_caches(MODES[mode], lengths, n_kv, hd, alive, ks, vs, cap=max(lengths) + 8)
    assert_storage_bitexact(layer, ocs, torch)
    assert layer.memory_bytes() == sum(o.memory_bytes() for o in ocs)
    assert layer.device_error() == 0


def test_explicit_freeze_is_idempotent_and_matches_oracle(torch, kvd):
    lengths = [64, 70, 10]
    n_kv, hd = 2, 128
    ks, vs = seq_rows(lengths, n_kv, hd, seed=6)
    layer = _layer(kvd, oracle.Q8, lengths, n_kv, hd, None, cap_extra=4)
    gpu_append_bulk(layer, ks, vs, torch)
    assert [layer.frozen(b) for b in range(3)] == [False, True, False]
    kvd.kv_freeze_colfield(layer)
    kvd.kv_freeze_colfield(layer)
    torch.cuda.synchronize()
    ocs = oracle_caches(oracle.Q8, lengths, n_kv, hd, None, ks, vs, cap=80)
    for oc in ocs:
        oc.freeze_if_due()
    assert [layer.frozen(b) for b in range(3)] == [True, True, False]
    assert_storage_bitexact(layer, ocs, torch)


def _decode_case(torch, kvd, mode, hd, hpk, lengths, alive, seed, with_imp=True, opts=None):
    n_kv = len(alive)
    n_q = n_kv * hpk
    ks, vs = seq_rows(lengths, n_kv, hd, seed=seed)
    layer = _layer(kvd, mode, lengths, n_kv, hd, alive, cap_extra=3)
    for b in layer.bufs[:6]:
        if b is not None:
            b.fill_(0xFF)
    gpu_append_bulk(layer, ks, vs, torch, pieces=(0.5, 1.0))
    q = synthetic.normal((len(lengths), n_q, hd), seed + 77)
    imp0 = synthetic.rng(seed + 78).uniform(0.0, 2.0, layer.imp_len).astype(np.float32)
    qd = torch.from_numpy(q).cuda()
    imp = torch.from_numpy(imp0).cuda() if with_imp else None
    scale = 1.0 / math.sqrt(hd)
    opts = dict(opts or {})
    sinks = opts.get("sinks")
    gpu_opts = dict(opts)
    if sinks is not None:
        gpu_opts["sinks"] = torch.from_numpy(np.asarray(sinks, np.float32)).cuda()
    out = kvd.decode_attention(qd, layer, imp=imp, scale=scale, **gpu_opts)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    out = out.cpu().numpy()
    ocs = oracle_caches(mode, lengths, n_kv, hd, alive, ks, vs, cap=max(lengths) + 4)
    assert_storage_bitexact(layer, ocs, torch)
    ref = np.zeros((len(lengths), n_q, hd))
    live_mask = np.zeros((len(lengths), n_q), bool)
    imp_ref = imp0.astype(np.float64).copy()
    for b, oc in enumerate(ocs):
        ib = int(layer.imp_base[b])
        seg = imp_ref[ib:ib + max(lengths[b], 1)].copy() if lengths[b] else None
        if opts:
            ref[b] = oc.decode_ex(q[b], n_q, np.float32(scale), opts.get("window", 0),
                                  opts.get("softcap", 0.0), sinks, seg)
        else:
            ref[b] = oc.decode(q[b], n_q, np.float32(scale), seg)
        if seg is not None:
            imp_ref[ib:ib + lengths[b]] = seg[:lengths[b]]
        for h in range(n_q):
            live_mask[b, h] = bool(alive[h // hpk]) and lengths[b] > 0
    # dead groups and empty sequences: exact zeros
    assert np.all(out[~live_mask] == 0.0)
    err = out_error(out, ref, live_mask)
    assert err <= OUT_TOL, err
    if with_imp:
        got = imp.cpu().numpy()
        for b in range(len(lengths)):
            ib = int(layer.imp_base[b])
            assert_imp_close(got[ib:ib + lengths[b]], imp_ref[ib:ib + lengths[b]])
        # rows beyond each sequence are untouched
        untouched = np.ones(layer.imp_len, bool)
        for b in range(len(lengths)):
            ib = int(layer.imp_base[b])
            untouched[ib:ib + lengths[b]] = False
        assert np.array_equal(got[untouched], imp0[untouched])
    return err


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("hpk", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 13, 16])
def test_decode_parity_hd128(torch, kvd, mode, hpk):
    _decode_case(torch, kvd, MODES[mode], 128, hpk, [0, 1, 64, 300, 777, 1030],
                 np.array([1, 1, 0, 1], np.uint8), seed=11 + hpk)


# More sequences than one launch describes (appends, freezes and the
# tensor-core tables go in slices of 256): every sequence against the oracle,
# storage bit-exact, on the tensor-core path (q8) and the CUDA-core one (q8k).
@pytest.mark.parametrize("mode", ["q8", "q8k"])
def test_decode_parity_over_two_launch_slices(torch, kvd, mode):
    lengths = [int(x) for x in synthetic.rng(97).integers(0, 180, 300)]
    _decode_case(torch, kvd, MODES[mode], 128, 4, lengths, np.array([1, 0, 1], np.uint8), seed=97)


# The tensor-core kernels compile the imp score stores out when the call has no
# imp: each of those variants (heads in N with packed or chained query terms,
# heads in M), the benchmark's roofline kernel among them.
@pytest.mark.parametrize("hpk", [1, 4, 8, 16])
def test_decode_q8_without_imp(torch, kvd, hpk):
    _decode_case(torch, kvd, oracle.Q8, 128, hpk, [0, 1, 64, 300, 777, 1030, 2100],
                 np.array([1, 1, 0, 1], np.uint8), seed=41 + hpk, with_imp=False)


# q8_2f at head_dim 128 runs on the tensor-core kernels, whose run partials are
# merged by one warp per query head (up to 16 slots per unit in one batch of
# loads, up to 32 in two) or by one CTA per query head beyond that.  With fewer
# tiles than resident workers every tile is its own run, so the longest
# sequence sets the slot count: 16 tiles (500 rows), 29 tiles (900 rows); the
# hd128 case above (1030 rows, 33 tiles) takes the CTA merge.
@pytest.mark.parametrize("hpk", [1, 3, 4, 8, 12, 16])
@pytest.mark.parametrize("longest", [500, 900])
def test_decode_q8_merge_paths(torch, kvd, hpk, longest):
    _decode_case(torch, kvd, oracle.Q8, 128, hpk, [0, 1, 64, 300, longest, 33],
                 np.array([1, 0, 1, 1], np.uint8), seed=31 + hpk + longest)


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("hpk", [2, 5, 8, 16])
def test_decode_parity_hd64(torch, kvd, mode, hpk):
    _decode_case(torch, kvd, MODES[mode], 64, hpk, [5, 257, 600], np.array([0, 1, 1], np.uint8),
                 seed=21 + hpk)


_OPTS = {
    "window": {"window": 75},
    "softcap": {"softcap": 1.5},
    "sinks": {"sinks": True},
    "all": {"window": 250, "softcap": 4.0, "sinks": True},
}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("hpk", [4, 8, 16])
@pytest.mark.parametrize("opt", list(_OPTS))
def test_decode_options_parity(torch, kvd, mode, hpk, opt):
    """[cortiq] attend_group_upto's window (first = stored - window), logit
    soft-capping and learned sinks, against the oracle: outputs, imp (rows
    before the window untouched), every storage mode, heads in N and in M."""
    opts = dict(_OPTS[opt])
    n_q = 4 * hpk
    if opts.pop("sinks", None):
        opts["sinks"] = (synthetic.normal((n_q,), 500 + hpk) * 2.0).astype(np.float32)
    _decode_case(torch, kvd, MODES[mode], 128, hpk, [0, 1, 64, 300, 777, 1030],
                 np.array([1, 1, 0, 1], np.uint8), seed=31 + hpk, opts=opts)


def test_decode_options_errors(torch, kvd):
    layer = _layer(kvd, oracle.Q8, [40], 2, 128, None, cap_extra=8)
    q = torch.zeros(1, 4, 128, device="cuda")
    for bad in ({"window": -1}, {"softcap": -1.0}, {"softcap": float("nan")}):
        with pytest.raises(kvd.KvdError):
            kvd.decode_attention(q, layer, **bad)
    with pytest.raises(ValueError):
        kvd.decode_attention(q, layer, sinks=torch.zeros(3, device="cuda"))


def test_tiny_f32_gqa_config(torch, kvd):
    """Tiny f32 GQA decode: 1 sequence, 4 Q / 2 KV heads, head_dim 64, 256 rows,
    K, V, q ~ N(0,1) from seed 0, scale 1/sqrt(64), output [4 x 64] plus imp[256]."""
    n_kv, hd, hpk, L = 2, 64, 2, 256
    k = synthetic.normal((L, n_kv, hd), 0)
    v = synthetic.normal((L, n_kv, hd), 1)
    q = synthetic.normal((1, n_kv * hpk, hd), 2)
    layer = kvd.LayerKvCache(1, n_kv, hd, "f32", L)
    kvd.kv_append(layer, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), [L])
    imp = torch.zeros(layer.imp_len, device="cuda")
    out = kvd.decode_attention(torch.from_numpy(q).cuda(), layer, imp=imp, scale=0.125)
    torch.cuda.synchronize()
    oc = oracle.OracleSeqCache(oracle.F32, n_kv, hd, L)
    oc.append_rows(k, v)
    imp_ref = np.zeros(L)
    ref = oc.decode(q[0], n_kv * hpk, np.float32(0.125), imp_ref)
    assert out_error(out.cpu().numpy()[0], ref) <= OUT_TOL
    got = imp.cpu().numpy()[:L]
    assert_imp_close(got, imp_ref)
    assert abs(got.sum() - n_kv * hpk) < 1e-3  # every head's weights sum to one


def test_bounded_wait_times_out_and_context_stays_usable(torch, kvd):
    """A wait that nothing satisfies gives up after its limit and reports it
    through the device error word (bit 0) -- no trap, no hang -- and the same
    context then decodes correctly with a clean word."""
    lengths = [300, 77]
    alive = np.array([1, 1], np.uint8)
    layer = _layer(kvd, MODES["q8"], lengths, 2, 128, alive, cap_extra=3)
    ks, vs = seq_rows(lengths, 2, 128, seed=5)
    gpu_append_bulk(layer, ks, vs, torch)
    assert layer.device_error() == 0
    layer.wait_timeout_selftest(2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert layer.device_error(clear=True) == 1  # bit 0: a bounded wait timed out
    assert layer.device_error() == 0
    with pytest.raises(kvd.KvdError):
        layer.wait_timeout_selftest(0)  # refused on the host, nothing launched
    _decode_case(torch, kvd, MODES["q8"], 128, 4, lengths, alive, seed=5)


@pytest.mark.parametrize("mode,hd", [("q8", 128), ("q8k", 128), ("q8v", 64), ("f32", 64)])
def test_metadata_guards_set_bit1_and_touch_nothing(torch, kvd, mode, hd):
    """The append, freeze and decode-split guards run on lengths one row past
    a capacity (kvd_bounds_selftest; q8 at head_dim 128 takes the tensor-core
    split, the others the CUDA-core one): the device error word reads bit 1
    alone, every storage byte and every length is unchanged, and the same
    context then decodes at parity with a clean word."""
    lengths = [100, 37]
    alive = np.array([1, 1], np.uint8)
    layer = _layer(kvd, MODES[mode], lengths, 2, hd, alive, cap_extra=3)
    ks, vs = seq_rows(lengths, 2, hd, seed=8)
    gpu_append_bulk(layer, ks, vs, torch)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    before = [b.clone() if b is not None else None for b in layer.bufs]
    scratch = layer.bounds_selftest()
    torch.cuda.synchronize()
    del scratch
    assert layer.device_error(clear=True) == 2  # bit 1 only: metadata out of range
    for a, b in zip(before, layer.bufs):
        if a is not None:
            assert torch.equal(a, b)
    assert [layer.seq_len(b) for b in range(2)] == lengths
    _decode_case(torch, kvd, MODES[mode], hd, 4, lengths, alive, seed=8)
    assert layer.device_error() == 0


def test_all_groups_dead_and_capacity_errors(torch, kvd):
    layer = kvd.LayerKvCache(2, 2, 128, "q8", [8, 8], alive=[0, 0])
    k = torch.randn(2, 2, 128, device="cuda")
    for _ in range(3):
        kvd.kv_append(layer, k, k)
    out = kvd.decode_attention(torch.randn(2, 4, 128, device="cuda"), layer)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    assert layer.memory_bytes() == 0 and layer.seq_len(0) == 3
    # capacity (8 rounds up to 16 rows): a bulk append that would overflow
    # sequence 1 changes nothing, not even sequence 0's length
    with pytest.raises(kvd.KvdError) as e:
        kvd.kv_append(layer, torch.randn(15, 2, 128, device="cuda"),
                      torch.randn(15, 2, 128, device="cuda"), [1, 14])
    assert e.value.status == -2
    assert layer.seq_len(0) == 3 and layer.seq_len(1) == 3
    with pytest.raises(kvd.KvdError):  # 3 query heads for 2 KV heads
        kvd.decode_attention(torch.randn(2, 3, 128, device="cuda"), layer)


# ------------------------------------------------------------------- R-SWA

def rope(x, pos, base=10000.0):
    hd = x.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    th = pos * base ** (-2.0 * i / hd)
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., 0::2].astype(np.float64), x[..., 1::2].astype(np.float64)
    out = np.empty(x.shape, np.float64)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out.astype(np.float32)


def test_rswa_ring_and_decode_parity(torch, kvd):
    """Three streams with different reference lengths (one empty); 300 decode steps
    wrap the ring (K rotated at the true absolute position by the harness); the
    device ring, its cursors and every decode step's output match the oracle."""
    B, H, hd, W, ref_cap = 3, 10, 128, 128, 1024
    prefill = [37, 0, 700]
    cache = kvd.RingCache(B, ref_cap, H, hd, W)
    o_ref_k = np.zeros((B, H, ref_cap, hd), np.float32)
    o_ref_v = np.zeros_like(o_ref_k)
    o_ring_k = np.zeros((B, H, W, hd), np.float32)
    o_ring_v = np.zeros_like(o_ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(B)]
    for s in range(B):
        m = prefill[s]
        k = np.stack([rope(synthetic.normal((H, hd), 100 * s + r), r) for r in range(m)], axis=1) \
            if m else np.zeros((H, 0, hd), np.float32)
        v = synthetic.normal((H, m, hd), 100 * s + 99)
        kvd.rswa_record_prefill(cache, s, torch.from_numpy(np.ascontiguousarray(k)).cuda(),
                                torch.from_numpy(v).cuda())
        o_ref_k[s, :, :m] = k
        o_ref_v[s, :, :m] = v
    scale = np.float32(1.0 / math.sqrt(hd))
    worst = 0.0
    for t in range(300):
        kt = np.stack([rope(synthetic.normal((H, hd), 5000 + 7 * t + s), prefill[s] + t) for s in range(B)])
        vt = synthetic.normal((B, H, hd), 9000 + t)
        qt = np.stack([rope(synthetic.normal((H, hd), 13000 + 7 * t + s), prefill[s] + t) for s in range(B)])
        slots = kvd.rswa_ring_write(cache, torch.from_numpy(kt).cuda(), torch.from_numpy(vt).cuda())
        for s in range(B):
            assert slots[s] == oracle.rswa_write(o_ring_k[s], o_ring_v[s], kt[s], vt[s], True, cursors[s])
            assert cache.ring_len[s] == cursors[s][0] and cache.ring_pos[s] == cursors[s][1]
        if t in (0, 1, 127, 128, 200, 299):
            out = kvd.rswa_decode(torch.from_numpy(qt).cuda(), cache).cpu().numpy()
            for s in range(B):
                ref = oracle.rswa_decode(qt[s], o_ref_k[s], o_ref_v[s], prefill[s], o_ring_k[s],
                                         o_ring_v[s], cursors[s][0], scale)
                err = out_error(out[s].reshape(H, hd), ref)
                worst = max(worst, err)
                assert err <= OUT_TOL, (t, s, err)
    assert cursors[0].tolist() == [128, 300 % 128]
    assert np.array_equal(cache.ring_k.cpu().numpy(), o_ring_k)
    assert np.array_equal(cache.ring_v.cpu().numpy(), o_ring_v)
    assert cache.device_error() == 0


def test_rswa_page_closed_form_on_gpu(torch, kvd):
    """rswa attention_entry_writes_then_attends: out = (e^{10/sqrt(128)} 5 + 1) /
    (e^{10/sqrt(128)} + 1) ~ 3.831 for every element."""
    H, hd = 10, 128
    cache = kvd.RingCache(1, 16, H, hd, 128)
    k = torch.zeros(H, 1, hd, device="cuda")
    k[:, :, 1] = 1.0
    kvd.rswa_record_prefill(cache, 0, k, torch.ones(H, 1, hd, device="cuda"))
    q = torch.zeros(1, H, hd, device="cuda")
    q[..., 0] = 10.0
    kt = torch.zeros(1, H, hd, device="cuda")
    kt[..., 0] = 1.0
    out = kvd.rswa_attention(cache, q, kt, torch.full((1, H, hd), 5.0, device="cuda"))
    w = math.exp(10.0 / math.sqrt(128.0))
    assert torch.allclose(out, torch.full_like(out, (w * 5 + 1) / (w + 1)), atol=1e-4)
    assert cache.ring_len[0] == 1


def test_rswa_errors_do_not_mutate(torch, kvd):
    cache = kvd.RingCache(2, 32, 10, 128, 128)
    t = torch.ones(2, 10, 128, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.rswa_ring_write(cache, t, t)
    assert e.value.status == -3
    assert cache.ring_len.tolist() == [0, 0] and cache.ring_pos.tolist() == [0, 0]
    with pytest.raises(kvd.KvdError) as e:
        kvd.rswa_decode(t, cache)
    assert e.value.status == -3
    kvd.rswa_record_prefill(cache, 0, torch.ones(10, 4, 128, device="cuda"),
                            torch.ones(10, 4, 128, device="cuda"))
    kvd.rswa_record_prefill(cache, 1, torch.ones(10, 0, 128, device="cuda"),
                            torch.ones(10, 0, 128, device="cuda"))
    with pytest.raises(kvd.KvdError) as e:  # stream 1 has no keys at all
        kvd.rswa_decode(t, cache)
    assert e.value.status == -4
    with pytest.raises(kvd.KvdError) as e:
        kvd.rswa_record_prefill(cache, 0, torch.ones(10, 40, 128, device="cuda"),
                                torch.ones(10, 40, 128, device="cuda"))
    assert e.value.status == -2 and cache.prefill_len.tolist() == [4, 0]


# ------------------------------------------------- R-SWA int8 mirror (NEXT-2)

def _mirror_of(ref_k, ref_v, ring_k, ring_v):
    rk8, rks = oracle.rswa_mirror(ref_k)
    rv8, rvs = oracle.rswa_mirror(ref_v)
    gk8, gks = oracle.rswa_mirror(ring_k)
    gv8, gvs = oracle.rswa_mirror(ring_v)
    return rk8, rks, rv8, rvs, gk8, gks, gv8, gvs


@pytest.mark.parametrize("hd,H", [(128, 10), (64, 4)])
def test_rswa_i8_mirror_and_decode_parity(torch, kvd, hd, H):
    """Three streams (reference 37, 0 and 700 rows), 150 decode steps that wrap
    the ring: the int8 mirror (codes and row scales) is bit-exact with the
    oracle's quantize_row_i8 of the f32 rows, the f32 regions are still written,
    and decode_attention_int8 outputs match the oracle at several steps."""
    B, W, ref_cap = 3, 128, 1024
    prefill = [37, 0, 700]
    cache = kvd.RingCache(B, ref_cap, H, hd, W, int8=True)
    o_ref_k = np.zeros((B, H, ref_cap, hd), np.float32)
    o_ref_v = np.zeros_like(o_ref_k)
    o_ring_k = np.zeros((B, H, W, hd), np.float32)
    o_ring_v = np.zeros_like(o_ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(B)]
    for s in range(B):
        m = prefill[s]
        k = synthetic.normal((H, m, hd), 300 * s + 1)
        v = synthetic.normal((H, m, hd), 300 * s + 2) * np.float32(3.0)
        kvd.rswa_record_prefill(cache, s, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        o_ref_k[s, :, :m] = k
        o_ref_v[s, :, :m] = v
        if m:
            ck, sk = oracle.rswa_mirror(k)
            cv, sv = oracle.rswa_mirror(v)
            assert np.array_equal(cache.ref_k8[s, :, :m].cpu().numpy(), ck)
            assert np.array_equal(cache.ref_ks[s, :, :m].cpu().numpy().view(np.uint32), sk.view(np.uint32))
            assert np.array_equal(cache.ref_v8[s, :, :m].cpu().numpy(), cv)
            assert np.array_equal(cache.ref_vs[s, :, :m].cpu().numpy().view(np.uint32), sv.view(np.uint32))
    assert np.array_equal(cache.ref_k.cpu().numpy(), o_ref_k)
    scale = np.float32(1.0 / math.sqrt(hd))
    for t in range(150):
        kt = synthetic.normal((B, H, hd), 7000 + t)
        vt = synthetic.normal((B, H, hd), 8000 + t)
        qt = synthetic.normal((B, H, hd), 9000 + t)
        slots = kvd.rswa_ring_write(cache, torch.from_numpy(kt).cuda(), torch.from_numpy(vt).cuda())
        for s in range(B):
            assert slots[s] == oracle.rswa_write(o_ring_k[s], o_ring_v[s], kt[s], vt[s], True, cursors[s])
            assert cache.ring_len[s] == cursors[s][0] and cache.ring_pos[s] == cursors[s][1]
        if t in (0, 1, 127, 128, 149):
            out = kvd.rswa_decode_i8(torch.from_numpy(qt).cuda(), cache).cpu().numpy()
            for s in range(B):
                mir = _mirror_of(o_ref_k[s], o_ref_v[s], o_ring_k[s], o_ring_v[s])
                ref = oracle.rswa_decode_i8(qt[s], mir[0], mir[1], mir[2], mir[3], prefill[s], mir[4],
                                            mir[5], mir[6], mir[7], cursors[s][0], scale)
                err = out_error(out[s].reshape(H, hd), ref)
                assert err <= OUT_TOL, (t, s, err)
    assert np.array_equal(cache.ring_k.cpu().numpy(), o_ring_k)
    assert np.array_equal(cache.ring_v.cpu().numpy(), o_ring_v)
    gk8, gks = oracle.rswa_mirror(o_ring_k)
    gv8, gvs = oracle.rswa_mirror(o_ring_v)
    assert np.array_equal(cache.ring_k8.cpu().numpy(), gk8)
    assert np.array_equal(cache.ring_v8.cpu().numpy(), gv8)
    assert np.array_equal(cache.ring_ks.cpu().numpy().view(np.uint32), gks.view(np.uint32))
    assert np.array_equal(cache.ring_vs.cpu().numpy().view(np.uint32), gvs.view(np.uint32))
    assert cache.device_error() == 0


def _bits(b):
    return np.frombuffer(np.uint32(b).tobytes(), np.float32)[0]


def test_rswa_i8_quantiser_edge_rows_on_gpu(torch, kvd):
    """The page's worked rows through the device quantiser: ties to even, the
    division-not-reciprocal fixture, an all-zero row (scale 1.0), and rows whose
    magnitude sweeps 2^-20 .. 2^20 (the page's LCG contract) are bit-exact with
    the oracle and the printed codes."""
    from conftest import load_golden

    H, hd = 10, 128
    ties = load_golden("quant_ties_to_even.txt")
    div = load_golden("quant_division.txt")
    rows = np.zeros((H, 48, hd), np.float32)
    rows[0, 0, :9] = [float(x) for x in ties["row_head"].split()]
    rows[0, 1, 0], rows[0, 1, 1] = _bits(int(div["x0_bits"], 16)), _bits(int(div["x1_bits"], 16))
    state = 0xD1B54A32D192ED03
    for i in range(2, 43):
        mag = np.float32(2.0) ** np.float32(i - 2 - 20)
        for d in range(hd):
            state = (state * 6364136223846793005 + 1442695040888963407) & (2 ** 64 - 1)
            unit = np.float32((state >> 40) & 0xFFFFFFFF) / np.float32((1 << 24) - 1)
            rows[1 + i % (H - 1), i, d] = (unit * np.float32(2.0) - np.float32(1.0)) * mag
    cache = kvd.RingCache(1, 48, H, hd, 128, int8=True)
    t = torch.from_numpy(rows).cuda()
    kvd.rswa_record_prefill(cache, 0, t, t)
    codes = cache.ref_k8[0].cpu().numpy()
    scales = cache.ref_ks[0].cpu().numpy()
    assert codes[0, 0, :9].tolist() == [int(x) for x in ties["codes_head"].split()]
    assert scales[0, 0].view(np.uint32) == int(ties["scale_bits"], 16)
    assert codes[0, 1, :2].tolist() == [int(x) for x in div["codes"].split()]
    assert scales[0, 47] == np.float32(1.0) and not codes[0, 47].any()  # an all-zero row
    ck, sk = oracle.rswa_mirror(rows)
    assert np.array_equal(codes, ck)
    assert np.array_equal(scales.view(np.uint32), sk.view(np.uint32))
    assert np.array_equal(cache.ref_v8[0].cpu().numpy(), ck)


def test_rswa_i8_errors(torch, kvd):
    plain = kvd.RingCache(1, 32, 10, 128, 128)
    t = torch.ones(1, 10, 128, device="cuda")
    with pytest.raises(ValueError):
        kvd.rswa_decode_i8(t, plain)
    cache = kvd.RingCache(2, 32, 10, 128, 128, int8=True)
    t2 = torch.ones(2, 10, 128, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.rswa_decode_i8(t2, cache)
    assert e.value.status == -3
    with pytest.raises(kvd.KvdError) as e:
        kvd.rswa_ring_write(cache, t2, t2)
    assert e.value.status == -3 and cache.ring_len.tolist() == [0, 0]
    kvd.rswa_record_prefill(cache, 0, torch.ones(10, 4, 128, device="cuda"),
                            torch.ones(10, 4, 128, device="cuda"))
    kvd.rswa_record_prefill(cache, 1, torch.ones(10, 0, 128, device="cuda"),
                            torch.ones(10, 0, 128, device="cuda"))
    with pytest.raises(kvd.KvdError) as e:  # stream 1 has no keys at all
        kvd.rswa_decode_i8(t2, cache)
    assert e.value.status == -4
    # the mirror writers take head_dim 64 or 128 only, and a mirror is required
    import ctypes as C

    lib = kvd.lib()
    x = torch.ones(10, 4, 96, device="cuda")
    pl, rl, rp = (np.array(a, np.int32) for a in (cache.prefill_len, cache.ring_len, cache.ring_pos))
    args = (C.c_void_p(x.data_ptr()), C.c_void_p(x.data_ptr()), 0, 4, 2, 10, 96, 32, 128,
            pl.ctypes.data_as(C.c_void_p), rl.ctypes.data_as(C.c_void_p), rp.ctypes.data_as(C.c_void_p), None,
            None)
    ref = (C.c_void_p(cache.ref_k.data_ptr()), C.c_void_p(cache.ref_v.data_ptr()))
    assert lib.rswa_record_prefill_i8(*ref, C.byref(cache.mirror), *args) == -1
    assert lib.rswa_record_prefill_i8(*ref, None, *args) == -1
    assert pl.tolist() == [4, 0]


# --------------------------------------------------- Born eviction (NEXT-3)

def _mass(lengths, imp_base, imp_len, seed):
    """Seeded masses with many exact ties (small integers / 8), the same array
    for the device buffer and every oracle sequence."""
    rng = np.random.default_rng(seed)
    full = np.zeros(imp_len, np.float32)
    per = []
    for b, L in enumerate(lengths):
        m = (rng.integers(0, 12, size=int(L)) / 8.0).astype(np.float32)
        full[imp_base[b]:imp_base[b] + int(L)] = m
        per.append(m)
    return full, per


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("hd", [128, 64])
@pytest.mark.parametrize("recent", [60, 146])
def test_born_eviction_parity(torch, kvd, mode, hd, recent):
    """Sequences above, at and below the budget, a dead head, many tied masses:
    after kv_evict_born every storage, imp and the lengths equal the oracle's
    evict_born bit for bit; decode over the evicted cache and over rows appended
    afterwards matches the oracle.  recent 146 leaves no middle budget: the long
    sequences keep their sinks and last rows, whose sources all lie past the
    kept range (the gather copies them directly), while the 151-row one moves
    through the workspace copy."""
    lengths = [700, 150, 151, 40, 2300]
    n_kv, alive, extra = 4, [1, 1, 0, 1], 40
    keep, sink = 150, 4
    ks, vs = seq_rows(lengths, n_kv, hd, seed=61)
    layer = _layer(kvd, MODES[mode], lengths, n_kv, hd, alive, cap_extra=extra)
    gpu_append_bulk(layer, ks, vs, torch, pieces=(0.5, 1.0))
    ocs = oracle_caches(MODES[mode], lengths, n_kv, hd, alive, ks, vs, cap=max(lengths) + extra)
    for oc in ocs:
        oc.freeze_if_due()
    full, per = _mass(lengths, layer.imp_base, layer.imp_len, seed=62)
    imp = torch.from_numpy(full.copy()).cuda()
    kvd.kv_evict_born(layer, imp, keep, sink, recent)
    got_imp = imp.cpu().numpy()
    o_imps = []
    for b, oc in enumerate(ocs):
        o_imp = np.zeros(oc.cap, np.float32)
        o_imp[:lengths[b]] = per[b]
        assert oc.evict_born(keep, sink, recent, o_imp) == min(lengths[b], keep)
        n_old = lengths[b]
        # kept masses gathered, the dropped rows' entries cleared
        assert np.array_equal(got_imp[layer.imp_base[b]:layer.imp_base[b] + n_old].view(np.uint32),
                              o_imp[:n_old].view(np.uint32)), b
        o_imps.append(o_imp.astype(np.float64))
    assert_storage_bitexact(layer, ocs, torch)
    assert layer.device_error() == 0
    n_q = n_kv * 2
    scale = np.float32(1.0 / math.sqrt(hd))
    for step in range(2):
        q = synthetic.normal((len(lengths), n_q, hd), 63 + step)
        out = kvd.decode_attention(torch.from_numpy(q).cuda(), layer, imp=imp, scale=float(scale)).cpu().numpy()
        for b, oc in enumerate(ocs):
            ref = oc.decode(q[b], n_q, scale, o_imps[b])
            live = np.repeat(np.array(alive, bool), 2)
            assert out_error(out[b], ref, live) <= OUT_TOL, (step, b)
        # rows appended after the eviction land behind the kept rows
        k_new = synthetic.normal((len(lengths), n_kv, hd), 64 + step)
        v_new = synthetic.normal((len(lengths), n_kv, hd), 65 + step)
        kvd.kv_append(layer, torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda())
        for b, oc in enumerate(ocs):
            oc.append(k_new[b], v_new[b])
            oc.freeze_if_due()
    assert_storage_bitexact(layer, ocs, torch)
    got_imp = imp.cpu().numpy()
    for b, oc in enumerate(ocs):  # masses accumulated after the eviction, on the kept and new rows
        assert_imp_close(got_imp[layer.imp_base[b]:layer.imp_base[b] + oc.seq_len], o_imps[b][:oc.seq_len])


def test_born_page_example_on_gpu(torch, kvd):
    """cortiq born_eviction_keeps_high_mass_position: kept keys 0, 3, 6, 7."""
    from conftest import load_golden

    g = load_golden("born_eviction.txt")
    hd = 64
    layer = _layer(kvd, MODES["f32"], [8], 1, hd, [1], cap_extra=8)
    k = np.repeat(np.arange(8, dtype=np.float32)[:, None, None], hd, axis=2)
    kvd.kv_append(layer, torch.from_numpy(k).cuda(), torch.from_numpy(k + 100).cuda(), np.array([8], np.int32))
    imp = torch.full((layer.imp_len,), float(g["light_mass"]), device="cuda")
    imp[int(g["heavy_position"])] = float(g["heavy_mass"])
    kvd.kv_evict_born(layer, imp, int(g["keep_last"]), sink=int(g["sink"]))  # recent = max(4 // 2, 1)
    keys = layer.component(kvd._abi.BUF_K)[:4, 0].cpu().numpy().tolist()
    assert keys == [float(x) for x in g["kept_keys"].split()]
    assert layer.seq_len(0) == 4 and layer.device_error() == 0


def test_born_edges_and_errors(torch, kvd):
    """keep_last 0 empties a sequence (fields stay frozen), a budget at or above
    every length is a no-op, sink >= keep_last keeps the first rows, and a
    negative argument is refused before anything changes."""
    lengths = [90, 30]
    ks, vs = seq_rows(lengths, 2, 128, seed=71)
    layer = _layer(kvd, MODES["q8"], lengths, 2, 128, None, cap_extra=16)
    gpu_append_bulk(layer, ks, vs, torch)
    ocs = oracle_caches(MODES["q8"], lengths, 2, 128, None, ks, vs, cap=106)
    for oc in ocs:
        oc.freeze_if_due()
    imp = torch.zeros(layer.imp_len, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.kv_evict_born(layer, imp, 10, sink=-1, recent=2)
    assert e.value.status == -1 and layer.seq_len(0) == 90
    kvd.kv_evict_born(layer, imp, 100, 4, 8)  # nobody above the budget
    assert_storage_bitexact(layer, ocs, torch)
    kvd.kv_evict_born(layer, imp, 50, 60, 8)  # sinks take the whole budget
    for b, oc in enumerate(ocs):
        o_imp = np.zeros(oc.cap, np.float32)
        oc.evict_born(50, 60, 8, o_imp)
    assert layer.seq_len(0) == 50 and layer.seq_len(1) == 30
    assert_storage_bitexact(layer, ocs, torch)
    kvd.kv_evict_born(layer, imp, 0, 4, 8)
    assert layer.seq_len(0) == 0 and layer.seq_len(1) == 0 and layer.frozen(0)
    assert layer.device_error() == 0


# ------------------------------- truncate_last and ring rollback (NEXT-4)

@pytest.mark.parametrize("mode", list(MODES))
def test_truncate_last_parity(torch, kvd, mode):
    """cortiq truncate_last per sequence (0, 3, more than stored, 70 rows: below
    the freeze point of a frozen sequence): lengths and storages match the
    oracle, imp of the dropped rows is cleared, and rows appended afterwards
    (quantised against the kept fields) decode like the oracle's."""
    lengths = [90, 200, 30, 150]
    n_kv, hd = 2, 128
    ks, vs = seq_rows(lengths, n_kv, hd, seed=81)
    layer = _layer(kvd, MODES[mode], lengths, n_kv, hd, None, cap_extra=8)
    gpu_append_bulk(layer, ks, vs, torch)
    ocs = oracle_caches(MODES[mode], lengths, n_kv, hd, None, ks, vs, cap=max(lengths) + 8)
    for oc in ocs:
        oc.freeze_if_due()
    rng = np.random.default_rng(82)
    full = rng.random(layer.imp_len).astype(np.float32)
    imp = torch.from_numpy(full.copy()).cuda()
    drop = np.array([0, 3, 100, 70], np.int32)
    kvd.kv_truncate_last(layer, drop, imp)
    got = imp.cpu().numpy()
    o_imps = []
    for b, oc in enumerate(ocs):
        o_imp = full[layer.imp_base[b]:layer.imp_base[b] + oc.cap].copy()
        oc.truncate_last(int(drop[b]), o_imp)
        n_old = lengths[b]
        assert np.array_equal(got[layer.imp_base[b]:layer.imp_base[b] + n_old], o_imp[:n_old]), b
        o_imps.append(o_imp.astype(np.float64))
    assert [layer.seq_len(b) for b in range(4)] == [90, 197, 0, 80]
    assert_storage_bitexact(layer, ocs, torch)
    k_new = synthetic.normal((4, n_kv, hd), 83)
    v_new = synthetic.normal((4, n_kv, hd), 84)
    kvd.kv_append(layer, torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda())
    for b, oc in enumerate(ocs):
        oc.append(k_new[b], v_new[b])
        oc.freeze_if_due()
    assert_storage_bitexact(layer, ocs, torch)
    n_q = 4
    q = synthetic.normal((4, n_q, hd), 85)
    scale = np.float32(1.0 / math.sqrt(hd))
    out = kvd.decode_attention(torch.from_numpy(q).cuda(), layer, imp=imp, scale=float(scale)).cpu().numpy()
    got = imp.cpu().numpy()
    for b, oc in enumerate(ocs):
        ref = oc.decode(q[b], n_q, scale, o_imps[b])
        assert out_error(out[b], ref) <= OUT_TOL, b
        assert_imp_close(got[layer.imp_base[b]:layer.imp_base[b] + oc.seq_len], o_imps[b][:oc.seq_len])
    assert layer.device_error() == 0


@pytest.mark.parametrize("int8", [False, True])
def test_rswa_rollback_erases_speculative_steps(torch, kvd, int8):
    """rswa checkpoint -> three draft writes -> rollback: the decode after the
    rollback is bit-identical to the decode before the drafts, and the steps
    written afterwards match a cache that never saw the drafts."""
    B, H, hd, W, ref_cap = 2, 10, 128, 128, 64
    mk = lambda: kvd.RingCache(B, ref_cap, H, hd, W, int8=int8)
    spec, plain = mk(), mk()
    dec = kvd.rswa_decode_i8 if int8 else kvd.rswa_decode
    for c in (spec, plain):
        for s in range(B):
            k = synthetic.normal((H, 40, hd), 90 + s)
            kvd.rswa_record_prefill(c, s, torch.from_numpy(k).cuda(), torch.from_numpy(k * 0.5).cuda())
    steps = [(synthetic.normal((B, H, hd), 100 + t), synthetic.normal((B, H, hd), 200 + t)) for t in range(6)]
    q = torch.from_numpy(synthetic.normal((B, H, hd), 300)).cuda()
    for t in range(2):
        for c in (spec, plain):
            kvd.rswa_ring_write(c, torch.from_numpy(steps[t][0]).cuda(), torch.from_numpy(steps[t][1]).cuda())
    before = dec(q, spec).cpu().numpy()
    cps = [spec.checkpoint(s) for s in range(B)]
    for t in range(3):  # drafts
        d = synthetic.normal((B, H, hd), 400 + t)
        kvd.rswa_ring_write(spec, torch.from_numpy(d).cuda(), torch.from_numpy(d).cuda())
    assert not np.array_equal(dec(q, spec).cpu().numpy(), before)
    for s in range(B):
        spec.rollback_to(s, cps[s])
    assert spec.ring_len.tolist() == [2, 2] and spec.ring_pos.tolist() == [2, 2]
    assert np.array_equal(dec(q, spec).cpu().numpy(), before)
    with pytest.raises(kvd.KvdError) as e:  # the abandoned branch cannot be replayed
        spec.rollback_to(0, cps[0])
    assert e.value.status == -3
    for t in range(2, 6):
        for c in (spec, plain):
            kvd.rswa_ring_write(c, torch.from_numpy(steps[t][0]).cuda(), torch.from_numpy(steps[t][1]).cuda())
    assert np.array_equal(dec(q, spec).cpu().numpy(), dec(q, plain).cpu().numpy())
    assert spec.device_error() == 0


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("hd,hg,K", [(128, 4, 4), (64, 2, 3), (128, 16, 1), (128, 1, 8)])
def test_verify_parity(torch, kvd, mode, hd, hg, K):
    """Query-batched verify of K drafts (appended by kv_append, then verified in
    one call; causal among them) against the oracle, plain and with window +
    softcap + sinks, over sequences shorter than K, around a tile edge and long
    enough for several chunks; a dead group gives zeros.  Rejecting the last
    drafts with kv_truncate_last then leaves a cache that decodes like the
    oracle's."""
    n_kv = 3
    n_q = hg * n_kv
    lengths = [2, 40, 1200, 3000]
    alive = [1, 0, 1]
    ks, vs = seq_rows([L - K if L >= K else 0 for L in lengths], n_kv, hd, seed=91)
    layer = _layer(kvd, MODES[mode], lengths, n_kv, hd, alive, cap_extra=8)
    pre = [k.shape[0] for k in ks]
    if max(pre) > 0:
        gpu_append_bulk(layer, ks, vs, torch)
    ocs = oracle_caches(MODES[mode], pre, n_kv, hd, alive, ks, vs, cap=max(lengths) + 8)
    for oc in ocs:
        oc.freeze_if_due()
    dk, dv = seq_rows([L - p for L, p in zip(lengths, pre)], n_kv, hd, seed=92)
    nn = np.array([d.shape[0] for d in dk], np.int32)
    kvd.kv_append(layer, torch.from_numpy(np.concatenate(dk)).cuda(), torch.from_numpy(np.concatenate(dv)).cuda(), nn)
    for b, oc in enumerate(ocs):
        for i in range(nn[b]):  # the oracle appends one row at a time
            oc.append(dk[b][i], dv[b][i])
            oc.freeze_if_due()
    assert_storage_bitexact(layer, ocs, torch)
    q = synthetic.normal((len(lengths), K, n_q, hd), 93)
    sinks = synthetic.normal((n_q,), 94)
    scale = np.float32(1.0 / math.sqrt(hd))
    live = np.repeat(np.array(alive, bool), hg)
    for opts in ({}, {"window": 700, "softcap": 3.0, "sinks": sinks}):
        kw = dict(opts)
        if "sinks" in kw:
            kw["sinks"] = torch.from_numpy(kw["sinks"]).cuda()
        out = kvd.decode_attention_verify(torch.from_numpy(q).cuda(), layer, K, scale=float(scale), **kw)
        out = out.cpu().numpy()
        for b, oc in enumerate(ocs):
            ref = oc.decode_verify(q[b], n_q, K, scale, opts.get("window", 0), opts.get("softcap", 0.0),
                                   opts.get("sinks"))
            for k in range(K):
                if not np.any(ref[k][live]):  # no visible row: zeros
                    assert not out[b, k].any(), (b, k)
                    continue
                assert out_error(out[b, k], ref[k], live) <= OUT_TOL, (opts.keys(), b, k)
            assert not out[b][:, ~live].any()
    assert layer.device_error() == 0
    # reject the last two drafts everywhere
    drop = min(2, K)
    kvd.kv_truncate_last(layer, drop)
    for oc in ocs:
        oc.truncate_last(drop)
    q1 = synthetic.normal((len(lengths), n_q, hd), 95)
    out = kvd.decode_attention(torch.from_numpy(q1).cuda(), layer, scale=float(scale)).cpu().numpy()
    for b, oc in enumerate(ocs):
        if oc.seq_len:
            assert out_error(out[b], oc.decode(q1[b], n_q, scale), live) <= OUT_TOL, b


def test_verify_errors(torch, kvd):
    layer = _layer(kvd, MODES["q8"], [100], 2, 128, None)
    q = torch.zeros(1, 4, 8, 128, device="cuda")  # hg 4 x K 4 = 16 query rows per group
    kvd.decode_attention_verify(q, layer, 4)
    with pytest.raises(kvd.KvdError) as e:  # 4 heads per group x 5 drafts > 16
        kvd.decode_attention_verify(torch.zeros(1, 5, 8, 128, device="cuda"), layer, 5)
    assert e.value.status == -1
    with pytest.raises(kvd.KvdError) as e:
        kvd.decode_attention_verify(q, layer, 4, window=-1)
    assert e.value.status == -1


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("hd,H", [(128, 10), (64, 3)])
def test_rswa_verify_parity(torch, kvd, int8, hd, H):
    """rswa verify_attention, query-batched over K = 5, 16 and 1 drafts, against the
    oracle's write-then-decode on a private ring copy: streams with a long, a
    short and no reference block, full rings (each draft evicts the oldest
    row); the device cache and cursors stay as they were."""
    B, W, ref_cap = 3, 128, 1024
    prefill = [700, 30, 0]
    cache = kvd.RingCache(B, ref_cap, H, hd, W, int8=int8)
    o_ref_k = np.zeros((B, H, ref_cap, hd), np.float32)
    o_ref_v = np.zeros_like(o_ref_k)
    o_ring_k = np.zeros((B, H, W, hd), np.float32)
    o_ring_v = np.zeros_like(o_ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(B)]
    for s in range(B):
        m = prefill[s]
        k = synthetic.normal((H, m, hd), 500 + s)
        v = synthetic.normal((H, m, hd), 510 + s)
        kvd.rswa_record_prefill(cache, s, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        o_ref_k[s, :, :m], o_ref_v[s, :, :m] = k, v
    for t in range(140):
        kt = synthetic.normal((B, H, hd), 600 + t)
        vt = synthetic.normal((B, H, hd), 700 + t)
        kvd.rswa_ring_write(cache, torch.from_numpy(kt).cuda(), torch.from_numpy(vt).cuda())
        for s in range(B):
            oracle.rswa_write(o_ring_k[s], o_ring_v[s], kt[s], vt[s], True, cursors[s])
    scale = np.float32(1.0 / math.sqrt(hd))
    for K in (5, 16, 1):
        q = synthetic.normal((B, K, H, hd), 800 + K)
        dk = synthetic.normal((B, K, H, hd), 810 + K)
        dv = synthetic.normal((B, K, H, hd), 820 + K)
        snap = (cache.ring_len.copy(), cache.ring_pos.copy(), cache.ring_k.clone())
        out = kvd.rswa_verify(torch.from_numpy(q).cuda(), torch.from_numpy(dk).cuda(), torch.from_numpy(dv).cuda(),
                              cache, int8=int8).cpu().numpy()
        assert np.array_equal(cache.ring_len, snap[0]) and np.array_equal(cache.ring_pos, snap[1])
        assert torch.equal(cache.ring_k, snap[2])
        for s in range(B):
            ref = oracle.rswa_verify(q[s], dk[s], dv[s], o_ref_k[s], o_ref_v[s], prefill[s], o_ring_k[s],
                                     o_ring_v[s], cursors[s], scale, int8=int8)
            for i in range(K):
                err = out_error(out[s, i].reshape(H, hd), ref[i])
                assert err <= OUT_TOL, (K, s, i, err)
    assert cache.device_error() == 0


@pytest.mark.parametrize("K,ref_cap", [(4, 6144), (8, 6144), (2, 6144), (3, 2096)])
def test_rswa_i8_verify_reference_runs(torch, kvd, K, ref_cap):
    """The int8 mirror's verify with long reference blocks: at head_dim 128 with
    up to 8 drafts and a block of whole 32-row tiles the block runs on the
    tensor-core kernel (many tiles per head, several workers and partial runs
    per head, a ragged last tile, a stream without a block); ref_cap 2096 (not
    a whole number of tiles) keeps the CUDA-core kernel.  Against the oracle's
    write-then-decode over the mirror."""
    B, H, hd, W = 3, 3, 128, 128
    prefill = [ref_cap - 144, 2077, 0]
    cache = kvd.RingCache(B, ref_cap, H, hd, W, int8=True)
    o_ref_k = np.zeros((B, H, ref_cap, hd), np.float32)
    o_ref_v = np.zeros_like(o_ref_k)
    o_ring_k = np.zeros((B, H, W, hd), np.float32)
    o_ring_v = np.zeros_like(o_ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(B)]
    for s in range(B):
        m = prefill[s]
        k = synthetic.normal((H, m, hd), 5500 + s)
        v = synthetic.normal((H, m, hd), 5510 + s)
        kvd.rswa_record_prefill(cache, s, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        o_ref_k[s, :, :m], o_ref_v[s, :, :m] = k, v
    for t in range(90):
        kt = synthetic.normal((B, H, hd), 5600 + t)
        vt = synthetic.normal((B, H, hd), 5700 + t)
        kvd.rswa_ring_write(cache, torch.from_numpy(kt).cuda(), torch.from_numpy(vt).cuda())
        for s in range(B):
            oracle.rswa_write(o_ring_k[s], o_ring_v[s], kt[s], vt[s], True, cursors[s])
    scale = np.float32(1.0 / math.sqrt(hd))
    q = synthetic.normal((B, K, H, hd), 5800 + K)
    dk = synthetic.normal((B, K, H, hd), 5810 + K)
    dv = synthetic.normal((B, K, H, hd), 5820 + K)
    out = kvd.rswa_verify(torch.from_numpy(q).cuda(), torch.from_numpy(dk).cuda(), torch.from_numpy(dv).cuda(),
                          cache, int8=True).cpu().numpy()
    assert cache.device_error() == 0
    for s in range(B):
        ref = oracle.rswa_verify(q[s], dk[s], dv[s], o_ref_k[s], o_ref_v[s], prefill[s], o_ring_k[s],
                                 o_ring_v[s], cursors[s], scale, int8=True)
        for i in range(K):
            err = out_error(out[s, i].reshape(H, hd), ref[i])
            assert err <= OUT_TOL, (s, i, err)


def test_rswa_i8_verify_more_streams_than_one_launch(torch, kvd):
    """260 streams: the tensor-core route of the int8 verify runs in two launch
    slices (256 + 4 streams) that reuse the workspace's stream tables, unit
    slot ranges and run partials; blocks of 0..96 rows (ragged tiles, empty
    blocks), rings filling and full."""
    B, H, hd, W, ref_cap, K = 260, 2, 128, 16, 96, 3
    prefill = [(37 * s) % (ref_cap + 1) for s in range(B)]
    cache = kvd.RingCache(B, ref_cap, H, hd, W, int8=True)
    o_ref_k = np.zeros((B, H, ref_cap, hd), np.float32)
    o_ref_v = np.zeros_like(o_ref_k)
    k = synthetic.normal((B, H, ref_cap, hd), 6100)
    v = synthetic.normal((B, H, ref_cap, hd), 6101)
    for s in range(B):
        m = prefill[s]
        kvd.rswa_record_prefill(cache, s, torch.from_numpy(np.ascontiguousarray(k[s, :, :m])).cuda(),
                                torch.from_numpy(np.ascontiguousarray(v[s, :, :m])).cuda())
        o_ref_k[s, :, :m], o_ref_v[s, :, :m] = k[s, :, :m], v[s, :, :m]
    o_ring_k = np.zeros((B, H, W, hd), np.float32)
    o_ring_v = np.zeros_like(o_ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(B)]
    for t in range(20):
        kt = synthetic.normal((B, H, hd), 6200 + t)
        vt = synthetic.normal((B, H, hd), 6300 + t)
        kvd.rswa_ring_write(cache, torch.from_numpy(kt).cuda(), torch.from_numpy(vt).cuda())
        for s in range(B):
            oracle.rswa_write(o_ring_k[s], o_ring_v[s], kt[s], vt[s], True, cursors[s])
    scale = np.float32(1.0 / math.sqrt(hd))
    q = synthetic.normal((B, K, H, hd), 6400)
    dk = synthetic.normal((B, K, H, hd), 6401)
    dv = synthetic.normal((B, K, H, hd), 6402)
    out = kvd.rswa_verify(torch.from_numpy(q).cuda(), torch.from_numpy(dk).cuda(), torch.from_numpy(dv).cuda(),
                          cache, int8=True).cpu().numpy()
    assert cache.device_error() == 0
    for s in list(range(0, B, 7)) + [255, 256, 257, 258, 259]:
        ref = oracle.rswa_verify(q[s], dk[s], dv[s], o_ref_k[s], o_ref_v[s], prefill[s], o_ring_k[s],
                                 o_ring_v[s], cursors[s], scale, int8=True)
        for i in range(K):
            err = out_error(out[s, i].reshape(H, hd), ref[i])
            assert err <= OUT_TOL, (s, i, err)


@pytest.mark.parametrize("int8", [False, True])
def test_rswa_verify_steady_ring_and_fill(torch, kvd, int8):
    """One stream per ring state (warm with room for the drafts, filling during
    them, full: each draft evicts the oldest row) with a reference block; K = 6."""
    H, hd, W, ref_cap, K = 4, 128, 128, 64, 6
    scale = np.float32(1.0 / math.sqrt(hd))
    for n_gen in (10, 124, 333):
        cache = kvd.RingCache(1, ref_cap, H, hd, W, int8=int8)
        k = synthetic.normal((H, 50, hd), 900)
        v = synthetic.normal((H, 50, hd), 901)
        kvd.rswa_record_prefill(cache, 0, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        rk = np.zeros((H, ref_cap, hd), np.float32)
        rv = np.zeros_like(rk)
        rk[:, :50], rv[:, :50] = k, v
        gk = np.zeros((H, W, hd), np.float32)
        gv = np.zeros_like(gk)
        cur = np.zeros(2, np.int32)
        for t in range(n_gen):
            kt = synthetic.normal((1, H, hd), 1000 + t)
            vt = synthetic.normal((1, H, hd), 2000 + t)
            kvd.rswa_ring_write(cache, torch.from_numpy(kt).cuda(), torch.from_numpy(vt).cuda())
            oracle.rswa_write(gk, gv, kt[0], vt[0], True, cur)
        q = synthetic.normal((1, K, H, hd), 3000 + n_gen)
        dk = synthetic.normal((1, K, H, hd), 3100 + n_gen)
        dv = synthetic.normal((1, K, H, hd), 3200 + n_gen)
        out = kvd.rswa_verify(torch.from_numpy(q).cuda(), torch.from_numpy(dk).cuda(), torch.from_numpy(dv).cuda(),
                              cache, int8=int8).cpu().numpy()
        ref = oracle.rswa_verify(q[0], dk[0], dv[0], rk, rv, 50, gk, gv, cur, scale, int8=int8)
        for i in range(K):
            assert out_error(out[0, i].reshape(H, hd), ref[i]) <= OUT_TOL, (n_gen, i)
        assert cache.ring_len[0] == cur[0] and cache.ring_pos[0] == cur[1]
