"""Full-size parity: the benchmark's own workloads (built by the same builders,
decoded by the same calls and launch configuration as bench.py), checked on
sampled sequences that the CPU oracle recomputes from the regenerated inputs.

Every oracle input is regenerated from the workload's seeds (never read back
from the device); the device's stored codes, scales, fields and ring rows are
compared bit for bit with the oracle's, outputs within 2e-5 of the output RMS,
imp within 1e-5 relative.
"""

import math

import numpy as np
import pytest

import oracle
from helpers import OUT_TOL, assert_imp_close, out_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300 import workloads as W
    from kv_cache_decode_attention_gb300.build import build

    build()
    return torch, kvd, W


def _oracle_seq(wl, b, heads=None):
    """Oracle cache of sequence b (all KV heads, or the listed ones) from the
    regenerated rows."""
    k, v = wl.rows(b)
    k, v = k.cpu().numpy(), v.cpu().numpy()
    if heads is None:
        oc = oracle.OracleSeqCache(wl.mode, wl.n_kv, wl.hd, int(wl.lengths[b]), alive=wl.alive)
        oc.append_rows(k, v)
        return oc, None
    kk = np.ascontiguousarray(k[:, heads])
    vv = np.ascontiguousarray(v[:, heads])
    oc = oracle.OracleSeqCache(wl.mode, len(heads), wl.hd, int(wl.lengths[b]))
    oc.append_rows(kk, vv)
    return oc, heads


def _check_storage(kvd, wl, b, oc, heads):
    from kv_cache_decode_attention_gb300 import _abi

    L = int(wl.lengths[b])
    # the oracle cache holds either every KV head (index = head) or just the
    # listed heads (index = position in the list)
    pairs = ([(h, h) for h in range(wl.n_kv) if wl.alive[h]] if heads is None
             else [(h, i) for i, h in enumerate(heads)])
    for h, oh in pairs:
        r0, _ = wl.layer.region(b, h)
        gl = wl.layer.live_heads.index(h)
        if oc.kq is not None:
            kq = wl.layer.component(_abi.BUF_KQ)[r0:r0 + L].cpu().numpy()
            ks = wl.layer.component(_abi.BUF_KS)[r0:r0 + L].cpu().numpy()
            assert np.array_equal(kq, oc.kq[oh, :L]), (b, h)
            assert np.array_equal(ks.view(np.uint32), oc.ks[oh, :L].view(np.uint32)), (b, h)
            col = wl.layer.component(_abi.BUF_KCOL)[b, gl].cpu().numpy()
            assert np.array_equal(col.view(np.uint32), oc.kcol[oh].view(np.uint32)), (b, h)
        else:
            kf = wl.layer.component(_abi.BUF_K)[r0:r0 + L].cpu().numpy()
            assert np.array_equal(kf.view(np.uint32), oc.k[oh, :L].view(np.uint32)), (b, h)
        if oc.vq is not None:
            vq = wl.layer.component(_abi.BUF_VQ)[r0:r0 + L].cpu().numpy()
            vs = wl.layer.component(_abi.BUF_VS)[r0:r0 + L].cpu().numpy()
            assert np.array_equal(vq, oc.vq[oh, :L]), (b, h)
            assert np.array_equal(vs.view(np.uint32), oc.vs[oh, :L].view(np.uint32)), (b, h)
            col = wl.layer.component(_abi.BUF_VCOL)[b, gl].cpu().numpy()
            assert np.array_equal(col.view(np.uint32), oc.vcol[oh].view(np.uint32)), (b, h)
        else:
            vf = wl.layer.component(_abi.BUF_V)[r0:r0 + L].cpu().numpy()
            assert np.array_equal(vf.view(np.uint32), oc.v[oh, :L].view(np.uint32)), (b, h)


def _decode_and_check(torch, kvd, wl, samples, heads_per_sample=None, with_imp=True, errors=None):
    q = wl.query(0)
    imp = torch.zeros(wl.layer.imp_len, device="cuda") if with_imp else None
    ws = torch.empty(wl.layer.workspace_bytes(wl.n_q, with_imp), dtype=torch.uint8, device="cuda")
    out = kvd.decode_attention(q, wl.layer, imp=imp, scale=wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert wl.layer.device_error() == 0
    out = out.cpu().numpy()
    qh = q.cpu().numpy()
    got_imp = imp.cpu().numpy() if with_imp else None
    for b in samples:
        heads = heads_per_sample
        oc, hs = _oracle_seq(wl, b, heads)
        _check_storage(kvd, wl, b, oc, hs)
        L = int(wl.lengths[b])
        if hs is None:
            imp_ref = np.zeros(max(L, 1))
            ref = oc.decode(qh[b], wl.n_q, np.float32(wl.scale), imp_ref)
            live = np.array([bool(wl.alive[h // wl.hpk]) for h in range(wl.n_q)])
            assert np.all(out[b][~live] == 0.0)
            err = out_error(out[b], ref, live)
            if errors is not None:
                errors.append((wl.name, b, int(wl.lengths[b]), err))
            else:
                assert err <= OUT_TOL, (b, err)
            if with_imp:
                ib = int(wl.layer.imp_base[b])
                assert_imp_close(got_imp[ib:ib + L], imp_ref[:L])
        else:
            qg = np.concatenate([qh[b, g * wl.hpk:(g + 1) * wl.hpk] for g in hs])
            ref = oc.decode(qg, len(hs) * wl.hpk, np.float32(wl.scale))
            gq = np.concatenate([out[b, g * wl.hpk:(g + 1) * wl.hpk] for g in hs])
            err = out_error(gq, ref)
            assert err <= OUT_TOL, (b, err)


def test_q8_gqa_full_size(env):
    """32 seq x 4096 rows, 32 Q / 8 KV heads, q8_2f built one row at a time."""
    torch, kvd, W = env
    wl = W.q8_gqa(extra_cap=64)
    _decode_and_check(torch, kvd, wl, samples=[0, 17, 31])
    del wl
    torch.cuda.empty_cache()


def test_long_q8_full_size(env):
    """4 seq x 131072 rows, 64 Q / 4 KV heads (16 per group), the benchmark's
    decode with imp (split_h16_kernel with the score stores + imp_kernel):
    sequences 1 and 2 in full (every group, imp per element over all 131072
    rows), sequences 0 and 3 on one group each."""
    torch, kvd, W = env
    wl = W.long_q8(extra_cap=64)
    q = wl.query(0)
    imp = torch.zeros(wl.layer.imp_len, device="cuda")
    ws = torch.empty(wl.layer.workspace_bytes(wl.n_q, True), dtype=torch.uint8, device="cuda")
    out = kvd.decode_attention(q, wl.layer, imp=imp, scale=wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert wl.layer.device_error() == 0
    out, qh, got_imp = out.cpu().numpy(), q.cpu().numpy(), imp.cpu().numpy()
    full = [_oracle_seq(wl, b)[0] for b in (1, 2)]
    imps = [np.zeros(oc.cap) for oc in full]
    refs, _ = oracle.decode_many(full, [qh[1], qh[2]], wl.n_q, np.float32(wl.scale), imps)
    L = int(wl.lengths[0])
    for b, ref, imp_ref, oc in zip((1, 2), refs, imps, full):
        _check_storage(kvd, wl, b, oc, None)
        err = out_error(out[b], ref)
        assert err <= OUT_TOL, (b, err)
        ib = int(wl.layer.imp_base[b])
        assert_imp_close(got_imp[ib:ib + L], imp_ref[:L])
        assert abs(imp_ref[:L].sum() - wl.n_q) < 1e-6 * wl.n_q
    for b, g in ((0, 3), (3, 0)):
        oc, hs = _oracle_seq(wl, b, [g])
        ref = oc.decode(qh[b, g * wl.hpk:(g + 1) * wl.hpk], wl.hpk, np.float32(wl.scale))
        err = out_error(out[b, g * wl.hpk:(g + 1) * wl.hpk], ref)
        assert err <= OUT_TOL, (b, g, err)
    del wl
    torch.cuda.empty_cache()


def test_verify_q8_full_size(env):
    """The benchmark's speculative step on q8_gqa (32 seq x 4096 rows): 4 draft
    rows appended per sequence, one query-batched verify (16 query rows per
    group on split_h16_kernel), three sampled sequences against the oracle's
    decode_verify, then kv_truncate_last of the 4 drafts and a plain decode
    that matches the cache without them."""
    torch, kvd, W = env
    import synthetic

    K = 4
    wl = W.q8_gqa(extra_cap=64)
    n_seq, n_q, n_kv, hd = wl.n_seq, wl.n_q, wl.n_kv, wl.hd
    dk = synthetic.normal((n_seq, K, n_kv, hd), 81_000)
    dv = synthetic.normal((n_seq, K, n_kv, hd), 82_000)
    vq = synthetic.normal((n_seq, K, n_q, hd), 80_000)
    kvd.kv_append(wl.layer, torch.from_numpy(dk.reshape(-1, n_kv, hd)).cuda(),
                  torch.from_numpy(dv.reshape(-1, n_kv, hd)).cuda(), np.full(n_seq, K, np.int32))
    out = kvd.decode_attention_verify(torch.from_numpy(vq).cuda(), wl.layer, K, scale=wl.scale).cpu().numpy()
    assert wl.layer.device_error() == 0
    samples = (0, 13, 31)
    for b in samples:
        oc_full = oracle.OracleSeqCache(wl.mode, n_kv, hd, int(wl.lengths[b]) + K, alive=wl.alive)
        k, v = wl.rows(b)
        oc_full.append_rows(k.cpu().numpy(), v.cpu().numpy())
        oc_full.append_rows(dk[b], dv[b])
        ref = oc_full.decode_verify(vq[b], n_q, K, np.float32(wl.scale))
        for i in range(K):
            err = out_error(out[b, i], ref[i])
            assert err <= OUT_TOL, (b, i, err)
    kvd.kv_truncate_last(wl.layer, K)
    assert all(wl.layer.seq_len(b) == int(wl.lengths[b]) for b in range(n_seq))
    _decode_and_check(torch, kvd, wl, samples=[13], with_imp=True)
    del wl
    torch.cuda.empty_cache()


def test_ragged_full_size(env):
    """256 seq, L ~ U{1..16384}, four layers (f32, q8, q8k, q8v), 2 of 8 KV heads
    dead per layer: shortest, longest, and sequences around the freeze point."""
    torch, kvd, W = env
    layers = W.ragged(extra_cap=16)
    L = layers[0].lengths
    order = np.argsort(L)
    picks = {int(order[0]), int(order[-1]), int(np.argmin(np.abs(L - 64))),
             int(np.argmin(np.abs(L - 100))), int(order[len(order) // 2])}
    errors = []
    for wl in layers:
        _decode_and_check(torch, kvd, wl, samples=sorted(picks), errors=errors)
    print("ragged output errors (layer, sequence, rows, max err / rms):", errors)
    bad = [e for e in errors if e[3] > OUT_TOL]
    assert not bad, bad
    del layers
    torch.cuda.empty_cache()


def test_rswa_steady_full_size(env):
    """16 streams, 10 heads, prefix 32640 rows, ring after 500 steps: ring bytes
    bit-exact and outputs of two sampled streams against the oracle (which
    replays the 500 ring writes itself)."""
    torch, kvd, W = env
    wl = W.rswa_steady()
    c = wl.cache
    assert c.ring_len.tolist() == [128] * c.B and c.ring_pos.tolist() == [500 % 128] * c.B
    q = wl.query(0)
    out = kvd.rswa_decode(q, c).cpu().numpy()
    assert c.device_error() == 0
    qh = q.cpu().numpy()
    scale = np.float32(1.0 / math.sqrt(128))
    ring_k = np.zeros((c.B, c.H, c.W, c.head_dim), np.float32)
    ring_v = np.zeros_like(ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(c.B)]
    for t in range(wl.steps):
        k, v = wl.step_rows(t)
        k, v = k.cpu().numpy(), v.cpu().numpy()
        for s in range(c.B):
            oracle.rswa_write(ring_k[s], ring_v[s], k[s], v[s], True, cursors[s])
    assert np.array_equal(c.ring_k.cpu().numpy(), ring_k)
    assert np.array_equal(c.ring_v.cpu().numpy(), ring_v)
    for s in (3, 15):
        pk, pv = wl.prefill_rows(s)
        pk, pv = pk.cpu().numpy(), pv.cpu().numpy()
        ref = oracle.rswa_decode(qh[s], pk, pv, wl.prefill, ring_k[s], ring_v[s], cursors[s][0], scale)
        err = out_error(out[s].reshape(c.H, c.head_dim), ref)
        assert err <= OUT_TOL, (s, err)
    del wl, c
    torch.cuda.empty_cache()


def test_rswa_i8_steady_full_size(env):
    """The same workload with the int8 mirror (about 1.4 GB of codes and scales
    read per decode): the ring mirror bit-exact, the reference mirror of two
    sampled streams bit-exact, and their decode_attention_int8 outputs against
    the oracle."""
    torch, kvd, W = env
    wl = W.rswa_steady(int8=True)
    c = wl.cache
    q = wl.query(0)
    out = kvd.rswa_decode_i8(q, c).cpu().numpy()
    assert c.device_error() == 0
    qh = q.cpu().numpy()
    scale = np.float32(1.0 / math.sqrt(128))
    ring_k = np.zeros((c.B, c.H, c.W, c.head_dim), np.float32)
    ring_v = np.zeros_like(ring_k)
    cursors = [np.zeros(2, np.int32) for _ in range(c.B)]
    for t in range(wl.steps):
        k, v = wl.step_rows(t)
        k, v = k.cpu().numpy(), v.cpu().numpy()
        for s in range(c.B):
            oracle.rswa_write(ring_k[s], ring_v[s], k[s], v[s], True, cursors[s])
    gk8, gks = oracle.rswa_mirror(ring_k)
    gv8, gvs = oracle.rswa_mirror(ring_v)
    assert np.array_equal(c.ring_k8.cpu().numpy(), gk8)
    assert np.array_equal(c.ring_v8.cpu().numpy(), gv8)
    assert np.array_equal(c.ring_ks.cpu().numpy().view(np.uint32), gks.view(np.uint32))
    assert np.array_equal(c.ring_vs.cpu().numpy().view(np.uint32), gvs.view(np.uint32))
    for s in (3, 15):
        pk, pv = wl.prefill_rows(s)
        rk8, rks = oracle.rswa_mirror(pk.cpu().numpy())
        rv8, rvs = oracle.rswa_mirror(pv.cpu().numpy())
        assert np.array_equal(c.ref_k8[s].cpu().numpy(), rk8)
        assert np.array_equal(c.ref_vs[s].cpu().numpy().view(np.uint32), rvs.view(np.uint32))
        ref = oracle.rswa_decode_i8(qh[s], rk8, rks, rv8, rvs, wl.prefill, gk8[s], gks[s], gv8[s], gvs[s],
                                    cursors[s][0], scale)
        err = out_error(out[s].reshape(c.H, c.head_dim), ref)
        assert err <= OUT_TOL, (s, err)
    # the benchmark's speculative step: 4 drafts verified over the same mirror
    # (the reference block on the tensor-core kernel), two sampled streams
    import synthetic

    K = 4
    vq = synthetic.normal((c.B, K, c.H, c.head_dim), 5900)
    vk = synthetic.normal((c.B, K, c.H, c.head_dim), 5901)
    vv = synthetic.normal((c.B, K, c.H, c.head_dim), 5902)
    dev = torch.device("cuda")
    vout = kvd.rswa_verify(torch.from_numpy(vq).to(dev), torch.from_numpy(vk).to(dev),
                           torch.from_numpy(vv).to(dev), c, int8=True).cpu().numpy()
    assert c.device_error() == 0
    for s in (0, 11):
        pk, pv = wl.prefill_rows(s)
        ref = oracle.rswa_verify(vq[s], vk[s], vv[s], pk.cpu().numpy(), pv.cpu().numpy(), wl.prefill, ring_k[s],
                                 ring_v[s], cursors[s], scale, int8=True)
        for i in range(K):
            err = out_error(vout[s, i].reshape(c.H, c.head_dim), ref[i])
            assert err <= OUT_TOL, (s, i, err)
    del wl, c
    torch.cuda.empty_cache()


def test_born_eviction_long_full_size(env):
    """Born eviction at full size: 4 seq x 131072 rows (q8_2f, 16 heads per group)
    cut to 65536 rows with seeded masses full of ties; one sampled group's codes,
    scales and imp bit-exact against the oracle's evict_born, then its decode."""
    torch, kvd, W = env
    wl = W.long_q8(extra_cap=64)
    rng = np.random.default_rng(4242)
    masses = (rng.integers(0, 64, size=wl.layer.imp_len) / 16.0).astype(np.float32)
    imp = torch.from_numpy(masses.copy()).cuda()
    keep, sink, recent = 65536, 4, 8192
    import ctypes as C

    from kv_cache_decode_attention_gb300 import _abi as abi

    n = C.c_int64(0)
    abi.call("kv_evict_workspace_bytes", C.byref(wl.layer.L), keep, C.byref(n))
    ws = torch.empty(int(n.value), dtype=torch.uint8, device="cuda")  # allocated outside the timing
    # a first eviction on a small layer loads every kernel of the path, so the
    # timing below is a steady-state call
    small = kvd.LayerKvCache(1, 1, 128, "q8", 256)
    kvd.kv_append(small, torch.randn(200, 1, 128, device="cuda"), torch.randn(200, 1, 128, device="cuda"),
                  np.array([200], np.int32))
    kvd.kv_evict_born(small, torch.rand(small.imp_len, device="cuda"), 100, 4, 10)
    torch.cuda.synchronize()
    ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev[0].record()
    kvd.kv_evict_born(wl.layer, imp, keep, sink, recent, workspace=ws)
    ev[1].record()
    torch.cuda.synchronize()
    print("kv_evict_born 4 x 131072 -> 65536 rows: %.1f us" % (ev[0].elapsed_time(ev[1]) * 1e3))
    assert wl.layer.device_error() == 0
    b, h = 2, 1
    oc, _ = _oracle_seq(wl, b, [h])
    L = int(wl.lengths[b])
    ib = int(wl.layer.imp_base[b])
    o_imp = np.zeros(oc.cap, np.float32)
    o_imp[:L] = masses[ib:ib + L]
    assert oc.evict_born(keep, sink, recent, o_imp) == keep
    got = imp.cpu().numpy()
    assert np.array_equal(got[ib:ib + L].view(np.uint32), o_imp[:L].view(np.uint32))
    assert all(wl.layer.seq_len(s) == keep for s in range(wl.n_seq))
    from kv_cache_decode_attention_gb300 import _abi

    r0, _ = wl.layer.region(b, h)
    for slot, arr in ((_abi.BUF_KQ, oc.kq), (_abi.BUF_VQ, oc.vq)):
        assert np.array_equal(wl.layer.component(slot)[r0:r0 + keep].cpu().numpy(), arr[0, :keep])
    for slot, arr in ((_abi.BUF_KS, oc.ks), (_abi.BUF_VS, oc.vs)):
        assert np.array_equal(wl.layer.component(slot)[r0:r0 + keep].cpu().numpy().view(np.uint32),
                              arr[0, :keep].view(np.uint32))
    q = wl.query(0)
    out = kvd.decode_attention(q, wl.layer, scale=wl.scale).cpu().numpy()
    qg = q.cpu().numpy()[b, h * wl.hpk:(h + 1) * wl.hpk]
    ref = oc.decode(qg, wl.hpk, np.float32(wl.scale))
    assert out_error(out[b, h * wl.hpk:(h + 1) * wl.hpk], ref) <= OUT_TOL
    del wl
    torch.cuda.empty_cache()
