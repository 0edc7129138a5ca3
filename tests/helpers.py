"""Shared helpers for the GPU parity tests: build the same cache on the device
(through the library's C ABI) and in the CPU oracle from the same seeded rows,
and compare the results element by element."""

from __future__ import annotations

import math

import numpy as np

import oracle
import synthetic

# Tolerances fixed for this path:
#  - quantised codes and scales: bit-exact;
#  - outputs: max |gpu - oracle| / RMS(oracle output over the live heads) <= 2e-5;
#  - imp: per element |gpu - oracle| <= 1e-5 |oracle| + 1e-12.
OUT_TOL = 2e-5
IMP_RTOL, IMP_ATOL = 1e-5, 1e-12


def seq_rows(lengths, n_kv, hd, seed, outliers=True):
    """Per-sequence K, V rows [L_b, n_kv, hd] f32 (per-channel log-uniform sigma)."""
    ks, vs = [], []
    for b, L in enumerate(lengths):
        if outliers:
            sig_k = synthetic.channel_sigma((n_kv, hd), seed * 1000 + 3 * b)
            sig_v = synthetic.channel_sigma((n_kv, hd), seed * 1000 + 3 * b + 1)
            ks.append(synthetic.outlier_rows(int(L), n_kv, hd, sig_k, seed * 1000 + 3 * b + 2))
            vs.append(synthetic.outlier_rows(int(L), n_kv, hd, sig_v, seed * 7919 + b))
        else:
            ks.append(synthetic.normal((int(L), n_kv, hd), seed * 1000 + 2 * b))
            vs.append(synthetic.normal((int(L), n_kv, hd), seed * 1000 + 2 * b + 1))
    return ks, vs


def oracle_caches(mode, lengths, n_kv, hd, alive, ks, vs, cap=None):
    out = []
    for b, L in enumerate(lengths):
        c = oracle.OracleSeqCache(mode, n_kv, hd, max(int(cap or L), 1), alive=alive)
        c.append_rows(ks[b], vs[b])
        out.append(c)
    return out


def gpu_append_stepwise(layer, ks, vs, torch):
    """Append row t of every sequence that still has one, one row per call."""
    import kv_cache_decode_attention_gb300 as kvd

    n_seq = len(ks)
    T = max(k.shape[0] for k in ks)
    for t in range(T):
        nn = np.array([1 if ks[b].shape[0] > t else 0 for b in range(n_seq)], np.int32)
        if not nn.any():
            continue
        kk = np.concatenate([ks[b][t:t + 1] for b in range(n_seq) if nn[b]])
        vv = np.concatenate([vs[b][t:t + 1] for b in range(n_seq) if nn[b]])
        kvd.kv_append(layer, torch.from_numpy(kk).cuda(), torch.from_numpy(vv).cuda(), nn)


def gpu_append_bulk(layer, ks, vs, torch, pieces=(1,)):
    """Append every sequence's rows in `len(pieces)` bulk calls splitting each
    sequence's rows at the given fractions."""
    import kv_cache_decode_attention_gb300 as kvd

    n_seq = len(ks)
    bounds = [[0] + [int(round(f * k.shape[0])) for f in pieces] for k in ks]
    for i in range(len(pieces)):
        nn = np.array([bounds[b][i + 1] - bounds[b][i] for b in range(n_seq)], np.int32)
        kk = np.concatenate([ks[b][bounds[b][i]:bounds[b][i + 1]] for b in range(n_seq)])
        vv = np.concatenate([vs[b][bounds[b][i]:bounds[b][i + 1]] for b in range(n_seq)])
        kvd.kv_append(layer, torch.from_numpy(np.ascontiguousarray(kk)).cuda(),
                      torch.from_numpy(np.ascontiguousarray(vv)).cuda(), nn)


def assert_storage_bitexact(layer, ocs, torch):
    """Codes, scales, fields and f32 rows on the device equal the oracle's bit for bit."""
    from kv_cache_decode_attention_gb300 import _abi

    comp = {s: layer.component(s) for s in range(_abi.BUF_COUNT)}
    host = {s: (t.cpu().numpy() if t is not None else None) for s, t in comp.items()}
    for b, oc in enumerate(ocs):
        assert layer.seq_len(b) == oc.seq_len
        assert layer.frozen(b) == oc.frozen, b
        for h in layer.live_heads:
            r0, _ = layer.region(b, h)
            n = oc.seq_len
            gl = layer.live_heads.index(h)
            if oc.kq is not None:
                assert np.array_equal(host[_abi.BUF_KQ][r0:r0 + n], oc.kq[h, :n]), (b, h)
                assert np.array_equal(host[_abi.BUF_KS][r0:r0 + n].view(np.uint32),
                                      oc.ks[h, :n].view(np.uint32)), (b, h)
                assert np.array_equal(host[_abi.BUF_KCOL][b, gl].view(np.uint32),
                                      oc.kcol[h].view(np.uint32)), (b, h)
            else:
                assert np.array_equal(host[_abi.BUF_K][r0:r0 + n].view(np.uint32),
                                      oc.k[h, :n].view(np.uint32)), (b, h)
            if oc.vq is not None:
                assert np.array_equal(host[_abi.BUF_VQ][r0:r0 + n], oc.vq[h, :n]), (b, h)
                assert np.array_equal(host[_abi.BUF_VS][r0:r0 + n].view(np.uint32),
                                      oc.vs[h, :n].view(np.uint32)), (b, h)
                assert np.array_equal(host[_abi.BUF_VCOL][b, gl].view(np.uint32),
                                      oc.vcol[h].view(np.uint32)), (b, h)
            else:
                assert np.array_equal(host[_abi.BUF_V][r0:r0 + n].view(np.uint32),
                                      oc.v[h, :n].view(np.uint32)), (b, h)


def out_error(gpu, ref, live_rows_mask=None):
    """max |gpu - ref| / RMS(ref) over the rows selected (default: all)."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    if live_rows_mask is not None:
        g, r = g[live_rows_mask], r[live_rows_mask]
    rms = math.sqrt(float(np.mean(r * r)))
    return float(np.max(np.abs(g - r))) / rms


def assert_imp_close(gpu_imp, ref_imp):
    g = np.asarray(gpu_imp, np.float64)
    r = np.asarray(ref_imp, np.float64)
    bad = np.abs(g - r) > IMP_RTOL * np.abs(r) + IMP_ATOL
    assert not bad.any(), "imp mismatch at %s: gpu %s ref %s" % (
        np.nonzero(bad)[0][:5], g[bad][:5], r[bad][:5])
