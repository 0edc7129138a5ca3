"""Failure detection without a GPU fault: the library's host-side hook
(kvd_test_fail_after) makes the Nth launch or copy of a call report failure.

For every entry point that changes host-mirrored state (sequence lengths,
frozen flags, ring cursors, write histories) each launch of the call in turn
is made to fail: the call must return KVD_ECUDA and leave that state exactly
as it was (the pages' "a refused call changes nothing", extended to a failed
launch).  The device may hold the partial work of the launches that went in
before the failure, so each case then resets what it touched and checks that
the same calls, repeated without the hook, match the CPU oracle.  No kernel
faults, traps or hangs: the hook only changes the status the host sees.
"""

import math

import numpy as np
import pytest

import oracle
import synthetic
from helpers import OUT_TOL, out_error

pytestmark = pytest.mark.gpu

ECUDA = -5


@pytest.fixture(scope="module")
def env():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300 import _abi
    from kv_cache_decode_attention_gb300.build import build

    build()
    yield torch, kvd, _abi
    _abi.lib().kvd_test_fail_after(-1)


def _fail_after(abi, n):
    assert abi.lib().kvd_test_fail_after(n) == 0


def _host_state(layer):
    return ([layer.seq_len(b) for b in range(layer.n_seq)], [layer.frozen(b) for b in range(layer.n_seq)])


def _expect_failure(abi, fn, n):
    """Arm the hook at launch n, run fn; True if it failed (KVD_ECUDA), False if
    the call issued no more than n launches (it then ran to completion)."""
    _fail_after(abi, n)
    try:
        fn()
        return False
    except abi.KvdError as e:
        assert e.status == ECUDA, e
        return True
    finally:
        _fail_after(abi, -1)  # disarm what a shorter call left armed


def test_append_across_the_freeze_fails_at_every_launch(env):
    """kv_append of rows crossing row 64 (append, freeze, append): each launch
    failing leaves the lengths and frozen flags as they were."""
    torch, kvd, abi = env
    n_kv, hd, lengths = 2, 128, [30, 30, 10]
    rng = np.random.default_rng(5)
    first = [synthetic.normal((L, n_kv, hd), 500 + b) for b, L in enumerate(lengths)]
    more = [synthetic.normal((n, n_kv, hd), 600 + b) for b, n in enumerate([50, 40, 5])]
    vfirst = [synthetic.normal(x.shape, 700 + b) for b, x in enumerate(first)]
    vmore = [synthetic.normal(x.shape, 800 + b) for b, x in enumerate(more)]
    layer = kvd.LayerKvCache(3, n_kv, hd, "q8", 128)

    def put(ks, vs):
        kvd.kv_append(layer, torch.from_numpy(np.concatenate(ks)).cuda(), torch.from_numpy(np.concatenate(vs)).cuda(),
                      np.array([x.shape[0] for x in ks], np.int32))

    put(first, vfirst)
    torch.cuda.synchronize()
    before = _host_state(layer)
    failed = 0
    for n in range(8):
        if not _expect_failure(abi, lambda: put(more, vmore), n):
            break
        failed += 1
        assert _host_state(layer) == before, n
        # the launches before the failure may have written rows: start over
        torch.cuda.synchronize()
        layer.reset()
        put(first, vfirst)
        torch.cuda.synchronize()
        assert _host_state(layer) == before
    assert failed >= 3  # append, freeze, append
    # the call that ran to completion at the last n matches the oracle
    assert layer.seq_len(0) == 80 and layer.frozen(0) and layer.frozen(1) and not layer.frozen(2)
    q = rng.standard_normal((3, n_kv * 4, hd)).astype(np.float32)
    out = kvd.decode_attention(torch.from_numpy(q).cuda(), layer).cpu().numpy()
    for b in range(3):
        oc = oracle.OracleSeqCache(oracle.Q8, n_kv, hd, 128)
        oc.append_rows(np.concatenate([first[b], more[b]]), np.concatenate([vfirst[b], vmore[b]]))
        ref = oc.decode(q[b], n_kv * 4, np.float32(1.0 / math.sqrt(hd)))
        assert out_error(out[b], ref) <= OUT_TOL, b
    assert layer.device_error() == 0


def test_truncate_over_two_slices_fails_without_changing_lengths(env):
    """kv_truncate_last over 300 sequences (two launches of 256 and 44)."""
    torch, kvd, abi = env
    n_seq = 300
    layer = kvd.LayerKvCache(n_seq, 1, 64, "f32", 8)
    kvd.kv_append(layer, torch.randn(n_seq * 5, 1, 64, device="cuda"), torch.randn(n_seq * 5, 1, 64, device="cuda"),
                  np.full(n_seq, 5, np.int32))
    torch.cuda.synchronize()
    before = _host_state(layer)
    for n in (0, 1):
        assert _expect_failure(abi, lambda: kvd.kv_truncate_last(layer, 2), n)
        assert _host_state(layer) == before
    kvd.kv_truncate_last(layer, 2)
    assert all(layer.seq_len(b) == 3 for b in range(n_seq))


def test_ring_write_and_prefill_keep_their_cursors(env):
    """rswa_record_prefill and rswa_ring_write (f32 regions and the int8 mirror):
    a failed launch leaves prefill_len, ring_len, ring_pos and the write
    history as they were."""
    torch, kvd, abi = env
    for int8 in (False, True):
        cache = kvd.RingCache(2, 32, 2, 64, 4, int8=int8)
        for s in range(2):
            kvd.rswa_record_prefill(cache, s, torch.randn(2, 20, 64, device="cuda"), torch.randn(2, 20, 64, device="cuda"))
        for _ in range(5):
            kvd.rswa_ring_write(cache, torch.randn(2, 2, 64, device="cuda"), torch.randn(2, 2, 64, device="cuda"))
        torch.cuda.synchronize()

        def cursors():
            return (cache.prefill_len.tolist(), cache.ring_len.tolist(), cache.ring_pos.tolist(),
                    [(h.decode_writes, h.lineage_epoch) for h in cache.history])

        before = cursors()
        k, v = torch.randn(2, 2, 64, device="cuda"), torch.randn(2, 2, 64, device="cuda")
        assert _expect_failure(abi, lambda: kvd.rswa_ring_write(cache, k, v), 0)
        assert cursors() == before
        pk, pv = torch.randn(2, 10, 64, device="cuda"), torch.randn(2, 10, 64, device="cuda")
        assert _expect_failure(abi, lambda: kvd.rswa_record_prefill(cache, 1, pk, pv), 0)
        assert cursors() == before
        kvd.rswa_ring_write(cache, k, v)
        assert cache.ring_pos.tolist() == [(before[2][s] + 1) % 4 for s in range(2)]


def test_decode_failing_at_each_launch_reports_and_recovers(env):
    """decode_attention (split, merge, imp pass): each launch failing returns
    KVD_ECUDA and leaves the lengths; the next call, unarmed, is exact."""
    torch, kvd, abi = env
    n_kv, hd, hpk, L = 2, 128, 4, 300
    layer = kvd.LayerKvCache(2, n_kv, hd, "q8", L + 4)
    k = [synthetic.normal((L, n_kv, hd), 900 + b) for b in range(2)]
    v = [synthetic.normal((L, n_kv, hd), 910 + b) for b in range(2)]
    kvd.kv_append(layer, torch.from_numpy(np.concatenate(k)).cuda(), torch.from_numpy(np.concatenate(v)).cuda(),
                  np.array([L, L], np.int32))
    q = torch.randn(2, n_kv * hpk, hd, device="cuda")
    imp = torch.zeros(layer.imp_len, device="cuda")
    failed = 0
    for n in range(6):
        if not _expect_failure(abi, lambda: kvd.decode_attention(q, layer, imp=imp), n):
            break
        failed += 1
    assert failed >= 3  # split, merge, imp pass
    assert all(layer.seq_len(b) == L for b in range(2))
    out = kvd.decode_attention(q, layer).cpu().numpy()
    qh = q.cpu().numpy()
    for b in range(2):
        oc = oracle.OracleSeqCache(oracle.Q8, n_kv, hd, L)
        oc.append_rows(k[b], v[b])
        assert out_error(out[b], oc.decode(qh[b], n_kv * hpk, np.float32(1.0 / math.sqrt(hd)))) <= OUT_TOL
    assert layer.device_error() == 0
