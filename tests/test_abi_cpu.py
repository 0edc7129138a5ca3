"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
entry point include/kvd.h declares, and its host validation returns the
documented status codes before touching the device (no device buffer is ever
dereferenced here: every call below fails validation or only computes sizes)."""

import ctypes as C
import os

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def abi():
    from kv_cache_decode_attention_gb300 import _abi
    from kv_cache_decode_attention_gb300.build import build

    build()
    return _abi


def test_library_exports_every_declared_symbol(abi):
    names = abi.declared_symbols()
    assert len(names) >= 16
    L = abi.lib()
    for n in names:
        assert hasattr(L, n), n
    # and the binding declares exactly those
    assert set(abi._SIGS) == set(names)


def test_header_has_no_torch_types():
    text = open(os.path.join(ROOT, "include", "kvd.h")).read()
    for bad in ("torch", "at::", "Tensor", "c10"):
        assert bad not in text


def _bytes(abi, n_seq, n_kv, hd, mode, cap, alive=None):
    cap = np.ascontiguousarray(cap, np.int64)
    out = np.zeros(abi.BUF_COUNT, np.int64)
    hb = C.c_int64(0)
    al = None if alive is None else C.c_void_p(np.ascontiguousarray(alive, np.uint8).ctypes.data)
    st = abi.lib().kvd_layer_bytes(n_seq, n_kv, hd, mode, C.c_void_p(cap.ctypes.data), al,
                                   C.c_void_p(out.ctypes.data), C.byref(hb))
    return st, out, hb.value


def test_layer_bytes_layout(abi):
    # q8 (K and V int8), hd 128, 2 sequences of 100 (-> 112) and 16 rows, 8 heads, 2 dead
    alive = np.array([1, 1, 0, 1, 1, 1, 0, 1], np.uint8)
    st, out, hb = _bytes(abi, 2, 8, 128, abi.Q8, [100, 16], alive)
    assert st == abi.OK
    rows = (112 + 16) * 6 + 16  # live rows + spare rows
    r256 = lambda x: (x + 255) // 256 * 256
    assert out[abi.BUF_KQ] == r256(rows * 128) and out[abi.BUF_VQ] == r256(rows * 128)
    assert out[abi.BUF_KS] == r256(rows * 4 * 4) and out[abi.BUF_VS] == r256(rows * 4)
    assert out[abi.BUF_K] == 0 and out[abi.BUF_V] == 0
    assert out[abi.BUF_KCOL] == r256(2 * 6 * 128 * 4)
    assert out[abi.BUF_META] > 0 and hb > 0
    st, out, _ = _bytes(abi, 1, 2, 64, abi.F32, [256])
    assert out[abi.BUF_K] == r256((256 * 2 + 16) * 64 * 4) and out[abi.BUF_KQ] == 0
    st, out, _ = _bytes(abi, 1, 2, 64, abi.Q8K, [256])
    assert out[abi.BUF_KQ] > 0 and out[abi.BUF_V] > 0 and out[abi.BUF_VQ] == 0 and out[abi.BUF_VCOL] == 0


@pytest.mark.parametrize("args", [
    (0, 8, 128, 1, [10]),     # no sequences
    (1, 0, 128, 1, [10]),     # no heads
    (1, 8, 96, 1, [10]),      # unsupported head_dim
    (1, 8, 128, 7, [10]),     # bad mode
    (1, 8, 128, 1, [-1]),     # negative capacity
])
def test_layer_bytes_rejects(abi, args):
    st, _, _ = _bytes(abi, *args)
    assert st == abi.EINVAL


def test_rswa_host_validation_before_any_launch(abi):
    L = abi.lib()
    B, H, hd, W = 2, 10, 128, 128
    pl = np.array([-1, 5], np.int32)
    rl = np.zeros(B, np.int32)
    rp = np.zeros(B, np.int32)
    fake = C.c_void_p(1 << 20)  # never dereferenced: validation fails first
    p = lambda a: C.c_void_p(a.ctypes.data)
    # a stream without prefill: ESTATE and the cursors stay untouched
    st = L.rswa_ring_write(fake, fake, fake, fake, p(pl), p(rl), p(rp), None, B, H, hd, W, None, None)
    assert st == abi.ESTATE and rl.tolist() == [0, 0] and rp.tolist() == [0, 0]
    n = C.c_int64(0)
    assert L.rswa_decode_workspace_bytes(B, H, hd, 32640, W, C.byref(n)) == abi.OK and n.value > 0
    ws = C.c_void_p(1 << 21)
    st = L.rswa_decode(fake, fake, fake, fake, fake, p(pl), p(rl), p(rp), B, H, hd, 32640, W,
                       C.c_float(0.088), fake, ws, n.value, None)
    assert st == abi.ESTATE
    pl[:] = [0, 5]
    st = L.rswa_decode(fake, fake, fake, fake, fake, p(pl), p(rl), p(rp), B, H, hd, 32640, W,
                       C.c_float(0.088), fake, ws, n.value, None)
    assert st == abi.EEMPTY  # stream 0: no keys
    # capacity: a prefill longer than the reference block
    st = L.rswa_record_prefill(fake, fake, fake, fake, 0, 33000, B, H, hd, 32640, W, p(pl), p(rl),
                               p(rp), None, None)
    assert st == abi.ECAPACITY and pl.tolist() == [0, 5]
    # ragged region sizes are refused (bulk copies move 16-row groups)
    pl[:] = [3, 5]
    st = L.rswa_decode(fake, fake, fake, fake, fake, p(pl), p(rl), p(rp), B, H, hd, 1000, 100,
                       C.c_float(0.088), fake, ws, n.value, None)
    assert st == abi.EINVAL


def test_layer_calls_reject_uninitialised_descriptor(abi):
    L = abi.lib()
    lay = abi.kvd_layer()  # zeroed: not initialised
    n = C.c_int64(0)
    assert L.kvd_decode_workspace_bytes(C.byref(lay), 8, 0, C.byref(n)) == abi.EINVAL
    assert L.kv_append(C.byref(lay), C.c_void_p(16), C.c_void_p(16), None, None) == abi.EINVAL
    assert L.kv_freeze_colfield(C.byref(lay), None) == abi.EINVAL
    assert L.kvd_wait_timeout_selftest(C.byref(lay), 1000, None) == abi.EINVAL
    assert L.kvd_bounds_selftest_bytes(C.byref(lay), C.byref(n)) == abi.EINVAL
    assert L.kvd_bounds_selftest(C.byref(lay), C.c_void_p(256), 1 << 20, None) == abi.EINVAL
    assert L.kvd_status_string(abi.ECAPACITY) == b"capacity exceeded"


def test_api_fails_loudly_without_library(tmp_path, monkeypatch):
    from kv_cache_decode_attention_gb300 import _abi

    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _abi.lib()


def test_rswa_checkpoint_rollback_contract(abi):
    """rswa RingCache::checkpoint / rollback_to (host cursors only): a rollback
    restores ring_len, ring_pos and the write count and starts a new lineage;
    a checkpoint from another cache, another prefill boundary, an abandoned
    lineage or the future, or one whose discarded writes wrapped over a row
    live at the checkpoint, is refused with nothing changed."""
    L = abi.lib()
    B, W, cid = 2, 128, 77
    pl = np.array([10, 40], np.int32)
    rl = np.array([5, 128], np.int32)
    rp = np.array([5, 9], np.int32)
    hist = (abi.rswa_history * B)()
    hist[0].decode_writes, hist[0].lineage_epoch = 5, 1
    hist[1].decode_writes, hist[1].lineage_epoch = 300, 1
    p = lambda a: C.c_void_p(a.ctypes.data)
    cp = abi.rswa_checkpoint()
    assert L.rswa_checkpoint_take(cid, p(pl), p(rl), p(rp), hist, 0, C.byref(cp)) == abi.OK
    assert (cp.prefill_len, cp.ring_len, cp.ring_pos, cp.decode_writes, cp.lineage_epoch) == (10, 5, 5, 5, 1)

    def state():
        return (rl.tolist(), rp.tolist(), hist[0].decode_writes, hist[0].lineage_epoch)

    # three speculative writes into the warm ring, as rswa_ring_write applies them
    rl[0], rp[0], hist[0].decode_writes = 8, 8, 8
    before = state()
    for bad_id, bad in ((cid + 1, None), (cid, "prefill"), (cid, "future")):
        c2 = abi.rswa_checkpoint.from_buffer_copy(cp)
        if bad == "prefill":
            c2.prefill_len = 11
        if bad == "future":
            c2.decode_writes = 9
        assert L.rswa_rollback_to(bad_id, p(pl), p(rl), p(rp), hist, 0, W, C.byref(c2)) == abi.ESTATE
        assert state() == before
    assert L.rswa_rollback_to(cid, p(pl), p(rl), p(rp), hist, 0, W, C.byref(cp)) == abi.OK
    assert state() == ([5, 128], [5, 9], 5, 2)
    # the same checkpoint now belongs to an abandoned lineage
    assert L.rswa_rollback_to(cid, p(pl), p(rl), p(rp), hist, 0, W, C.byref(cp)) == abi.ESTATE
    # a rollback that discards nothing keeps the lineage
    cp2 = abi.rswa_checkpoint()
    assert L.rswa_checkpoint_take(cid, p(pl), p(rl), p(rp), hist, 0, C.byref(cp2)) == abi.OK
    assert L.rswa_rollback_to(cid, p(pl), p(rl), p(rp), hist, 0, W, C.byref(cp2)) == abi.OK
    assert hist[0].lineage_epoch == 2
    # steady state (ring full): any discarded write overwrote a live row
    cp3 = abi.rswa_checkpoint()
    assert L.rswa_checkpoint_take(cid, p(pl), p(rl), p(rp), hist, 1, C.byref(cp3)) == abi.OK
    rp[1], hist[1].decode_writes = 10, 301
    assert L.rswa_rollback_to(cid, p(pl), p(rl), p(rp), hist, 1, W, C.byref(cp3)) == abi.ESTATE
    assert (rl[1], rp[1], hist[1].decode_writes, hist[1].lineage_epoch) == (128, 10, 301, 1)
    # warm ring: exactly W - ring_len discarded writes are still lossless, one more is not
    rl[0], rp[0], hist[0].decode_writes = 100, 100, 40
    cp4 = abi.rswa_checkpoint()
    assert L.rswa_checkpoint_take(cid, p(pl), p(rl), p(rp), hist, 0, C.byref(cp4)) == abi.OK
    rl[0], rp[0], hist[0].decode_writes = 128, 0, 68
    assert L.rswa_rollback_to(cid, p(pl), p(rl), p(rp), hist, 0, W, C.byref(cp4)) == abi.OK
    assert (rl[0], rp[0], hist[0].decode_writes) == (100, 100, 40)
    cp5 = abi.rswa_checkpoint()
    assert L.rswa_checkpoint_take(cid, p(pl), p(rl), p(rp), hist, 0, C.byref(cp5)) == abi.OK
    rl[0], rp[0], hist[0].decode_writes = 128, 1, 69
    assert L.rswa_rollback_to(cid, p(pl), p(rl), p(rp), hist, 0, W, C.byref(cp5)) == abi.ESTATE


def test_rswa_verify_and_mirror_host_validation(abi):
    """rswa_verify(_i8), the mirrored writers and the workspace sizes refuse bad
    arguments on the host (nothing is launched or changed)."""
    L = abi.lib()
    B, H, hd, W, ref_cap = 2, 10, 128, 128, 64
    p = lambda a: C.c_void_p(a.ctypes.data)
    fake = C.c_void_p(1 << 20)  # never dereferenced
    n = C.c_int64(0)
    assert L.rswa_verify_workspace_bytes(B, H, hd, ref_cap, W, 4, C.byref(n)) == abi.OK and n.value > 0
    n1 = C.c_int64(0)
    assert L.rswa_verify_workspace_bytes(B, H, hd, ref_cap, W, 1, C.byref(n1)) == abi.OK and n1.value < n.value
    for K in (0, 17):
        assert L.rswa_verify_workspace_bytes(B, H, hd, ref_cap, W, K, C.byref(n1)) == abi.EINVAL
    assert L.rswa_verify_workspace_bytes(B, H, 96, ref_cap, W, 4, C.byref(n1)) == abi.EINVAL
    pl = np.array([-1, 5], np.int32)
    rl = np.zeros(B, np.int32)
    rp = np.zeros(B, np.int32)
    ws = C.c_void_p(1 << 21)
    args = (p(pl), p(rl), p(rp), B, H, hd, ref_cap, W, C.c_float(0.088), fake, ws, n.value, None)
    # a stream without prefill: the verify would have to write into it
    assert L.rswa_verify(fake, fake, fake, 4, fake, fake, fake, fake, *args) == abi.ESTATE
    pl[0] = 3
    assert L.rswa_verify(fake, fake, fake, 17, fake, fake, fake, fake, *args) == abi.EINVAL
    assert L.rswa_verify(fake, None, fake, 4, fake, fake, fake, fake, *args) == abi.EINVAL
    small = (p(pl), p(rl), p(rp), B, H, hd, ref_cap, W, C.c_float(0.088), fake, ws, 256, None)
    assert L.rswa_verify(fake, fake, fake, 4, fake, fake, fake, fake, *small) == abi.EINVAL
    # the int8 entry points need a complete, aligned mirror
    assert L.rswa_verify_i8(fake, fake, fake, 4, None, *args) == abi.EINVAL
    m = abi.rswa_i8_mirror(fake.value, fake.value, fake.value, fake.value, fake.value, fake.value, fake.value, None)
    assert L.rswa_verify_i8(fake, fake, fake, 4, C.byref(m), *args) == abi.EINVAL
    assert L.rswa_decode_i8(fake, C.byref(m), *args) == abi.EINVAL
    hist = (abi.rswa_history * B)()
    assert L.rswa_ring_write_i8(fake, fake, C.byref(m), fake, fake, p(pl), p(rl), p(rp), hist, B, H, hd, W,
                                None, None) == abi.EINVAL
    assert rl.tolist() == [0, 0] and hist[0].decode_writes == 0
    assert L.rswa_record_prefill_i8(fake, fake, None, fake, fake, 0, 4, B, H, hd, ref_cap, W, p(pl), p(rl), p(rp),
                                    hist, None) == abi.EINVAL
    assert pl.tolist() == [3, 5] and hist[0].lineage_epoch == 0


def test_failure_injection_hook_arms_and_disarms(abi):
    """kvd_test_fail_after is host-only: arming and disarming it needs no
    device (the GPU tests make calls fail with it)."""
    lib = abi.lib()
    assert lib.kvd_test_fail_after(3) == abi.OK
    assert lib.kvd_test_fail_after(-1) == abi.OK
