"""Writes stay inside the buffers a call is given.

Every device buffer a call writes -- its workspace (exactly the size the
library reports), its output, the imp accumulator -- is handed over as the
middle of a larger allocation whose 4 KB guard bands on both sides hold a
fixed byte pattern; after the call the bands must be untouched.  This is the
stand-in for a memory checker on this hardware: it catches a write past the
end (or before the start) of a scratch region that parity alone could miss,
on both split paths (tensor-core q8_2f kernels at 4, 8 and 16 heads per group,
the CUDA-core kernel for the other modes), with imp on and off, for the
query-batched verify, Born eviction and the R-SWA decode and verify.  The
results are also compared with the same call on plainly allocated buffers
(bitwise: every kernel is deterministic).
"""

import ctypes as C
import math

import pytest

from helpers import gpu_append_bulk, seq_rows

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def env():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300.build import build

    build()
    return torch, kvd


class Guarded:
    """`nbytes` usable bytes between two guard bands of PATTERN."""

    def __init__(self, torch, nbytes, fill=0):
        self.torch = torch
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.mid = self.buf[GUARD:GUARD + self.n]
        self.mid.fill_(fill)

    def f32(self, shape):
        return self.mid.view(self.torch.float32).view(*shape)

    def intact(self):
        return bool((self.buf[:GUARD] == PATTERN).all()) and bool((self.buf[GUARD + self.n:] == PATTERN).all())


def _layer(torch, kvd, mode, lengths, n_kv, hd, alive, seed):
    ks, vs = seq_rows(lengths, n_kv, hd, seed)
    layer = kvd.LayerKvCache(len(lengths), n_kv, hd, mode, [max(L, 1) + 8 for L in lengths], alive=alive)
    gpu_append_bulk(layer, ks, vs, torch)
    return layer


@pytest.mark.parametrize("mode,hd,hpk", [("q8", 128, 4), ("q8", 128, 8), ("q8", 128, 16), ("f32", 64, 4),
                                         ("q8k", 128, 2), ("q8v", 128, 16)])
@pytest.mark.parametrize("with_imp", [False, True])
def test_decode_writes_stay_in_workspace_out_and_imp(env, mode, hd, hpk, with_imp):
    torch, kvd = env
    n_kv, lengths = 2, [700, 0, 2100, 65, 1]
    layer = _layer(torch, kvd, mode, lengths, n_kv, hd, [1, 0] if hpk != 16 else [1, 1], seed=hpk + hd)
    n_q = n_kv * hpk
    q = torch.randn(len(lengths), n_q, hd, device="cuda")
    need = layer.workspace_bytes(n_q, with_imp)
    ws = Guarded(torch, need)
    out = Guarded(torch, len(lengths) * n_q * hd * 4, fill=0xFF)
    imp = Guarded(torch, layer.imp_len * 4) if with_imp else None
    kvd.decode_attention(q, layer, out=out.f32((len(lengths), n_q, hd)), imp=imp.f32((layer.imp_len,)) if imp else None,
                         workspace=ws.mid)
    imp_ref = torch.zeros(layer.imp_len, device="cuda") if with_imp else None
    ref = kvd.decode_attention(q, layer, imp=imp_ref)
    torch.cuda.synchronize()
    assert ws.intact() and out.intact() and (imp is None or imp.intact())
    assert torch.equal(out.f32((len(lengths), n_q, hd)), ref)
    if with_imp:
        assert torch.equal(imp.f32((layer.imp_len,)), imp_ref)
    assert layer.device_error() == 0


@pytest.mark.parametrize("mode,hd,hg", [("q8", 128, 4), ("f32", 64, 2)])
def test_verify_writes_stay_in_workspace_and_out(env, mode, hd, hg):
    torch, kvd = env
    from kv_cache_decode_attention_gb300 import _abi

    n_kv, lengths, K = 2, [600, 3, 1500], 4
    layer = _layer(torch, kvd, mode, lengths, n_kv, hd, [1, 1], seed=hd + K)
    n_q = n_kv * hg
    q = torch.randn(len(lengths), K, n_q, hd, device="cuda")
    n = C.c_int64(0)
    _abi.call("kvd_verify_workspace_bytes", C.byref(layer.L), n_q, K, C.byref(n))
    ws = Guarded(torch, n.value)
    out = Guarded(torch, q.numel() * 4, fill=0xFF)
    kvd.decode_attention_verify(q, layer, K, out=out.f32(q.shape), workspace=ws.mid)
    ref = kvd.decode_attention_verify(q, layer, K)
    torch.cuda.synchronize()
    assert ws.intact() and out.intact()
    assert torch.equal(out.f32(q.shape), ref)
    assert layer.device_error() == 0


@pytest.mark.parametrize("mode", ["q8", "f32"])
def test_eviction_writes_stay_in_workspace_and_imp(env, mode):
    torch, kvd = env
    from kv_cache_decode_attention_gb300 import _abi

    n_kv, hd, lengths, keep = 2, 128, [900, 40, 3000], 256
    layer = _layer(torch, kvd, mode, lengths, n_kv, hd, [1, 1], seed=17)
    imp = Guarded(torch, layer.imp_len * 4)
    imp.f32((layer.imp_len,)).copy_(torch.rand(layer.imp_len, device="cuda"))
    n = C.c_int64(0)
    _abi.call("kv_evict_workspace_bytes", C.byref(layer.L), keep, C.byref(n))
    ws = Guarded(torch, max(int(n.value), 256))
    kvd.kv_evict_born(layer, imp.f32((layer.imp_len,)), keep, workspace=ws.mid)
    torch.cuda.synchronize()
    assert ws.intact() and imp.intact()
    assert [layer.seq_len(b) for b in range(3)] == [min(L, keep) for L in lengths]
    assert layer.device_error() == 0


@pytest.mark.parametrize("int8", [False, True])
def test_rswa_writes_stay_in_workspace_and_out(env, int8):
    torch, kvd = env
    from kv_cache_decode_attention_gb300 import _abi

    B, H, hd, ref_cap, W = 3, 2, 128, 640, 16
    cache = kvd.RingCache(B, ref_cap, H, hd, W, int8=int8)
    for s, pl in enumerate([600, 33, 640]):
        kvd.rswa_record_prefill(cache, s, torch.randn(H, pl, hd, device="cuda"),
                                torch.randn(H, pl, hd, device="cuda"))
    for _ in range(21):  # the ring wraps
        kvd.rswa_ring_write(cache, torch.randn(B, H, hd, device="cuda"), torch.randn(B, H, hd, device="cuda"))
    q = torch.randn(B, H, hd, device="cuda")
    ref = (kvd.rswa_decode_i8 if int8 else kvd.rswa_decode)(q, cache)
    plain_ws = cache.workspace
    ws = Guarded(torch, plain_ws.numel())
    cache.workspace = ws.mid
    out = Guarded(torch, B * H * hd * 4, fill=0xFF)
    (kvd.rswa_decode_i8 if int8 else kvd.rswa_decode)(q, cache, out=out.f32((B, H * hd)))
    torch.cuda.synchronize()
    assert ws.intact() and out.intact()
    assert torch.equal(out.f32((B, H * hd)), ref)
    assert cache.device_error() == 0
    cache.workspace = plain_ws

    # the read-only verify of K drafts, straight through the C ABI
    K = 3
    qv, dk, dv = (torch.randn(B, K, H, hd, device="cuda") for _ in range(3))
    n = C.c_int64(0)
    _abi.call("rswa_verify_workspace_bytes", B, H, hd, ref_cap, W, K, C.byref(n))
    vws = Guarded(torch, n.value)
    vout = Guarded(torch, qv.numel() * 4, fill=0xFF)
    tail = (cache.prefill_len.ctypes.data_as(C.c_void_p), cache.ring_len.ctypes.data_as(C.c_void_p),
            cache.ring_pos.ctypes.data_as(C.c_void_p), B, H, hd, ref_cap, W, C.c_float(1.0 / math.sqrt(hd)),
            C.c_void_p(vout.mid.data_ptr()), C.c_void_p(vws.mid.data_ptr()), int(n.value), None)
    ptr = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
    if int8:
        _abi.call("rswa_verify_i8", ptr(qv), ptr(dk), ptr(dv), K, C.byref(cache.mirror), *tail)
    else:
        _abi.call("rswa_verify", ptr(qv), ptr(dk), ptr(dv), K, ptr(cache.ref_k), ptr(cache.ref_v),
                  ptr(cache.ring_k), ptr(cache.ring_v), *tail)
    vref = kvd.rswa_verify(qv, dk, dv, cache, int8=int8)
    torch.cuda.synchronize()
    assert vws.intact() and vout.intact()
    assert torch.equal(vout.f32((B, K, H * hd)), vref)
