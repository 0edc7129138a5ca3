"""Python binding over the C ABI: torch tensors in, raw device pointers out.

Every computation runs in libkvd.so; this module only allocates the device
buffers the library asks for (torch owns them), marshals pointers, shapes
and the current CUDA stream, and raises on a non-OK status.

Names follow the pages: ``LayerKvCache`` (cortiq kv_cache.rs, batched over
sequences) with ``kv_append``, ``kv_freeze_colfield``, ``decode_attention``;
``RingCache`` (franken_ocr rswa.rs, batched over streams) with
``rswa_record_prefill``, ``rswa_ring_write`` (write_decode_step) and
``rswa_decode``.
"""

from __future__ import annotations

import ctypes as C
import math

import numpy as np
import torch

from . import _abi
from ._abi import F32, Q8, Q8K, Q8V  # noqa: F401

MODE_NAMES = {"f32": F32, "q8": Q8, "q8_2f": Q8, "q8k": Q8K, "q8v": Q8V}


# The current stream's raw handle without building a Stream object (the
# public torch.cuda.current_stream() costs microseconds per call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> C.c_void_p:
    if stream is not None:
        return C.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        return C.c_void_p(_raw_stream(torch.cuda.current_device()))
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: torch.Tensor | None) -> C.c_void_p | None:
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _f32_cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
        raise ValueError("%s must be a contiguous float32 CUDA tensor" % name)
    return t


def _np_ptr(a: np.ndarray) -> C.c_void_p:
    return C.c_void_p(a.ctypes.data)


class LayerKvCache:
    """One layer's KV cache for a batch of sequences (device buffers owned here).

    mode: 'f32' | 'q8' (q8_2f) | 'q8k' | 'q8v' or the integer kvd_mode.
    capacity: rows per sequence (int or per-sequence sequence of ints).
    alive: per-KV-head 0/1 mask (dead heads store nothing), default all alive.
    """

    def __init__(self, n_seq: int, n_kv: int, head_dim: int, mode, capacity, alive=None,
                 device="cuda", stream=None):
        self.mode = MODE_NAMES[mode] if isinstance(mode, str) else int(mode)
        self.n_seq, self.n_kv, self.head_dim = int(n_seq), int(n_kv), int(head_dim)
        cap = np.broadcast_to(np.asarray(capacity, np.int64), (self.n_seq,)).copy()
        self.capacity = cap
        self.alive = (np.ones(self.n_kv, np.uint8) if alive is None
                      else np.ascontiguousarray(alive, dtype=np.uint8))
        sizes = np.zeros(_abi.BUF_COUNT, np.int64)
        host_bytes = C.c_int64(0)
        _abi.call("kvd_layer_bytes", self.n_seq, self.n_kv, self.head_dim, self.mode,
                  _np_ptr(cap), _np_ptr(self.alive), _np_ptr(sizes), C.byref(host_bytes))
        self.buf_bytes = sizes
        self.device = torch.device(device)
        self.bufs = [torch.empty(int(n), dtype=torch.uint8, device=self.device) if n > 0 else None
                     for n in sizes]
        self._ptrs = (C.c_void_p * _abi.BUF_COUNT)(
            *[b.data_ptr() if b is not None else None for b in self.bufs])
        self._host = np.zeros(int(host_bytes.value) + 64, np.uint8)
        self.L = _abi.kvd_layer()
        _abi.call("kvd_layer_init", C.byref(self.L), self.n_seq, self.n_kv, self.head_dim,
                  self.mode, _np_ptr(cap), _np_ptr(self.alive), self._ptrs,
                  _np_ptr(self._host), _stream(stream))
        self.n_live = int(self.alive.astype(bool).sum())
        self.cap16 = (cap + 15) // 16 * 16
        self.row_base = np.concatenate([[0], np.cumsum(self.cap16 * self.n_live)[:-1]]).astype(np.int64)
        self.imp_base = np.concatenate([[0], np.cumsum(self.cap16)[:-1]]).astype(np.int64)
        self.imp_len = int(self.cap16.sum())
        self.live_heads = [h for h in range(self.n_kv) if self.alive[h]]
        self._ws_bytes = {}

    # ---- host-mirrored state -------------------------------------------
    def seq_len(self, b: int) -> int:
        n, f = C.c_int64(0), C.c_int32(0)
        _abi.call("kvd_layer_seq_len", C.byref(self.L), int(b), C.byref(n), C.byref(f))
        return int(n.value)

    def frozen(self, b: int) -> bool:
        n, f = C.c_int64(0), C.c_int32(0)
        _abi.call("kvd_layer_seq_len", C.byref(self.L), int(b), C.byref(n), C.byref(f))
        return bool(f.value)

    def memory_bytes(self) -> int:
        n = C.c_int64(0)
        _abi.call("kvd_layer_memory_bytes", C.byref(self.L), C.byref(n))
        return int(n.value)

    def device_error(self, clear: bool = True) -> int:
        w = C.c_uint32(0)
        st = _abi.lib().kvd_layer_device_error(C.byref(self.L), int(clear), C.byref(w))
        if st not in (_abi.OK, _abi.EDEVICE):
            _abi.check("kvd_layer_device_error", st)
        return int(w.value)

    def wait_timeout_selftest(self, limit_ns: int = 2_000_000, stream=None):
        """Run the bounded-wait path on purpose: one warp waits for a barrier
        phase nothing completes, gives up after limit_ns and sets bit 0 of the
        device error word (read it with device_error() after synchronising)."""
        _abi.call("kvd_wait_timeout_selftest", C.byref(self.L), int(limit_ns), _stream(stream))

    def bounds_selftest(self, stream=None):
        """Run the kernels' metadata guards on purpose: the append, freeze and
        decode split kernels are launched on lengths that put sequence 0 one
        row past its capacity (held in a scratch buffer, not the layer's
        metadata); each guard sets bit 1 of the device error word and returns
        before touching the cache (read it with device_error() after
        synchronising)."""
        n = C.c_int64(0)
        _abi.call("kvd_bounds_selftest_bytes", C.byref(self.L), C.byref(n))
        scratch = torch.empty(int(n.value), dtype=torch.uint8, device=self.device)
        _abi.call("kvd_bounds_selftest", C.byref(self.L), _ptr(scratch), int(scratch.numel()), _stream(stream))
        return scratch  # keep it alive until the launches have run

    def reset(self, seq: int = -1, stream=None):
        _abi.call("kvd_layer_reset", C.byref(self.L), int(seq), _stream(stream))

    def workspace_bytes(self, n_q: int, with_imp: bool) -> int:
        key = (int(n_q), bool(with_imp))
        got = self._ws_bytes.get(key)
        if got is None:  # depends only on the layer's shape: ask the library once
            n = C.c_int64(0)
            _abi.call("kvd_decode_workspace_bytes", C.byref(self.L), key[0], int(key[1]), C.byref(n))
            got = self._ws_bytes[key] = int(n.value)
        return got

    # ---- views of the stored rows (for inspection and tests) ------------
    def region(self, b: int, kv_head: int) -> tuple[int, int]:
        """(first storage row, rows) of sequence b's live KV head `kv_head`."""
        gl = self.live_heads.index(kv_head)
        return int(self.row_base[b] + gl * self.cap16[b]), int(self.cap16[b])

    def component(self, slot: int) -> torch.Tensor | None:
        """Typed view of a row buffer: f32 [rows, hd], int8 [rows, hd], K scales
        [rows, hd/32], V scales [rows], fields [n_seq, n_live, hd]."""
        b = self.bufs[slot]
        if b is None:
            return None
        hd = self.head_dim
        if slot in (_abi.BUF_K, _abi.BUF_V):
            return b.view(torch.float32)[: (b.numel() // 4) // hd * hd].view(-1, hd)
        if slot in (_abi.BUF_KQ, _abi.BUF_VQ):
            return b.view(torch.int8)[: b.numel() // hd * hd].view(-1, hd)
        if slot == _abi.BUF_KS:
            ng = hd // 32
            return b.view(torch.float32)[: (b.numel() // 4) // ng * ng].view(-1, ng)
        if slot == _abi.BUF_VS:
            return b.view(torch.float32)
        if slot in (_abi.BUF_KCOL, _abi.BUF_VCOL):
            n = self.n_seq * self.n_live * hd
            return b.view(torch.float32)[:n].view(self.n_seq, self.n_live, hd)
        return b


def kv_append(layer: LayerKvCache, k: torch.Tensor, v: torch.Tensor, n_new=None, stream=None):
    """Append rows: k, v [sum n_new, n_kv, hd] (or [n_seq, n_kv, hd] with n_new None)."""
    _f32_cuda(k, "k")
    _f32_cuda(v, "v")
    rows = k.numel() // (layer.n_kv * layer.head_dim)
    if n_new is None:
        if rows != layer.n_seq or v.numel() != k.numel():
            raise ValueError("k/v must hold one row per sequence")
        nn = None
    else:
        nn = np.ascontiguousarray(n_new, dtype=np.int32)
        if nn.shape != (layer.n_seq,) or rows != int(nn.sum()) or v.numel() != k.numel():
            raise ValueError("k/v rows must equal sum(n_new)")
    _abi.call("kv_append", C.byref(layer.L), _ptr(k), _ptr(v),
              None if nn is None else _np_ptr(nn), _stream(stream))


def kv_freeze_colfield(layer: LayerKvCache, stream=None):
    _abi.call("kv_freeze_colfield", C.byref(layer.L), _stream(stream))


def decode_attention_verify(q: torch.Tensor, cache: LayerKvCache, K: int, out: torch.Tensor | None = None,
                            scale: float | None = None, window: int = 0, softcap: float = 0.0,
                            sinks: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Query-batched verify of the last K rows (drafts already appended): q and out
    [n_seq, K, n_q, hd]; query k attends up to and including draft k."""
    _f32_cuda(q, "q")
    n_q = q.numel() // (cache.n_seq * K * cache.head_dim)
    if n_q * cache.n_seq * K * cache.head_dim != q.numel():
        raise ValueError("q must be [n_seq, K, n_q, head_dim]")
    if out is None:
        out = torch.empty(cache.n_seq, K, n_q, cache.head_dim, device=q.device)
    _f32_cuda(out, "out")
    if scale is None:
        scale = 1.0 / math.sqrt(cache.head_dim)
    if sinks is not None:
        _f32_cuda(sinks, "sinks")
        if sinks.numel() != n_q:
            raise ValueError("sinks must hold one logit per query head (%d)" % n_q)
    if workspace is None:
        n = C.c_int64(0)
        _abi.call("kvd_verify_workspace_bytes", C.byref(cache.L), int(n_q), int(K), C.byref(n))
        workspace = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=q.device)
    _abi.call("decode_attention_verify", _ptr(q), C.byref(cache.L), int(n_q), int(K), C.c_float(scale),
              int(window), C.c_float(softcap), _ptr(sinks), _ptr(out), _ptr(workspace),
              int(workspace.numel()), _stream(stream))
    return out


def kv_truncate_last(layer: LayerKvCache, n_drop=1, imp: torch.Tensor | None = None, stream=None):
    """cortiq truncate_last: drop the last n_drop rows of every sequence (an int for
    all, or one count per sequence); with imp, the dropped rows' masses are cleared."""
    counts = np.broadcast_to(np.asarray(n_drop, np.int32), (layer.n_seq,)).copy()
    if imp is not None:
        _f32_cuda(imp, "imp")
        if imp.numel() < layer.imp_len:
            raise ValueError("imp must hold %d floats" % layer.imp_len)
    _abi.call("kv_truncate_last", C.byref(layer.L), _np_ptr(counts), _ptr(imp) if imp is not None else None,
              _stream(stream))


def kv_evict_born(layer: LayerKvCache, imp: torch.Tensor, keep_last: int, sink: int = 4,
                  recent: int | None = None, workspace: torch.Tensor | None = None, stream=None):
    """cortiq evict_born on every sequence holding more than keep_last rows: keep the
    sinks, the recents and the middle rows of highest mass in imp (the buffer
    decode_attention accumulates), gathered in row order in every storage.  With
    recent=None it is cortiq KvCache::evict's Born rule, recent = max(keep_last // 2, 1)."""
    _f32_cuda(imp, "imp")
    if imp.numel() < layer.imp_len:
        raise ValueError("imp must hold %d floats" % layer.imp_len)
    if recent is None:
        recent = max(int(keep_last) // 2, 1)
    n = C.c_int64(0)
    _abi.call("kv_evict_workspace_bytes", C.byref(layer.L), int(keep_last), C.byref(n))
    if workspace is None:
        workspace = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=imp.device)
    _abi.call("kv_evict_born", C.byref(layer.L), _ptr(imp), int(keep_last), int(sink), int(recent),
              _ptr(workspace), int(workspace.numel()), _stream(stream))


def decode_attention(q: torch.Tensor, cache: LayerKvCache, out: torch.Tensor | None = None,
                     imp: torch.Tensor | None = None, scale: float | None = None,
                     workspace: torch.Tensor | None = None, stream=None, window: int = 0,
                     softcap: float = 0.0, sinks: torch.Tensor | None = None) -> torch.Tensor:
    """q [n_seq, n_q, hd] -> out [n_seq, n_q, hd]; imp (float32 [imp_len]) accumulates.

    window > 0 keeps each sequence's last `window` rows; softcap > 0 caps the
    scores as softcap * tanh(s / softcap); sinks (float32 [n_q]) adds one
    learned sink logit per query head to the softmax (decode_attention_ex)."""
    _f32_cuda(q, "q")
    n_q = q.numel() // (cache.n_seq * cache.head_dim)
    if q.numel() != cache.n_seq * n_q * cache.head_dim:
        raise ValueError("q must be [n_seq, n_q, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    _f32_cuda(out, "out")
    if imp is not None:
        _f32_cuda(imp, "imp")
        if imp.numel() < cache.imp_len:
            raise ValueError("imp must hold %d floats" % cache.imp_len)
    need = cache.workspace_bytes(n_q, imp is not None)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(cache.head_dim)
    if window or softcap or sinks is not None:
        if sinks is not None:
            _f32_cuda(sinks, "sinks")
            if sinks.numel() != n_q:
                raise ValueError("sinks must hold one logit per query head (%d)" % n_q)
        _abi.call("decode_attention_ex", _ptr(q), C.byref(cache.L), int(n_q), C.c_float(scale),
                  int(window), C.c_float(softcap), _ptr(sinks), _ptr(out), _ptr(imp), _ptr(workspace),
                  int(workspace.numel()), _stream(stream))
    else:
        _abi.call("decode_attention", _ptr(q), C.byref(cache.L), int(n_q), C.c_float(scale),
                  _ptr(out), _ptr(imp), _ptr(workspace), int(workspace.numel()), _stream(stream))
    return out


def decode_attention_static(q: torch.Tensor, cache: LayerKvCache, out: torch.Tensor | None = None,
                            scale: float | None = None, stream=None) -> torch.Tensor:
    """decode_attention without imp and without a workspace, for callers that
    cannot allocate device memory on their decode path: the library's own
    16 MiB scratch array holds the partial results.  Raises KvdError with
    status -2 when the call needs more scratch than that.  Calls that overlap
    on the GPU share the array and must be serialised."""
    _f32_cuda(q, "q")
    n_q = q.numel() // (cache.n_seq * cache.head_dim)
    if q.numel() != cache.n_seq * n_q * cache.head_dim:
        raise ValueError("q must be [n_seq, n_q, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    _f32_cuda(out, "out")
    if scale is None:
        scale = 1.0 / math.sqrt(cache.head_dim)
    _abi.call("decode_attention_static", _ptr(q), C.byref(cache.L), int(n_q), C.c_float(scale),
              _ptr(out), _stream(stream))
    return out


class RingCache:
    """R-SWA caches of B streams for one layer: reference block [B, H, ref_cap, hd]
    plus a W-slot ring [B, H, W, hd], cursors on the host.  With int8=True an
    int8 mirror (rswa Int8Kv: codes of the same shapes, one f32 scale per row)
    is kept beside the f32 regions and written by the same calls."""

    _next_id = 0

    def __init__(self, B: int, ref_cap: int, H: int = 10, head_dim: int = 128, W: int = 128,
                 device="cuda", int8: bool = False):
        self.B, self.H, self.head_dim, self.W, self.ref_cap = B, H, head_dim, W, ref_cap
        dev = torch.device(device)
        self.ref_k = torch.zeros(B, H, ref_cap, head_dim, device=dev)
        self.ref_v = torch.zeros(B, H, ref_cap, head_dim, device=dev)
        self.ring_k = torch.zeros(B, H, W, head_dim, device=dev)
        self.ring_v = torch.zeros(B, H, W, head_dim, device=dev)
        self.mirror = None
        if int8:
            i8 = dict(dtype=torch.int8, device=dev)
            self.ref_k8 = torch.zeros(B, H, ref_cap, head_dim, **i8)
            self.ref_v8 = torch.zeros(B, H, ref_cap, head_dim, **i8)
            self.ring_k8 = torch.zeros(B, H, W, head_dim, **i8)
            self.ring_v8 = torch.zeros(B, H, W, head_dim, **i8)
            self.ref_ks = torch.zeros(B, H, ref_cap, device=dev)
            self.ref_vs = torch.zeros(B, H, ref_cap, device=dev)
            self.ring_ks = torch.zeros(B, H, W, device=dev)
            self.ring_vs = torch.zeros(B, H, W, device=dev)
            self.mirror = _abi.rswa_i8_mirror(
                _ptr(self.ref_k8), _ptr(self.ref_v8), _ptr(self.ref_ks), _ptr(self.ref_vs),
                _ptr(self.ring_k8), _ptr(self.ring_v8), _ptr(self.ring_ks), _ptr(self.ring_vs))
        self.prefill_len = np.full(B, -1, np.int32)
        self.ring_len = np.zeros(B, np.int32)
        self.ring_pos = np.zeros(B, np.int32)
        # decode-write counts and branch lineages (checkpoint / rollback)
        self.history = (_abi.rswa_history * B)()
        RingCache._next_id += 1
        self.cache_id = RingCache._next_id
        n = C.c_int64(0)
        _abi.call("rswa_decode_workspace_bytes", B, H, head_dim, ref_cap, W, C.byref(n))
        self.workspace = torch.zeros(int(n.value), dtype=torch.uint8, device=dev)

    def checkpoint(self, s: int):
        """rswa RingCache::checkpoint of stream s (cursors only, no K/V copy)."""
        cp = _abi.rswa_checkpoint()
        _abi.call("rswa_checkpoint_take", self.cache_id, _np_ptr(self.prefill_len), _np_ptr(self.ring_len),
                  _np_ptr(self.ring_pos), self.history, int(s), C.byref(cp))
        return cp

    def rollback_to(self, s: int, cp) -> None:
        """rswa RingCache::rollback_to: discard stream s's ring writes since cp
        (KvdError with status -3, nothing changed, when the page refuses it)."""
        _abi.call("rswa_rollback_to", self.cache_id, _np_ptr(self.prefill_len), _np_ptr(self.ring_len),
                  _np_ptr(self.ring_pos), self.history, int(s), self.W, C.byref(cp))

    def device_error(self, clear: bool = True) -> int:
        w = C.c_uint32(0)
        st = _abi.lib().rswa_device_error(_ptr(self.workspace), int(clear), C.byref(w))
        if st not in (_abi.OK, _abi.EDEVICE):
            _abi.check("rswa_device_error", st)
        return int(w.value)


def rswa_record_prefill(cache: RingCache, s: int, k: torch.Tensor, v: torch.Tensor, stream=None):
    """Record stream s's prefill k, v [H, seq, hd] as its reference block."""
    _f32_cuda(k, "k")
    _f32_cuda(v, "v")
    seq = k.numel() // (cache.H * cache.head_dim)
    if k.numel() != cache.H * seq * cache.head_dim or v.numel() != k.numel():
        raise ValueError("prefill k/v must be [H, seq, head_dim]")
    args = (int(s), int(seq), cache.B, cache.H, cache.head_dim, cache.ref_cap, cache.W,
            _np_ptr(cache.prefill_len), _np_ptr(cache.ring_len), _np_ptr(cache.ring_pos),
            cache.history, _stream(stream))
    if cache.mirror is not None:
        _abi.call("rswa_record_prefill_i8", _ptr(cache.ref_k), _ptr(cache.ref_v), C.byref(cache.mirror),
                  _ptr(k), _ptr(v), *args)
    else:
        _abi.call("rswa_record_prefill", _ptr(cache.ref_k), _ptr(cache.ref_v), _ptr(k), _ptr(v), *args)


def rswa_ring_write(cache: RingCache, k: torch.Tensor, v: torch.Tensor, stream=None) -> np.ndarray:
    """write_decode_step for every stream: k, v [B, H, hd]; returns the slots written."""
    _f32_cuda(k, "k")
    _f32_cuda(v, "v")
    if k.numel() != cache.B * cache.H * cache.head_dim or v.numel() != k.numel():
        raise ValueError("k/v must be [B, H, head_dim]")
    slots = np.zeros(cache.B, np.int32)
    args = (_ptr(k), _ptr(v), _np_ptr(cache.prefill_len), _np_ptr(cache.ring_len),
            _np_ptr(cache.ring_pos), cache.history, cache.B, cache.H, cache.head_dim, cache.W,
            _np_ptr(slots), _stream(stream))
    if cache.mirror is not None:
        _abi.call("rswa_ring_write_i8", _ptr(cache.ring_k), _ptr(cache.ring_v), C.byref(cache.mirror),
                  *args)
    else:
        _abi.call("rswa_ring_write", _ptr(cache.ring_k), _ptr(cache.ring_v), *args)
    return slots


def rswa_decode(q: torch.Tensor, cache: RingCache, out: torch.Tensor | None = None,
                scale: float | None = None, stream=None) -> torch.Tensor:
    """q [B, H, hd] -> out [B, H * hd]: softmax over reference ++ ring per head."""
    _f32_cuda(q, "q")
    if q.numel() != cache.B * cache.H * cache.head_dim:
        raise ValueError("q must be [B, H, head_dim]")
    if out is None:
        out = torch.empty(cache.B, cache.H * cache.head_dim, device=q.device)
    _f32_cuda(out, "out")
    if scale is None:
        scale = 1.0 / math.sqrt(cache.head_dim)
    _abi.call("rswa_decode", _ptr(q), _ptr(cache.ref_k), _ptr(cache.ref_v), _ptr(cache.ring_k),
              _ptr(cache.ring_v), _np_ptr(cache.prefill_len), _np_ptr(cache.ring_len),
              _np_ptr(cache.ring_pos), cache.B, cache.H, cache.head_dim, cache.ref_cap, cache.W,
              C.c_float(scale), _ptr(out), _ptr(cache.workspace), int(cache.workspace.numel()),
              _stream(stream))
    return out


def rswa_decode_i8(q: torch.Tensor, cache: RingCache, out: torch.Tensor | None = None,
                   scale: float | None = None, stream=None) -> torch.Tensor:
    """rswa decode_attention_int8: q [B, H, hd] -> out [B, H * hd] over the int8
    mirror (the cache must have been built with int8=True)."""
    if cache.mirror is None:
        raise ValueError("rswa_decode_i8 needs a RingCache built with int8=True")
    _f32_cuda(q, "q")
    if q.numel() != cache.B * cache.H * cache.head_dim:
        raise ValueError("q must be [B, H, head_dim]")
    if out is None:
        out = torch.empty(cache.B, cache.H * cache.head_dim, device=q.device)
    _f32_cuda(out, "out")
    if scale is None:
        scale = 1.0 / math.sqrt(cache.head_dim)
    _abi.call("rswa_decode_i8", _ptr(q), C.byref(cache.mirror), _np_ptr(cache.prefill_len),
              _np_ptr(cache.ring_len), _np_ptr(cache.ring_pos), cache.B, cache.H, cache.head_dim,
              cache.ref_cap, cache.W, C.c_float(scale), _ptr(out), _ptr(cache.workspace),
              int(cache.workspace.numel()), _stream(stream))
    return out


def rswa_verify(q: torch.Tensor, draft_k: torch.Tensor, draft_v: torch.Tensor, cache: RingCache,
                int8: bool = False, out: torch.Tensor | None = None, scale: float | None = None,
                stream=None) -> torch.Tensor:
    """rswa verify_attention: K draft tokens q, draft_k, draft_v [B, K, H, hd] ->
    out [B, K, H * hd], query i as after writing drafts 0..i -- the cache is not
    written.  int8=True reads the int8 mirror (decode_attention_int8)."""
    for t, name in ((q, "q"), (draft_k, "draft_k"), (draft_v, "draft_v")):
        _f32_cuda(t, name)
    K = q.numel() // (cache.B * cache.H * cache.head_dim)
    if K * cache.B * cache.H * cache.head_dim != q.numel() or draft_k.numel() != q.numel() or \
            draft_v.numel() != q.numel():
        raise ValueError("q, draft_k, draft_v must be [B, K, H, head_dim]")
    if int8 and cache.mirror is None:
        raise ValueError("int8 verify needs a RingCache built with int8=True")
    if out is None:
        out = torch.empty(cache.B, K, cache.H * cache.head_dim, device=q.device)
    _f32_cuda(out, "out")
    if scale is None:
        scale = 1.0 / math.sqrt(cache.head_dim)
    n = C.c_int64(0)
    _abi.call("rswa_verify_workspace_bytes", cache.B, cache.H, cache.head_dim, cache.ref_cap, cache.W, int(K),
              C.byref(n))
    ws = torch.empty(int(n.value), dtype=torch.uint8, device=q.device)
    tail = (_np_ptr(cache.prefill_len), _np_ptr(cache.ring_len), _np_ptr(cache.ring_pos), cache.B, cache.H,
            cache.head_dim, cache.ref_cap, cache.W, C.c_float(scale), _ptr(out), _ptr(ws), int(ws.numel()),
            _stream(stream))
    if int8:
        _abi.call("rswa_verify_i8", _ptr(q), _ptr(draft_k), _ptr(draft_v), int(K), C.byref(cache.mirror), *tail)
    else:
        _abi.call("rswa_verify", _ptr(q), _ptr(draft_k), _ptr(draft_v), int(K), _ptr(cache.ref_k),
                  _ptr(cache.ref_v), _ptr(cache.ring_k), _ptr(cache.ring_v), *tail)
    return out


def rswa_attention(cache: RingCache, q, k, v, stream=None) -> torch.Tensor:
    """rswa attention(): write this step's K/V into every ring, then attend (the
    query sees itself as the newest ring row)."""
    rswa_ring_write(cache, k, v, stream)
    return rswa_decode(q, cache, stream=stream)
