"""ctypes binding of the C oracle (test infrastructure only; see package doc).

Every function here marshals numpy arrays into ``kvd_oracle.c`` and back;
none of the method's arithmetic is repeated in Python.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

F32, Q8, Q8K, Q8V = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvd_oracle.c")
_SO = os.path.join(_HERE, "_kvd_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile kvd_oracle.c into _kvd_oracle.so beside it (gcc, no FMA contraction)."""
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + ".tmp.%d" % os.getpid()
        cmd = [
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-o", tmp, _SRC, "-lm",
        ]
        # OpenMP only shares the multi-sequence decode's (sequence, head) pairs
        # among threads; without it the same code runs on one thread
        if subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True).returncode != 0:
            subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class _Cache(C.Structure):
    _fields_ = [
        ("mode", C.c_int32), ("n_kv", C.c_int32), ("hd", C.c_int32), ("cap", C.c_int32),
        ("alive", C.c_void_p), ("seq_len", C.c_int32), ("head_rows", C.c_void_p),
        ("kcol_set", C.c_void_p), ("vcol_set", C.c_void_p),
        ("k", C.c_void_p), ("v", C.c_void_p), ("kq", C.c_void_p), ("vq", C.c_void_p),
        ("ks", C.c_void_p), ("vs", C.c_void_p), ("kcol", C.c_void_p), ("vcol", C.c_void_p),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build_oracle())
            vp, i32, f32 = C.c_void_p, C.c_int, C.c_float
            L.kvo_quant_row.argtypes = [vp, vp, i32, i32, vp, vp]
            L.kvo_quant_row.restype = None
            L.kvo_quantize_row_i8.argtypes = [vp, i32, vp]
            L.kvo_quantize_row_i8.restype = f32
            L.kvo_quantize_rows_i8.argtypes = [vp, C.c_longlong, i32, vp, vp]
            L.kvo_quantize_rows_i8.restype = None
            L.kvo_needs_freeze.argtypes = [C.POINTER(_Cache)]
            L.kvo_freeze.argtypes = [C.POINTER(_Cache)]
            L.kvo_freeze.restype = None
            L.kvo_append.argtypes = [C.POINTER(_Cache), vp, vp]
            L.kvo_row.argtypes = [C.POINTER(_Cache), i32, i32, i32, vp]
            L.kvo_row.restype = None
            L.kvo_attend_head.argtypes = [C.POINTER(_Cache), vp, i32, f32, vp, vp]
            L.kvo_attend_group.argtypes = [C.POINTER(_Cache), vp, i32, i32, f32, vp, vp]
            L.kvo_attend_group_ex.argtypes = [C.POINTER(_Cache), vp, i32, i32, f32, i32, f32, C.c_longlong,
                                              vp, vp,
                                              vp]
            L.kvo_evict_born.argtypes = [C.POINTER(_Cache), vp, i32, i32, i32]
            L.kvo_truncate_last.argtypes = [C.POINTER(_Cache), vp, i32]
            L.kvo_memory_bytes.argtypes = [C.POINTER(_Cache)]
            L.kvo_memory_bytes.restype = C.c_longlong
            L.kvo_rswa_write.argtypes = [i32, i32, i32, vp, vp, vp, vp, i32, vp, vp]
            L.kvo_rswa_decode.argtypes = [i32, i32, vp, vp, vp, C.c_longlong, i32, vp, vp,
                                          i32, i32, f32, vp]
            L.kvo_rswa_decode_i8.argtypes = [i32, i32, vp, vp, vp, vp, vp, C.c_longlong, i32, vp, vp,
                                             vp, vp, i32, i32, f32, vp]
            L.kvo_decode_many.argtypes = [vp, i32, vp, i32, f32, vp, vp, i32]
            L.kvo_online_head.argtypes = [i32, i32, vp, vp, vp, f32, vp]
            L.kvo_online_head.restype = None
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


K_GROUP = None
COL_WARMUP = None


def _init_consts():
    global K_GROUP, COL_WARMUP
    L = lib()
    K_GROUP = int(L.kvo_k_group())
    COL_WARMUP = int(L.kvo_col_warmup())


_init_consts()


def quant_row(x, col=None, group=None):
    """cortiq quant_row on one f32 row: returns (codes int8[n], scales f32[ceil(n/group)])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[0]
    group = n if group is None else group
    q = np.zeros(n, np.int8)
    s = np.zeros((n + group - 1) // group, np.float32)
    colp = None if col is None else np.ascontiguousarray(col, dtype=np.float32)
    lib().kvo_quant_row(_p(x), _p(colp), n, group, _p(q), _p(s))
    return q, s


def quantize_row_i8(x):
    """rswa quantize_row_i8 on one f32 row: returns (codes int8[n], scale f32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.zeros(x.shape[0], np.int8)
    s = lib().kvo_quantize_row_i8(_p(x), x.shape[0], _p(q))
    return q, np.float32(s)


class OracleSeqCache:
    """One sequence's cache for one layer (cortiq LayerKvCache), oracle side."""

    def __init__(self, mode: int, n_kv: int, hd: int, cap: int, alive=None):
        self.mode, self.n_kv, self.hd, self.cap = mode, n_kv, hd, cap
        ng = (hd + K_GROUP - 1) // K_GROUP
        self.alive = np.ones(n_kv, np.uint8) if alive is None else np.asarray(alive, np.uint8).copy()
        self.head_rows = np.zeros(n_kv, np.int32)
        self.kcol_set = np.zeros(n_kv, np.uint8)
        self.vcol_set = np.zeros(n_kv, np.uint8)
        qk = mode in (Q8, Q8K)
        qv = mode in (Q8, Q8V)
        self.k = None if qk else np.zeros((n_kv, cap, hd), np.float32)
        self.v = None if qv else np.zeros((n_kv, cap, hd), np.float32)
        self.kq = np.zeros((n_kv, cap, hd), np.int8) if qk else None
        self.ks = np.zeros((n_kv, cap, ng), np.float32) if qk else None
        self.vq = np.zeros((n_kv, cap, hd), np.int8) if qv else None
        self.vs = np.zeros((n_kv, cap), np.float32) if qv else None
        self.kcol = np.ones((n_kv, hd), np.float32)
        self.vcol = np.ones((n_kv, hd), np.float32)
        self._s = _Cache()
        s = self._s
        s.mode, s.n_kv, s.hd, s.cap = mode, n_kv, hd, cap
        s.alive, s.seq_len, s.head_rows = _p(self.alive), 0, _p(self.head_rows)
        s.kcol_set, s.vcol_set = _p(self.kcol_set), _p(self.vcol_set)
        s.k, s.v, s.kq, s.vq = _p(self.k), _p(self.v), _p(self.kq), _p(self.vq)
        s.ks, s.vs, s.kcol, s.vcol = _p(self.ks), _p(self.vs), _p(self.kcol), _p(self.vcol)

    @property
    def seq_len(self) -> int:
        return int(self._s.seq_len)

    @property
    def frozen(self) -> bool:
        return bool(self.kcol_set.any() or self.vcol_set.any())

    def append(self, k_new, v_new):
        k_new = np.ascontiguousarray(k_new, dtype=np.float32).reshape(self.n_kv * self.hd)
        v_new = np.ascontiguousarray(v_new, dtype=np.float32).reshape(self.n_kv * self.hd)
        rc = lib().kvo_append(C.byref(self._s), _p(k_new), _p(v_new))
        if rc != 0:
            raise ValueError("oracle append: capacity exhausted")

    def append_rows(self, k_rows, v_rows):
        """Append rows one at a time: k_rows, v_rows are [n, n_kv, hd]."""
        for i in range(k_rows.shape[0]):
            self.append(k_rows[i], v_rows[i])

    def needs_freeze(self) -> bool:
        return bool(lib().kvo_needs_freeze(C.byref(self._s)))

    def freeze(self):
        lib().kvo_freeze(C.byref(self._s))

    def freeze_if_due(self):
        if self.needs_freeze():
            self.freeze()

    def row(self, h: int, p: int, which_v: bool) -> np.ndarray:
        out = np.zeros(self.hd, np.float64)
        lib().kvo_row(C.byref(self._s), h, p, int(which_v), _p(out))
        return out

    def dequant(self, h: int, which_v: bool) -> np.ndarray:
        n = int(self.head_rows[h])
        return np.stack([self.row(h, p, which_v) for p in range(n)]) if n else np.zeros((0, self.hd))

    def attend_head(self, q, kv_head: int, scale: float):
        q = np.ascontiguousarray(q, dtype=np.float32)
        out = np.zeros(self.hd, np.float64)
        probs = np.zeros(max(self.cap, 1), np.float64)
        n = lib().kvo_attend_head(C.byref(self._s), _p(q), kv_head, scale, _p(out), _p(probs))
        return out, probs[:n]

    def attend_group(self, q_group, kv_head: int, scale: float, imp=None):
        q_group = np.ascontiguousarray(q_group, dtype=np.float32)
        nheads = q_group.size // self.hd
        out = np.zeros((nheads, self.hd), np.float64)
        if imp is not None:
            assert imp.dtype == np.float64 and imp.flags.c_contiguous
        lib().kvo_attend_group(C.byref(self._s), _p(q_group), kv_head, nheads, scale,
                               _p(out), _p(imp))
        return out

    def attend_group_ex(self, q_group, kv_head: int, scale: float, first: int = 0,
                        softcap: float = 0.0, sinks=None, imp=None, upto: int = -1):
        """attend_group with a first visible row, logit soft-capping, learned
        sink logits (one per head of the group, or None) and the causal limit
        upto (rows [0, upto) only; -1 = all rows)."""
        q_group = np.ascontiguousarray(q_group, dtype=np.float32)
        nheads = q_group.size // self.hd
        out = np.zeros((nheads, self.hd), np.float64)
        if imp is not None:
            assert imp.dtype == np.float64 and imp.flags.c_contiguous
        sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float32)
        assert sk is None or sk.size == nheads
        lib().kvo_attend_group_ex(C.byref(self._s), _p(q_group), kv_head, nheads, scale, int(first),
                                  float(softcap), int(upto), _p(sk), _p(out), _p(imp))
        return out

    def decode_ex(self, q, n_q: int, scale: float, window: int = 0, softcap: float = 0.0,
                  sinks=None, imp=None):
        """decode with a sliding window (first = stored - window when stored >
        window; 0 = no window), soft-capping and per-query-head sinks [n_q]."""
        hpk = n_q // self.n_kv
        q = np.ascontiguousarray(q, dtype=np.float32).reshape(n_q, self.hd)
        out = np.zeros((n_q, self.hd), np.float64)
        for g in range(self.n_kv):
            stored = int(self.head_rows[g])
            first = stored - window if window > 0 and stored > window else 0
            sk = None if sinks is None else np.asarray(sinks, np.float32)[g * hpk:(g + 1) * hpk]
            out[g * hpk:(g + 1) * hpk] = self.attend_group_ex(q[g * hpk:(g + 1) * hpk], g, scale, first,
                                                              softcap, sk, imp)
        return out

    def decode_verify(self, q, n_q: int, K: int, scale: float, window: int = 0, softcap: float = 0.0,
                      sinks=None):
        """Query-batched verify of K draft rows already appended: query k ([K, n_q,
        hd]) attends with upto = stored - (K - 1 - k), i.e. the rows up to and
        including draft k (causal among the drafts), and a sliding window counted
        back from its own position.  Returns [K, n_q, hd] (f64)."""
        hpk = n_q // self.n_kv
        q = np.ascontiguousarray(q, dtype=np.float32).reshape(K, n_q, self.hd)
        out = np.zeros((K, n_q, self.hd), np.float64)
        for k in range(K):
            for g in range(self.n_kv):
                stored = int(self.head_rows[g])
                upto = max(stored - (K - 1 - k), 0)
                first = upto - window if window > 0 and upto > window else 0
                sk = None if sinks is None else np.asarray(sinks, np.float32)[g * hpk:(g + 1) * hpk]
                out[k, g * hpk:(g + 1) * hpk] = self.attend_group_ex(q[k, g * hpk:(g + 1) * hpk], g, scale, first,
                                                                     softcap, sk, None, upto)
        return out

    def decode(self, q, n_q: int, scale: float, imp=None):
        """All query heads of the layer: q [n_q, hd] -> out [n_q, hd] (f64); head h
        belongs to KV group h // (n_q // n_kv)."""
        hpk = n_q // self.n_kv
        q = np.ascontiguousarray(q, dtype=np.float32).reshape(n_q, self.hd)
        out = np.zeros((n_q, self.hd), np.float64)
        for g in range(self.n_kv):
            out[g * hpk:(g + 1) * hpk] = self.attend_group(q[g * hpk:(g + 1) * hpk], g, scale, imp)
        return out

    def memory_bytes(self) -> int:
        return int(lib().kvo_memory_bytes(C.byref(self._s)))

    def truncate_last(self, n_drop: int, imp: np.ndarray | None = None) -> int:
        """cortiq truncate_last: drop the last n_drop rows (imp entries cleared)."""
        if imp is not None:
            assert imp.dtype == np.float32 and imp.flags.c_contiguous and imp.shape[0] >= self.seq_len
        n = lib().kvo_truncate_last(C.byref(self._s), _p(imp), n_drop)
        if n < 0:
            raise ValueError("truncate_last: negative count")
        return n

    def evict_born(self, keep_last: int, sink: int, recent: int, imp: np.ndarray) -> int:
        """cortiq evict_born: keep sinks + recents + the middle rows of highest
        mass, gathered in row order; imp (f32 [cap], this sequence's mass per
        row) is gathered in place.  Returns the rows kept."""
        assert imp.dtype == np.float32 and imp.flags.c_contiguous and imp.shape[0] >= self.seq_len
        n = lib().kvo_evict_born(C.byref(self._s), _p(imp), keep_last, sink, recent)
        if n < 0:
            raise ValueError("evict_born: negative argument")
        return n


def decode_many(caches, qs, n_q: int, scale, imps=None, threads: int = 0):
    """Decode of several sequences at once (kvo_decode_many): the (sequence,
    query head) pairs shared among `threads` OpenMP threads (0 = every core the
    runtime sees), bitwise equal to calling OracleSeqCache.decode on each.
    caches: OracleSeqCache list; qs: [n_q, hd] f32 each; imps: None or an f64
    array per sequence (accumulated).  Returns (outputs [n_q, hd] f64 list,
    threads used)."""
    n = len(caches)
    qs = [np.ascontiguousarray(q, dtype=np.float32).reshape(n_q, c.hd) for q, c in zip(qs, caches)]
    outs = [np.zeros((n_q, c.hd), np.float64) for c in caches]
    cp = (C.c_void_p * n)(*[C.addressof(c._s) for c in caches])
    qp = (C.c_void_p * n)(*[q.ctypes.data for q in qs])
    op = (C.c_void_p * n)(*[o.ctypes.data for o in outs])
    ip = None
    if imps is not None:
        for a in imps:
            assert a is None or (a.dtype == np.float64 and a.flags.c_contiguous)
        ip = (C.c_void_p * n)(*[None if a is None else a.ctypes.data for a in imps])
    used = lib().kvo_decode_many(cp, n, qp, int(n_q), float(scale), op, ip, int(threads))
    if used < 0:
        raise MemoryError("oracle decode_many: allocation failed")
    return outs, int(used)


def rswa_write(ring_k, ring_v, k, v, prefill_recorded: bool, cursors):
    """rswa write_decode_step for one stream; ring_* are [H, W, hd] f32 (updated in
    place), cursors a np.int32[2] = (ring_len, ring_pos) updated in place.  Returns
    the slot written, or raises on the error the page specifies."""
    H, W, hd = ring_k.shape
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    rl = cursors[0:1]
    rp = cursors[1:2]
    slot = lib().kvo_rswa_write(H, hd, W, _p(ring_k), _p(ring_v), _p(k), _p(v),
                                int(prefill_recorded), rl.ctypes.data, rp.ctypes.data)
    if slot < 0:
        raise RuntimeError("rswa write before prefill")
    return slot


def rswa_decode(q, ref_k, ref_v, prefill_len, ring_k, ring_v, ring_len, scale):
    """rswa decode_attention for one stream.  ref_* [H, ref_cap, hd], ring_* [H, W, hd],
    q [H, hd].  Returns out [H, hd] f64; raises on no-prefill / empty key set."""
    H, ref_cap, hd = ref_k.shape
    W = ring_k.shape[1]
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.zeros((H, hd), np.float64)
    rc = lib().kvo_rswa_decode(H, hd, _p(q), _p(ref_k), _p(ref_v), ref_cap,
                               -1 if prefill_len is None else int(prefill_len),
                               _p(ring_k), _p(ring_v), W, int(ring_len), scale, _p(out))
    if rc == -3:
        raise RuntimeError("rswa decode before prefill")
    if rc == -4:
        raise RuntimeError("rswa empty attention key set")
    return out


def rswa_mirror(rows):
    """rswa int8 mirror of f32 rows [..., hd]: quantize_row_i8 on every row.
    Returns (codes int8 [..., hd], scales f32 [...])."""
    rows = np.ascontiguousarray(rows, dtype=np.float32)
    n = rows.shape[-1]
    n_rows = rows.size // n if n else 0
    codes = np.zeros(rows.shape, np.int8)
    scales = np.zeros(rows.shape[:-1], np.float32)
    if n_rows:
        lib().kvo_quantize_rows_i8(_p(rows), n_rows, n, _p(codes), _p(scales))
    return codes, scales


def rswa_decode_i8(q, ref_k8, ref_ks, ref_v8, ref_vs, prefill_len, ring_k8, ring_ks, ring_v8,
                   ring_vs, ring_len, scale):
    """rswa decode_attention_int8 for one stream over its int8 mirror: codes
    [H, rows, hd] int8 and scales [H, rows] f32 (rows = ref_cap, W), q [H, hd] f32.
    Returns out [H, hd] f64; raises on no-prefill / empty key set."""
    H, ref_cap, hd = ref_k8.shape
    W = ring_k8.shape[1]
    q = np.ascontiguousarray(q, dtype=np.float32)
    arrs = [np.ascontiguousarray(a, dtype=t) for a, t in
            ((ref_k8, np.int8), (ref_ks, np.float32), (ref_v8, np.int8), (ref_vs, np.float32),
             (ring_k8, np.int8), (ring_ks, np.float32), (ring_v8, np.int8), (ring_vs, np.float32))]
    out = np.zeros((H, hd), np.float64)
    rc = lib().kvo_rswa_decode_i8(H, hd, _p(q), _p(arrs[0]), _p(arrs[1]), _p(arrs[2]), _p(arrs[3]),
                                  ref_cap, -1 if prefill_len is None else int(prefill_len),
                                  _p(arrs[4]), _p(arrs[5]), _p(arrs[6]), _p(arrs[7]), W,
                                  int(ring_len), scale, _p(out))
    if rc == -3:
        raise RuntimeError("rswa decode before prefill")
    if rc == -4:
        raise RuntimeError("rswa empty attention key set")
    return out


def rswa_verify(q, draft_k, draft_v, ref_k, ref_v, prefill_len, ring_k, ring_v, cursors, scale,
                int8: bool = False):
    """rswa verify_attention for one stream: K draft tokens (q, draft_k, draft_v
    [K, H, hd]) against a PRIVATE copy of the ring: draft i is written
    (write_decode_step) before query i decodes (decode_attention, or
    decode_attention_int8 over the mirror of the copy when int8), so query i
    sees the reference rows and the ring after drafts 0..i.  The caller's
    arrays and cursors are left untouched.  Returns [K, H, hd] f64."""
    K = q.shape[0]
    gk, gv, cur = ring_k.copy(), ring_v.copy(), np.array(cursors, np.int32).copy()
    out = []
    if int8:
        rk8, rks = rswa_mirror(ref_k)
        rv8, rvs = rswa_mirror(ref_v)
    for i in range(K):
        rswa_write(gk, gv, draft_k[i], draft_v[i], prefill_len is not None, cur)
        if int8:
            gk8, gks = rswa_mirror(gk)
            gv8, gvs = rswa_mirror(gv)
            out.append(rswa_decode_i8(q[i], rk8, rks, rv8, rvs, prefill_len, gk8, gks, gv8, gvs, cur[0], scale))
        else:
            out.append(rswa_decode(q[i], ref_k, ref_v, prefill_len, gk, gv, cur[0], scale))
    return np.stack(out)


def online_head(q, keys, vals, scale):
    """rswa fold recurrence (f32) for one head over keys/vals [n, hd]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    keys = np.ascontiguousarray(keys, dtype=np.float32)
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    out = np.zeros(q.shape[0], np.float32)
    lib().kvo_online_head(keys.shape[0], q.shape[0], _p(q), _p(keys), _p(vals), scale, _p(out))
    return out
