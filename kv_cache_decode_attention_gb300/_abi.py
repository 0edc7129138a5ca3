"""ctypes declarations of the C ABI in include/kvd.h (argument marshalling only).

Loading fails loudly when libkvd.so has not been built: there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(PKG), "include", "kvd.h")
LIB_PATH = os.path.join(PKG, "libkvd.so")

# status codes (kvd_status)
OK, EINVAL, ECAPACITY, ESTATE, EEMPTY, ECUDA, EDEVICE = 0, -1, -2, -3, -4, -5, -6
# storage modes (kvd_mode)
F32, Q8, Q8K, Q8V = 0, 1, 2, 3
# buffer slots
BUF_K, BUF_V, BUF_KQ, BUF_VQ, BUF_KS, BUF_VS, BUF_KCOL, BUF_VCOL, BUF_META, BUF_COUNT = range(10)


class kvd_layer(C.Structure):
    _fields_ = [("opaque", C.c_uint64 * 128)]


class rswa_i8_mirror(C.Structure):
    _fields_ = [("ref_k", C.c_void_p), ("ref_v", C.c_void_p), ("ref_ks", C.c_void_p),
                ("ref_vs", C.c_void_p), ("ring_k", C.c_void_p), ("ring_v", C.c_void_p),
                ("ring_ks", C.c_void_p), ("ring_vs", C.c_void_p)]


class rswa_history(C.Structure):
    _fields_ = [("decode_writes", C.c_int64), ("lineage_epoch", C.c_uint64)]


class rswa_checkpoint(C.Structure):
    _fields_ = [("cache_id", C.c_uint64), ("lineage_epoch", C.c_uint64), ("decode_writes", C.c_int64),
                ("prefill_len", C.c_int32), ("ring_len", C.c_int32), ("ring_pos", C.c_int32),
                ("pad", C.c_int32)]


class KvdError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__("%s failed: %s (%d)" % (fn, msg, status))
        self.status = status


_vp, _i32, _i64, _f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
_P = C.POINTER

_SIGS = {
    "kvd_layer_bytes": [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp],
    "kvd_layer_init": [_P(kvd_layer), _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp],
    "kvd_layer_reset": [_P(kvd_layer), _i32, _vp],
    "kvd_layer_seq_len": [_P(kvd_layer), _i32, _P(_i64), _P(_i32)],
    "kvd_layer_memory_bytes": [_P(kvd_layer), _P(_i64)],
    "kv_append": [_P(kvd_layer), _vp, _vp, _vp, _vp],
    "kv_freeze_colfield": [_P(kvd_layer), _vp],
    "kv_truncate_last": [_P(kvd_layer), _vp, _vp, _vp],
    "kvd_verify_workspace_bytes": [_P(kvd_layer), _i32, _i32, _P(_i64)],
    "decode_attention_verify": [_vp, _P(kvd_layer), _i32, _i32, _f32, _i64, _f32, _vp, _vp, _vp, _i64, _vp],
    "kv_evict_workspace_bytes": [_P(kvd_layer), _i64, _P(_i64)],
    "kv_evict_born": [_P(kvd_layer), _vp, _i64, _i32, _i32, _vp, _i64, _vp],
    "kvd_decode_workspace_bytes": [_P(kvd_layer), _i32, _i32, _P(_i64)],
    "decode_attention": [_vp, _P(kvd_layer), _i32, _f32, _vp, _vp, _vp, _i64, _vp],
    "decode_attention_ex": [_vp, _P(kvd_layer), _i32, _f32, _i64, _f32, _vp, _vp, _vp, _vp, _i64, _vp],
    "decode_attention_static": [_vp, _P(kvd_layer), _i32, _f32, _vp, _vp],
    "kvd_layer_device_error": [_P(kvd_layer), _i32, _P(C.c_uint32)],
    "kvd_wait_timeout_selftest": [_P(kvd_layer), _i64, _vp],
    "kvd_bounds_selftest_bytes": [_P(kvd_layer), _P(_i64)],
    "kvd_bounds_selftest": [_P(kvd_layer), _vp, _i64, _vp],
    "kvd_test_fail_after": [_i64],
    "rswa_record_prefill": [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i32,
                            _vp, _vp, _vp, _vp, _vp],
    "rswa_ring_write": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp],
    "rswa_checkpoint_take": [C.c_uint64, _vp, _vp, _vp, _vp, _i32, _P(rswa_checkpoint)],
    "rswa_rollback_to": [C.c_uint64, _vp, _vp, _vp, _vp, _i32, _i32, _P(rswa_checkpoint)],
    "rswa_decode_workspace_bytes": [_i32, _i32, _i32, _i64, _i32, _P(_i64)],
    "rswa_decode": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _f32,
                    _vp, _vp, _i64, _vp],
    "rswa_record_prefill_i8": [_vp, _vp, _P(rswa_i8_mirror), _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                               _i64, _i32, _vp, _vp, _vp, _vp, _vp],
    "rswa_ring_write_i8": [_vp, _vp, _P(rswa_i8_mirror), _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                           _i32, _vp, _vp],
    "rswa_decode_i8": [_vp, _P(rswa_i8_mirror), _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _f32, _vp,
                       _vp, _i64, _vp],
    "rswa_verify_workspace_bytes": [_i32, _i32, _i32, _i64, _i32, _i32, _P(_i64)],
    "rswa_verify": [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32,
                    _f32, _vp, _vp, _i64, _vp],
    "rswa_verify_i8": [_vp, _vp, _vp, _i32, _P(rswa_i8_mirror), _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32,
                       _f32, _vp, _vp, _i64, _vp],
    "rswa_device_error": [_vp, _i32, _P(C.c_uint32)],
    "kvd_status_string": [_i32],
}

_lib = None


def declared_symbols() -> list[str]:
    """Every entry point include/kvd.h declares (the names after KVD_API)."""
    text = open(HEADER).read()
    return re.findall(r"KVD_API\s+(?:const\s+char\s*\*|kvd_status)\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", text)


def lib():
    """The loaded library; raises if it was not built (no CPU fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "libkvd.so is missing (%s): build it with `python -m "
                "kv_cache_decode_attention_gb300.build` (nvcc, sm_103a)" % LIB_PATH)
        L = C.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = C.c_char_p if name == "kvd_status_string" else C.c_int32
        _lib = L
    return _lib


def check(fn: str, status: int) -> int:
    if status != OK:
        raise KvdError(fn, status, lib().kvd_status_string(status).decode())
    return status


def call(fn: str, *args) -> int:
    """Call an entry point and raise KvdError on a non-OK status."""
    return check(fn, getattr(lib(), fn)(*args))
