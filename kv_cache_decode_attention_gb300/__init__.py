"""GB300 (sm_103a) KV-cache decode attention: GQA decode over an f32 / q8_2f /
q8k / q8v head-major cache, the R-SWA prefix + ring variant, and the
append/quantise kernel, behind the C ABI in include/kvd.h.

The CUDA library must be built first (``python -m
kv_cache_decode_attention_gb300.build``); importing the API without it raises.
"""

from ._abi import F32, Q8, Q8K, Q8V, KvdError, declared_symbols, lib  # noqa: F401
from .api import (  # noqa: F401
    LayerKvCache,
    RingCache,
    decode_attention,
    decode_attention_static,
    decode_attention_verify,
    kv_append,
    kv_evict_born,
    kv_freeze_colfield,
    kv_truncate_last,
    rswa_attention,
    rswa_decode,
    rswa_decode_i8,
    rswa_record_prefill,
    rswa_ring_write,
    rswa_verify,
)
