"""CPU oracle for the KV-cache decode-attention hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The CUDA library never imports,
links or calls anything here, and this package never imports the library.

The arithmetic lives in ``kvd_oracle.c`` (plain C, compiled with
``-ffp-contract=off`` so the f32 quantiser is bit-defined on x86-64 and
AArch64 alike); this module compiles it, binds it with ctypes and adds thin
numpy-array bookkeeping around it.
"""

from .oracle import (  # noqa: F401
    F32,
    Q8,
    Q8K,
    Q8V,
    COL_WARMUP,
    K_GROUP,
    OracleSeqCache,
    build_oracle,
    decode_many,
    lib,
    quant_row,
    quantize_row_i8,
    rswa_decode,
    rswa_decode_i8,
    rswa_mirror,
    rswa_verify,
    rswa_write,
    online_head,
)
