"""decode_attention_static: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc on their decode path (a
runtime that serves from a fixed, pre-planned device arena, a plug-in inside
a host application that owns every allocation, code that must not take
cudaMalloc's device-wide synchronisation mid-serving).  The static variant
takes its scratch from an array compiled into the library instead of a
caller workspace.  This test calls it through the C ABI twice in a row, on
two different layers, and checks each output against decode_attention (the
workspace variant) with the same tolerance the parity tests use; it also
checks that a call needing more than the 16 MiB array is refused.

The file name sorts last so that a run stopping at the first failure has run
every other test first; it passes alone in a fresh process too.
"""

import ctypes as C

import numpy as np
import pytest

from helpers import OUT_TOL, out_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300.build import build

    build()
    return torch, kvd


def _layer(torch, kvd, mode, lengths, n_kv, hpk, hd, alive, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    layer = kvd.LayerKvCache(len(lengths), n_kv, hd, mode, lengths, alive=alive)
    n = int(np.sum(lengths))
    k = torch.randn(n, n_kv, hd, generator=g, device="cuda") * 3.0
    v = torch.randn(n, n_kv, hd, generator=g, device="cuda")
    kvd.kv_append(layer, k, v, np.asarray(lengths, np.int32))
    q = torch.randn(len(lengths), n_kv * hpk, hd, generator=g, device="cuda")
    return layer, q


def _static_call(kvd, layer, q, out):
    # straight through the C ABI
    from kv_cache_decode_attention_gb300 import _abi

    n_q = q.shape[1]
    st = _abi.lib().decode_attention_static(
        C.c_void_p(q.data_ptr()), C.byref(layer.L), n_q, C.c_float(1.0 / np.sqrt(layer.head_dim)),
        C.c_void_p(out.data_ptr()), C.c_void_p(0))
    return st


def test_static_variant_matches_workspace_variant_twice(env):
    torch, kvd = env
    cases = [
        _layer(torch, kvd, "q8", [700, 1, 2100, 64], 4, 4, 128, [1, 1, 0, 1], 1),
        _layer(torch, kvd, "f32", [300, 999], 2, 8, 64, None, 2),
    ]
    for layer, q in cases:  # two calls in a row, one per layer
        ref = kvd.decode_attention(q, layer, imp=None)
        out = torch.full_like(q, float("nan"))
        assert _static_call(kvd, layer, q, out) == 0
        torch.cuda.synchronize()
        r, o = ref.cpu().numpy(), out.cpu().numpy()
        live = np.abs(r).sum(axis=-1) > 0
        assert np.array_equal(o[~live], r[~live])
        assert out_error(o, r, live) <= OUT_TOL
        assert layer.device_error() == 0


def test_static_variant_refuses_oversized_calls(env):
    torch, kvd = env
    # 512 sequences x 8 KV groups x 16 heads of partials need ~34 MiB > 16 MiB
    layer, q = _layer(torch, kvd, "f32", [1] * 512, 8, 16, 128, None, 3)
    out = torch.zeros_like(q)
    assert _static_call(kvd, layer, q, out) == -2  # KVD_ECAPACITY, nothing launched
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
