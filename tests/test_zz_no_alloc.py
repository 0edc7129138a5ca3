"""decode_attention_static: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc on their decode path (a
runtime that serves from a fixed, pre-planned device arena, a plug-in inside
a host application that owns every allocation, code that must not take
cudaMalloc's device-wide synchronisation mid-serving).  The static variant
takes its scratch from an array compiled into the library instead of a
caller workspace.  These tests call it through the C ABI, several times in a
row on different layers (the array keeps the last call's contents), and check
every output against the CPU oracle and against decode_attention (the
workspace variant), with the tolerance the parity tests use: all four storage
modes at head_dim 128 and 64, a layer whose groups are all dead, a call that
needs just under the 16 MiB array, and one that needs more (refused).

The file name sorts last so that a run stopping at the first failure has run
every other test first; it passes alone in a fresh process too.
"""

import ctypes as C

import numpy as np
import pytest

import oracle
from helpers import OUT_TOL, oracle_caches, out_error, seq_rows

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20  # bytes of the library's scratch array


@pytest.fixture(scope="module")
def env():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import kv_cache_decode_attention_gb300 as kvd
    from kv_cache_decode_attention_gb300.build import build

    build()
    return torch, kvd


def _static_call(layer, q, out):
    """decode_attention_static straight through the C ABI."""
    from kv_cache_decode_attention_gb300 import _abi

    return _abi.lib().decode_attention_static(
        C.c_void_p(q.data_ptr()), C.byref(layer.L), q.shape[1], C.c_float(1.0 / np.sqrt(layer.head_dim)),
        C.c_void_p(out.data_ptr()), C.c_void_p(0))


def _build(torch, kvd, mode, lengths, n_kv, hpk, hd, alive, seed):
    """The same seeded rows in a device layer and in the oracle."""
    ks, vs = seq_rows(lengths, n_kv, hd, seed)
    layer = kvd.LayerKvCache(len(lengths), n_kv, hd, mode, [max(L, 1) for L in lengths], alive=alive)
    kvd.kv_append(layer, torch.from_numpy(np.concatenate(ks)).cuda(), torch.from_numpy(np.concatenate(vs)).cuda(),
                  np.asarray(lengths, np.int32))
    q = np.random.default_rng(seed).standard_normal((len(lengths), n_kv * hpk, hd)).astype(np.float32)
    oc = oracle_caches(kvd.api.MODE_NAMES[mode], lengths, n_kv, hd, alive, ks, vs)
    return layer, q, oc


def _check(torch, kvd, layer, q, oc, samples=None):
    n_q, hd = q.shape[1], q.shape[2]
    qd = torch.from_numpy(q).cuda()
    out = torch.full_like(qd, float("nan"))
    assert _static_call(layer, qd, out) == 0
    ref_ws = kvd.decode_attention(qd, layer, imp=None)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    got, ws = out.cpu().numpy(), ref_ws.cpu().numpy()
    scale = np.float32(1.0 / np.sqrt(hd))
    for b in (range(len(oc)) if samples is None else samples):
        ref = oc[b].decode(q[b], n_q, scale)
        live = np.array([oc[b].alive[h // (n_q // oc[b].n_kv)] != 0 and oc[b].seq_len > 0 for h in range(n_q)])
        assert np.all(got[b][~live] == 0.0), b
        if live.any():
            assert out_error(got[b], ref, live) <= OUT_TOL, b
            assert out_error(got[b], ws[b], live) <= OUT_TOL, b


@pytest.mark.parametrize("hd", [128, 64])
def test_static_matches_oracle_every_mode(env, hd):
    """Four layers in a row (f32, q8, q8k, q8v): ragged lengths across the freeze
    at 64 rows, an empty sequence, a dead group."""
    torch, kvd = env
    for mi, mode in enumerate(("f32", "q8", "q8k", "q8v")):
        layer, q, oc = _build(torch, kvd, mode, [700, 0, 2100, 64, 65], 4, 4, hd, [1, 1, 0, 1], 10 * mi + hd)
        _check(torch, kvd, layer, q, oc)


def test_static_all_groups_dead_gives_zeros(env):
    torch, kvd = env
    layer, q, oc = _build(torch, kvd, "q8", [300, 5], 2, 8, 128, [0, 0], 3)
    _check(torch, kvd, layer, q, oc)


def test_static_call_just_under_the_limit(env):
    """252 sequences x 8 groups x 16 heads, one chunk each: the partials need
    16,773,120 bytes of the 16,777,216 (sampled sequences against the oracle)."""
    torch, kvd = env
    n_seq, n_kv, hpk, hd = 252, 8, 16, 128
    P = n_seq * n_kv * 1 * hpk
    need = 2 * (-(-P * 4 // 256) * 256) + -(-P * hd * 4 // 256) * 256
    assert need <= LIMIT < need + 130 * 1024
    lengths = [1 + (b * 37) % 256 for b in range(n_seq)]
    layer, q, oc = _build(torch, kvd, "f32", lengths, n_kv, hpk, hd, None, 4)
    _check(torch, kvd, layer, q, oc, samples=[0, 7, 100, 251])


def test_static_refuses_oversized_calls(env):
    torch, kvd = env
    # 512 sequences x 8 KV groups x 16 heads of partials need ~34 MiB > 16 MiB
    layer = kvd.LayerKvCache(512, 8, 128, "f32", 1)
    kvd.kv_append(layer, torch.randn(512, 8, 128, device="cuda"), torch.randn(512, 8, 128, device="cuda"))
    q = torch.randn(512, 128, 128, device="cuda")
    out = torch.zeros_like(q)
    assert _static_call(layer, q, out) == -2  # KVD_ECAPACITY, nothing launched
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
