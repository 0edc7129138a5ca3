"""Calls on different CUDA streams do not interfere.

The library keeps no device state of its own on the decode path (every
buffer is the caller's, passed per call), so two layers driven on two streams
at once must give exactly what the same calls give one after the other on
one stream.  Each stream runs appends and decodes with imp on its own layer
and workspace -- one layer on the q8_2f tensor-core path, one on the
CUDA-core path -- interleaved on the host so that their kernels overlap on
the device; the outputs and imp are compared bitwise with a serial replay
(every kernel is deterministic).
"""

import numpy as np
import pytest

from helpers import gpu_append_bulk, seq_rows

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


def _make(torch, kvd, mode, hd, seed):
    lengths = [900, 70, 2500, 33]
    n_kv, hpk = 2, 4
    ks, vs = seq_rows(lengths, n_kv, hd, seed)
    layer = kvd.LayerKvCache(len(lengths), n_kv, hd, mode, [L + 16 for L in lengths])
    gpu_append_bulk(layer, ks, vs, torch)
    g = torch.Generator(device="cuda").manual_seed(seed)
    steps = [(torch.randn(len(lengths), n_kv, hd, generator=g, device="cuda"),
              torch.randn(len(lengths), n_kv, hd, generator=g, device="cuda"),
              torch.randn(len(lengths), n_kv * hpk, hd, generator=g, device="cuda")) for _ in range(6)]
    return layer, steps


def _run(torch, kvd, layer, steps, stream):
    outs = []
    imp = torch.zeros(layer.imp_len, device="cuda")
    ws = torch.empty(layer.workspace_bytes(steps[0][2].shape[1], True), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for k, v, q in steps:
            kvd.kv_append(layer, k, v)
            outs.append(kvd.decode_attention(q, layer, imp=imp, workspace=ws))
    return outs, imp


def test_two_streams_match_a_serial_replay(env):
    torch, kvd = env
    a_layer, a_steps = _make(torch, kvd, "q8", 128, 31)
    b_layer, b_steps = _make(torch, kvd, "f32", 64, 32)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    # interleaved on two streams: the host alternates, the device overlaps
    a_outs, b_outs = [], []
    a_imp = torch.zeros(a_layer.imp_len, device="cuda")
    b_imp = torch.zeros(b_layer.imp_len, device="cuda")
    a_ws = torch.empty(a_layer.workspace_bytes(8, True), dtype=torch.uint8, device="cuda")
    b_ws = torch.empty(b_layer.workspace_bytes(8, True), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()  # everything made on the default stream is in place
    for (ka, va, qa), (kb, vb, qb) in zip(a_steps, b_steps):
        with torch.cuda.stream(sa):
            kvd.kv_append(a_layer, ka, va)
            a_outs.append(kvd.decode_attention(qa, a_layer, imp=a_imp, workspace=a_ws))
        with torch.cuda.stream(sb):
            kvd.kv_append(b_layer, kb, vb)
            b_outs.append(kvd.decode_attention(qb, b_layer, imp=b_imp, workspace=b_ws))
    torch.cuda.synchronize()
    assert a_layer.device_error() == 0 and b_layer.device_error() == 0

    # the same calls, one after the other on fresh layers, on one stream
    a2, _ = _make(torch, kvd, "q8", 128, 31)
    b2, _ = _make(torch, kvd, "f32", 64, 32)
    ra, ra_imp = _run(torch, kvd, a2, a_steps, torch.cuda.current_stream())
    rb, rb_imp = _run(torch, kvd, b2, b_steps, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for x, y in zip(a_outs + b_outs, ra + rb):
        assert torch.equal(x, y)
    assert torch.equal(a_imp, ra_imp) and torch.equal(b_imp, rb_imp)
    assert [a_layer.seq_len(b) for b in range(4)] == [a2.seq_len(b) for b in range(4)]
    assert np.all(np.isfinite(torch.stack(a_outs).cpu().numpy()))
