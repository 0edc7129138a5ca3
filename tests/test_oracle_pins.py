"""Pins for the CPU oracle: values the pages print, closed forms, invariants
and library cross-checks, chosen so that a plausible slip in the oracle (a
dropped field, a wrong group index, a transposed operand, reciprocal instead
of division, half-away rounding) fails at least one of them.

Page citations: [cortiq] = docs.rs cortiq-engine 0.8.49 kv_cache.rs;
[rswa] = franken_ocr 0.8.0 src/native_engine/rswa.rs.
"""

import math

import numpy as np
import pytest

import oracle
import synthetic
from conftest import load_golden

f32 = np.float32


def bits_to_f32(b: int) -> np.float32:
    return np.frombuffer(np.uint32(b).tobytes(), np.float32)[0]


# ---------------------------------------------------------------- quantiser

def test_ties_to_even_rswa_vector():
    """[rswa] test int8_row_quantization_uses_ties_to_even, verbatim."""
    g = load_golden("quant_ties_to_even.txt")
    row = np.zeros(int(g["width"]), f32)
    head = np.array(g["row_head"].split(), f32)
    row[: head.size] = head
    want = np.array(g["codes_head"].split(), np.int8)
    q, s = oracle.quantize_row_i8(row)
    assert np.array_equal(q[: want.size], want)
    assert s.view(np.uint32) == int(g["scale_bits"], 16)


@pytest.mark.parametrize("group", [32, 128])
def test_ties_to_even_q8_2f_row(group):
    """The same vector through the q8_2f quantiser ([cortiq] quant_row): absmax
    127 puts the scale at 1.0, above the 1e-12 floor, so the tie rule alone
    decides the codes (half away from zero would give 1, 2, 3, 4 ...)."""
    g = load_golden("quant_ties_to_even.txt")
    row = np.zeros(128, f32)
    head = np.array(g["row_head"].split(), f32)
    row[: head.size] = head
    want = np.array(g["codes_head"].split(), np.int8)
    q, s = oracle.quant_row(row, None, group)
    assert np.array_equal(q[: want.size], want)
    assert s[0].view(np.uint32) == int(g["scale_bits"], 16)


def test_division_not_reciprocal_rswa_fixture():
    """[rswa] test int8_row_quantization_divides_instead_of_multiplying_by_reciprocal."""
    g = load_golden("quant_division.txt")
    row = np.zeros(int(g["width"]), f32)
    row[0] = bits_to_f32(int(g["x0_bits"], 16))
    row[1] = bits_to_f32(int(g["x1_bits"], 16))
    q, s = oracle.quantize_row_i8(row)
    assert list(q[:2]) == [int(c) for c in g["codes"].split()]
    recip = np.rint(row[1] * (f32(1.0) / s))  # the formula the page rules out
    assert int(recip) == int(g["reciprocal_code1"])


def test_division_not_reciprocal_q8_2f_scaled():
    """The page fixture sits below the q8_2f 1e-12 scale floor, so it is scaled by
    2^67 (exact in f32: every quotient and scale scales by the same power of two)
    to bring it into the q8_2f quantiser's range; the codes must not change."""
    g = load_golden("quant_division.txt")
    row = np.zeros(128, f32)
    row[0] = bits_to_f32(int(g["x0_bits"], 16))
    row[1] = bits_to_f32(int(g["x1_bits"], 16))
    scaled = (row * f32(2.0 ** 67)).astype(f32)
    assert np.array_equal(scaled / f32(2.0 ** 67), row)  # the scaling is exact
    for group in (32, 128):
        q, s = oracle.quant_row(scaled, None, group)
        assert list(q[:2]) == [int(c) for c in g["codes"].split()]
        assert int(np.rint(scaled[1] * (f32(1.0) / s[0]))) == int(g["reciprocal_code1"])


def test_quantiser_lcg_sweep_matches_numpy_f32():
    """[rswa] test int8_row_quantization_matches_scalar_contract: 256 rows from the
    page's LCG over magnitudes 2^-20..2^20 (row 0 all zero).  Expected codes come
    from numpy's own f32 division and np.rint (IEEE round-half-even), an
    implementation independent of the C oracle; both quantisers are checked."""
    state = 0xD1B54A32D192ED03
    mask = (1 << 64) - 1
    for case in range(256):
        mag = f32(2.0) ** f32((case % 41) - 20)
        row = np.zeros(128, f32)
        for i in range(128):
            state = (state * 6364136223846793005 + 1442695040888963407) & mask
            unit = f32((state >> 40) & 0xFFFFFFFF) / f32((1 << 24) - 1)
            row[i] = (unit * f32(2.0) - f32(1.0)) * mag
        if case == 0:
            row[:] = 0.0
        absmax = np.max(np.abs(row))
        # rswa mirror: scale 1.0 for an all-zero row
        sc = absmax / f32(127.0) if absmax > 0 else f32(1.0)
        want = np.clip(np.rint(row / sc), -127, 127).astype(np.int8)
        q, s = oracle.quantize_row_i8(row)
        assert s.view(np.uint32) == f32(sc).view(np.uint32), case
        assert np.array_equal(q, want), case
        # q8_2f (cortiq): per 32-channel group, scale floored at 1e-12
        q2, s2 = oracle.quant_row(row, None, 32)
        for gi in range(4):
            seg = row[gi * 32:(gi + 1) * 32]
            sg = max(np.max(np.abs(seg)) / f32(127.0), f32(1e-12))
            assert s2[gi].view(np.uint32) == f32(sg).view(np.uint32), (case, gi)
            assert np.array_equal(q2[gi * 32:(gi + 1) * 32],
                                  np.clip(np.rint(seg / f32(sg)), -127, 127).astype(np.int8))


def test_quantiser_floor_and_zero_group():
    """[cortiq] quant_row: scale = max(absmax/127, 1e-12); an all-zero group takes
    the floor (not rswa's 1.0) and codes 0; a group below the floor quantises
    against the floor."""
    row = np.zeros(128, f32)
    row[40] = 1e-14
    row[64:96] = np.linspace(-3, 3, 32, dtype=f32)
    q, s = oracle.quant_row(row, None, 32)
    assert s[0] == f32(1e-12) and not q[:32].any()
    assert s[1] == f32(1e-12)
    assert q[40] == int(np.rint(f32(1e-14) / f32(1e-12)))
    assert s[2] == f32(3.0) / f32(127.0)
    assert q[64] == -127 and q[95] == 127


def test_quantiser_col_division_and_half_scale_bound():
    """Round-to-nearest bound: dequantised rows reproduce the originals within
    scale/2 per element; with a per-channel field the residual x/col is what is
    quantised."""
    x = synthetic.normal((50, 128), 11) * synthetic.channel_sigma((128,), 12)
    col = synthetic.channel_sigma((128,), 13)
    for r in x:
        q, s = oracle.quant_row(r, None, 32)
        deq = q.astype(np.float64) * np.repeat(s, 32)
        assert np.all(np.abs(deq - r) <= np.repeat(s, 32) / 2 * (1 + 1e-6))
        q, s = oracle.quant_row(r, col, 32)
        resid = (r / col).astype(f32)
        deq = q.astype(np.float64) * np.repeat(s, 32)
        assert np.all(np.abs(deq - resid) <= np.repeat(s, 32) / 2 * (1 + 1e-6))
        # V-style: one group over the whole row
        q, s = oracle.quant_row(r, col, 128)
        assert s.size == 1
        assert np.all(np.abs(q * np.float64(s[0]) - resid) <= s[0] / 2 * (1 + 1e-6))


# ------------------------------------------------------------------- freeze

def _integer_rows(n, hd, seed):
    """Rows of integers whose every 32-channel group peaks at exactly 127, so the
    pre-freeze q8 codes equal the values and the scale is 1.0 in every group."""
    r = synthetic.rng(seed)
    x = r.integers(-126, 127, size=(n, hd)).astype(f32)
    for g0 in range(0, hd, 32):
        x[np.arange(n), g0 + r.integers(0, 32, size=n)] = 127.0
    return x


def test_freeze_col_is_exact_channel_rms():
    """[cortiq] freeze_cols: col[d] = max(sqrt(sum_p row^2 / n), 1e-6).  With
    integer rows the f32 sum of squares is exact (< 2^24), /64 is exact, so col
    must equal the correctly rounded sqrt of the exact integer mean square."""
    hd = 128
    x = _integer_rows(64, hd, 21)
    c = oracle.OracleSeqCache(oracle.Q8, 1, hd, 80)
    for p in range(64):
        c.append(x[p][None], x[p][None])
    assert not c.frozen and c.needs_freeze()
    assert np.array_equal(c.kq[0, :64], x.astype(np.int8))
    sumsq = (x.astype(np.int64) ** 2).sum(axis=0)
    want = np.sqrt(sumsq.astype(np.float64) / 64.0).astype(f32)  # double rounding is safe for sqrt
    c.freeze()
    assert np.array_equal(c.kcol[0], want)
    assert np.array_equal(c.vcol[0], want)


def test_freeze_trigger_is_start_of_65th_append():
    """[cortiq] append: the freeze runs at the START of an append once seq_len >=
    KV_COL_WARMUP (64) and no field is set; after exactly 64 rows the cache is
    still unfrozen, the 65th append freezes over the first 64 rows."""
    hd, n_kv = 64, 2
    sig = synthetic.channel_sigma((n_kv, hd), 31)
    k = synthetic.outlier_rows(70, n_kv, hd, sig, 32)
    v = synthetic.outlier_rows(70, n_kv, hd, sig, 33)
    c = oracle.OracleSeqCache(oracle.Q8, n_kv, hd, 80)
    for p in range(64):
        c.append(k[p], v[p])
    assert not c.frozen and np.all(c.kcol == 1.0)
    c.append(k[64], v[64])
    assert c.frozen and c.seq_len == 65
    # the field is the RMS of the 64 dequantised rows, not of 65
    ref = oracle.OracleSeqCache(oracle.Q8, n_kv, hd, 80)
    for p in range(64):
        ref.append(k[p], v[p])
    deq = np.stack([[ref.row(h, p, False) for p in range(64)] for h in range(n_kv)])
    rms = np.sqrt((deq.astype(np.float32) ** 2).astype(np.float64).mean(axis=1))
    assert np.allclose(c.kcol, rms, rtol=1e-5)


def test_freeze_requantised_rows_stay_within_compound_bound():
    """Rows requantised at the freeze are re-read from their dequantised values, so
    relative to the ORIGINAL input the error is bounded by s/2 + s'*col/2 (the
    bound compounds); rows appended after the freeze are quantised once against
    col and obey s'*col/2."""
    hd = 128
    sig = synthetic.channel_sigma((1, hd), 41)
    k = synthetic.outlier_rows(100, 1, hd, sig, 42)
    c = oracle.OracleSeqCache(oracle.Q8K, 1, hd, 128)
    pre = oracle.OracleSeqCache(oracle.Q8K, 1, hd, 128)
    for p in range(100):
        c.append(k[p], k[p])
        if p < 64:
            pre.append(k[p], k[p])
    col = c.kcol[0].astype(np.float64)
    for p in range(100):
        s_new = np.repeat(c.ks[0, p], 32).astype(np.float64)
        err = np.abs(c.row(0, p, False) - k[p, 0])
        if p < 64:
            s_old = np.repeat(pre.ks[0, p], 32).astype(np.float64)
            assert np.all(err <= s_old / 2 + s_new * col / 2 + 1e-5 * np.abs(k[p, 0]))
        else:
            assert np.all(err <= s_new * col / 2 * (1 + 1e-5) + 1e-6 * np.abs(k[p, 0]))


def test_page_channel_structure_and_q8_grid_tolerance():
    """[cortiq] test q8_attend_matches_f32_within_grid, with the page's hash rows
    (even channels x4, odd x1/4), its query and its tolerances.  The frozen K
    field must also follow the 16:1 even/odd channel RMS ratio."""
    g = load_golden("q8_grid.txt")
    heads, hd, P = int(g["heads"]), int(g["hd"]), int(g["positions"])

    def synth(p, salt):
        i = np.arange(heads * hd)
        x = ((i * 31 + p * 17 + salt * 7 + 3) % 97).astype(f32) / f32(97.0) - f32(0.5)
        return np.where(i % 2 == 0, x * f32(4.0), x * f32(0.25)).astype(f32).reshape(heads, hd)

    fc = oracle.OracleSeqCache(oracle.F32, heads, hd, P)
    qc = oracle.OracleSeqCache(oracle.Q8, heads, hd, P)
    for p in range(P):
        k, v = synth(p, 1), synth(p, 2)
        fc.append(k, v)
        qc.append(k, v)
    assert qc.frozen
    ratio = qc.kcol[:, 0::2].mean() / qc.kcol[:, 1::2].mean()
    assert 12.0 < ratio < 20.0
    q = (((np.arange(hd) * 13 + 5) % 89).astype(f32) / f32(89.0) - f32(0.5)).astype(f32)
    scale = f32(1.0) / f32(math.sqrt(hd))
    for kvh in range(heads):
        of, pf = fc.attend_head(q, kvh, scale)
        o8, p8 = qc.attend_head(q, kvh, scale)
        m = max(np.max(np.abs(of)), 1e-6)
        assert np.all(np.abs(of - o8) <= m * float(g["out_rel_tol"]) + float(g["out_abs_tol"]))
        assert np.all(np.abs(pf - p8) < float(g["prob_tol"]))
    assert qc.memory_bytes() * int(g["memory_factor"]) < fc.memory_bytes()


# ------------------------------------------------------------ layout/memory

def test_layout_and_memory_page_values():
    """[cortiq] tests append_tracks_seq_len_and_layout and dead_head_stores_nothing."""
    g = load_golden("cortiq_memory.txt")
    H, hd = int(g["layout_heads"]), int(g["layout_hd"])
    c = oracle.OracleSeqCache(oracle.F32, H, hd, 4)
    k = np.arange(H * hd, dtype=f32).reshape(H, hd)
    c.append(k, np.full((H, hd), 2.0, f32))
    assert c.seq_len == 1 and c.head_rows[0] == 1
    assert np.array_equal(c.k[1, 0], k[1])
    assert c.memory_bytes() == int(g["layout_bytes"])
    H, hd = int(g["dead_heads"]), int(g["dead_hd"])
    c = oracle.OracleSeqCache(oracle.F32, H, hd, 4, alive=[1, 0])
    for _ in range(2):
        c.append(np.ones((H, hd), f32), np.full((H, hd), 2.0, f32))
    assert c.seq_len == 2 and c.head_rows[0] == 2 and c.head_rows[1] == 0
    assert c.memory_bytes() == int(g["dead_bytes"])


@pytest.mark.parametrize("hd,lo,hi", [(128, 3.70, 3.72), (64, 3.65, 3.67)])
def test_q8_memory_ratio(hd, lo, hi):
    """[cortiq] KvMode doc: q8_2f is ~3.7x smaller than f32.  Per position per head:
    f32 = 8*hd bytes; q8 = 2*hd codes + 4*(hd/32) K scales + 4 V scale."""
    g = load_golden("cortiq_memory.txt")
    n = 4096
    fc = oracle.OracleSeqCache(oracle.F32, 1, hd, n)
    qc = oracle.OracleSeqCache(oracle.Q8, 1, hd, n)
    # memory_bytes only counts rows, so fill head_rows directly (no values needed)
    fc.head_rows[0] = n
    qc.head_rows[0] = n
    ratio = fc.memory_bytes() / qc.memory_bytes()
    assert lo < ratio < hi
    assert abs(ratio - float(g["q8_ratio_approx"])) < 0.06


# ---------------------------------------------------------------- attention

def _softmax_ref(q, K, V, scale):
    """Library cross-check: scipy's softmax over numpy f64 scores."""
    from scipy.special import softmax

    w = softmax(np.float64(scale) * (K @ q.astype(np.float64)))
    return w @ V, w


@pytest.mark.parametrize("mode", [oracle.F32, oracle.Q8, oracle.Q8K, oracle.Q8V])
def test_attend_matches_scipy_on_dequantised_rows(mode):
    hd, n_kv, hpk, L = 64, 2, 3, 90
    sig = synthetic.channel_sigma((n_kv, hd), 51)
    k = synthetic.outlier_rows(L, n_kv, hd, sig, 52)
    v = synthetic.outlier_rows(L, n_kv, hd, sig, 53)
    c = oracle.OracleSeqCache(mode, n_kv, hd, L)
    c.append_rows(k, v)
    q = synthetic.normal((n_kv * hpk, hd), 54)
    scale = f32(1.0) / f32(math.sqrt(hd))
    imp = np.zeros(L, np.float64)
    out = c.decode(q, n_kv * hpk, scale, imp)
    imp_ref = np.zeros(L)
    for h in range(n_kv * hpk):
        g = h // hpk
        K, V = c.dequant(g, False), c.dequant(g, True)
        o, w = _softmax_ref(q[h], K, V, scale)
        assert np.allclose(out[h], o, rtol=1e-12, atol=1e-12)
        imp_ref += w
    assert np.allclose(imp, imp_ref, rtol=1e-12, atol=1e-15)
    # weights sum to one per head -> imp sums to the number of live Q heads
    assert abs(imp.sum() - n_kv * hpk) < 1e-9
    if mode == oracle.F32:  # f32 rows are used as stored
        assert np.array_equal(c.dequant(1, False), k[:, 1].astype(np.float64))


def test_dead_group_zero_output_and_untouched_imp():
    hd, n_kv, hpk, L = 32, 4, 2, 20
    alive = [1, 0, 1, 0]
    c = oracle.OracleSeqCache(oracle.Q8, n_kv, hd, L, alive=alive)
    c.append_rows(synthetic.normal((L, n_kv, hd), 61), synthetic.normal((L, n_kv, hd), 62))
    assert c.head_rows.tolist() == [L, 0, L, 0]
    imp = np.full(L, 0.25)
    out = c.decode(synthetic.normal((n_kv * hpk, hd), 63), n_kv * hpk, f32(0.125), imp)
    assert not out[2:4].any() and not out[6:8].any()
    assert abs(imp.sum() - (0.25 * L + 2 * hpk)) < 1e-9


def test_grouped_equals_per_head_bitwise():
    """[cortiq] test attend_group_equals_per_head_attend_bitexact (oracle side)."""
    hd, n_kv, hpk, L = 32, 2, 3, 70
    for mode in (oracle.F32, oracle.Q8):
        c = oracle.OracleSeqCache(mode, n_kv, hd, L)
        c.append_rows(synthetic.normal((L, n_kv, hd), 71), synthetic.normal((L, n_kv, hd), 72))
        q = synthetic.normal((n_kv * hpk, hd), 73)
        for g in range(n_kv):
            imp = np.zeros(L)
            out = c.attend_group(q[g * hpk:(g + 1) * hpk], g, f32(0.17), imp)
            imp_ref = np.zeros(L)
            for h in range(hpk):
                o, p = c.attend_head(q[g * hpk + h], g, f32(0.17))
                assert np.array_equal(out[h], o)
                imp_ref += p
            assert np.array_equal(imp, imp_ref)


def test_parallel_decode_is_bitwise_the_serial_decode():
    """[rswa] test parallel_heads_are_bit_identical_to_serial, for the oracle's
    multi-sequence driver: the (sequence, head) pairs shared among threads give
    the serial decode's outputs and imp bit for bit, with dead groups, an empty
    sequence and every storage mode, at 1 and several threads."""
    hd, n_kv, hpk = 32, 4, 3
    lengths = [70, 0, 1, 130]
    alive = [1, 0, 1, 1]
    for mode in (oracle.F32, oracle.Q8, oracle.Q8K, oracle.Q8V):
        caches = []
        for b, L in enumerate(lengths):
            c = oracle.OracleSeqCache(mode, n_kv, hd, max(L, 1), alive=alive)
            c.append_rows(synthetic.normal((L, n_kv, hd), 80 + b), synthetic.normal((L, n_kv, hd), 90 + b))
            caches.append(c)
        qs = [synthetic.normal((n_kv * hpk, hd), 100 + b) for b in range(len(lengths))]
        ref_out, ref_imp = [], []
        for c, q in zip(caches, qs):
            imp = np.full(c.cap, 0.5)
            ref_out.append(c.decode(q, n_kv * hpk, f32(0.2), imp))
            ref_imp.append(imp)
        for threads in (1, 3, 0):
            imps = [np.full(c.cap, 0.5) for c in caches]
            outs, used = oracle.decode_many(caches, qs, n_kv * hpk, f32(0.2), imps, threads)
            assert used >= 1
            for b in range(len(lengths)):
                assert np.array_equal(outs[b], ref_out[b]), (mode, threads, b)
                assert np.array_equal(imps[b], ref_imp[b]), (mode, threads, b)
            outs, _ = oracle.decode_many(caches, qs, n_kv * hpk, f32(0.2), None, threads)
            assert all(np.array_equal(o, r) for o, r in zip(outs, ref_out))


def test_closed_forms_single_key_and_equal_scores():
    """1 key -> its V; equal scores -> the mean of the V rows (for any query)."""
    c = oracle.OracleSeqCache(oracle.F32, 1, 16, 4)
    c.append(np.eye(16, dtype=f32)[0][None], np.full((1, 16), 7.0, f32))
    out, p = c.attend_head(np.arange(16, dtype=f32), 0, f32(0.25))
    assert np.all(out == 7.0) and p.tolist() == [1.0]
    c.append(np.eye(16, dtype=f32)[0][None], np.full((1, 16), 4.0, f32))
    c2 = oracle.OracleSeqCache(oracle.F32, 1, 16, 4)
    c2.append(np.eye(16, dtype=f32)[0][None], np.full((1, 16), 2.0, f32))
    c2.append(np.eye(16, dtype=f32)[0][None], np.full((1, 16), 4.0, f32))
    out, p = c2.attend_head(np.full(16, 3.0, f32), 0, f32(0.25))
    assert np.allclose(out, 3.0, rtol=0, atol=1e-15) and np.allclose(p, 0.5)


# ------------------------------------------- window / softcap / sinks options

def _ex_cache(mode=oracle.F32, L=40, hd=32, n_kv=2, seed=81):
    c = oracle.OracleSeqCache(mode, n_kv, hd, L)
    c.append_rows(synthetic.normal((L, n_kv, hd), seed), synthetic.normal((L, n_kv, hd), seed + 1))
    return c


def test_ex_defaults_equal_attend_group():
    """first = 0, no cap, no sinks is [cortiq] attend_group itself, bit for bit."""
    for mode in (oracle.F32, oracle.Q8):
        c = _ex_cache(mode)
        q = synthetic.normal((3, 32), 91)
        i1, i2 = np.zeros(40), np.zeros(40)
        a = c.attend_group(q, 1, f32(0.2), i1)
        b = c.attend_group_ex(q, 1, f32(0.2), 0, 0.0, None, i2)
        assert np.array_equal(a, b) and np.array_equal(i1, i2)


def test_sink_single_row_closed_form():
    """[cortiq] attend_group_upto: one stored row and a sink z: the row gets
    e^s / (e^s + e^z) of the mass, the sink's share has no value row."""
    c = oracle.OracleSeqCache(oracle.F32, 1, 8, 2)
    k = np.array([[[0.5, -1.0, 0.25, 2.0, 0.0, 1.0, -0.5, 0.75]]], f32)
    v = np.array([[[1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0]]], f32)
    c.append_rows(k, v)
    q = np.array([[1.0, 0.5, -2.0, 0.25, 3.0, -1.0, 0.5, 1.0]], f32)
    sc, z = f32(0.35), f32(-0.8)
    s = float(sc) * float(np.dot(q[0].astype(np.float64), k[0, 0].astype(np.float64)))
    share = math.exp(s) / (math.exp(s) + math.exp(float(z)))
    imp = np.zeros(2)
    out = c.attend_group_ex(q, 0, sc, 0, 0.0, np.array([z]), imp)
    assert np.allclose(out[0], share * v[0, 0].astype(np.float64), rtol=1e-14, atol=0)
    assert abs(imp[0] - share) < 1e-15 and imp[1] == 0.0


def test_sink_scales_output_by_visible_mass():
    """A sink only adds to the denominator: out_sink = out_plain * (visible
    mass), and that mass is what imp receives; a sink far below every score
    changes nothing."""
    c = _ex_cache(oracle.Q8, L=50, seed=95)
    q = synthetic.normal((4, 32), 96)
    plain = c.attend_group_ex(q, 0, f32(0.3))
    sinks = np.array([0.5, -2.0, 3.0, 0.0], f32)
    for h in range(4):
        imp = np.zeros(50)
        o = c.attend_group_ex(q[h:h + 1], 0, f32(0.3), 0, 0.0, sinks[h:h + 1], imp)
        mass = imp.sum()
        assert 0.0 < mass < 1.0
        assert np.allclose(o[0], plain[h] * mass, rtol=1e-12, atol=1e-15)
    far = c.attend_group_ex(q, 0, f32(0.3), 0, 0.0, np.full(4, -1e4, f32))
    assert np.array_equal(far, plain)


def test_window_equals_the_visible_suffix():
    """[cortiq] attend_group_upto: rows before `first` get probability 0, so the
    result equals attending a cache that holds only rows [first, stored); their
    imp entries are untouched."""
    L, f, hd = 40, 13, 32
    k = synthetic.normal((L, 2, hd), 97)
    v = synthetic.normal((L, 2, hd), 98)
    full = oracle.OracleSeqCache(oracle.F32, 2, hd, L)
    full.append_rows(k, v)
    tail = oracle.OracleSeqCache(oracle.F32, 2, hd, L)
    tail.append_rows(np.ascontiguousarray(k[f:]), np.ascontiguousarray(v[f:]))
    q = synthetic.normal((3, hd), 99)
    imp = np.full(L, 0.5)
    imp_t = np.zeros(L)
    out = full.attend_group_ex(q, 1, f32(0.25), f, 0.0, None, imp)
    ref = tail.attend_group(q, 1, f32(0.25), imp_t)
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-15)
    assert np.all(imp[:f] == 0.5)
    assert np.allclose(imp[f:] - 0.5, imp_t[:L - f], rtol=1e-12, atol=1e-15)


def test_window_clamps_to_the_last_row():
    """first >= stored is clamped to stored - 1: the last row alone, weight 1."""
    c = _ex_cache(oracle.F32, L=10, hd=32)
    q = synthetic.normal((2, 32), 100)
    imp = np.zeros(10)
    out = c.attend_group_ex(q, 0, f32(0.5), 25, 0.0, None, imp)
    last = c.dequant(0, True)[9]
    assert np.allclose(out, np.stack([last, last]), rtol=0, atol=1e-15)
    assert imp[:9].sum() == 0.0 and abs(imp[9] - 2.0) < 1e-15


def test_softcap_two_rows_closed_form():
    """The cap applies to the scaled score: with two rows the weight ratio is
    exp(c tanh(s1 / c) - c tanh(s2 / c)), s = scale * <q, k>."""
    c = oracle.OracleSeqCache(oracle.F32, 1, 4, 2)
    k = np.array([[[2.0, 0.0, 1.0, 0.0]], [[-1.0, 3.0, 0.0, 0.5]]], f32)
    c.append_rows(k, np.ones((2, 1, 4), f32))
    q = np.array([[1.5, -0.5, 2.0, 1.0]], f32)
    sc, cap = f32(0.9), 1.25
    s = [float(sc) * float(np.dot(q[0].astype(np.float64), k[i, 0].astype(np.float64))) for i in range(2)]
    imp = np.zeros(2)
    c.attend_group_ex(q, 0, sc, 0, cap, None, imp)
    want = math.exp(cap * math.tanh(s[0] / cap) - cap * math.tanh(s[1] / cap))
    assert abs(imp[0] / imp[1] - want) < 1e-12 * want


def test_softcap_limits_and_bound():
    """Gemma-2 soft-capping: a huge cap is the plain softmax; a small cap keeps
    every score inside (-c, c), so no two weights differ by more than e^(2c),
    which the uncapped scores here exceed by far."""
    c = _ex_cache(oracle.F32, L=30, hd=32, seed=101)
    q = (synthetic.normal((2, 32), 102) * 8.0).astype(f32)
    plain_imp, big_imp = np.zeros(30), np.zeros(30)
    plain = c.attend_group_ex(q, 1, f32(0.4), 0, 0.0, None, plain_imp)
    big = c.attend_group_ex(q, 1, f32(0.4), 0, 1e7, None, big_imp)
    assert np.allclose(big, plain, rtol=1e-9, atol=1e-12)
    cap = 0.75
    for h in range(2):
        imp_c, imp_p = np.zeros(30), np.zeros(30)
        c.attend_group_ex(q[h:h + 1], 1, f32(0.4), 0, cap, None, imp_c)
        c.attend_group_ex(q[h:h + 1], 1, f32(0.4), 0, 0.0, None, imp_p)
        assert imp_c.max() / imp_c.min() <= math.exp(2 * cap) * (1 + 1e-12)
        assert imp_p.max() / imp_p.min() > math.exp(2 * cap) * 10


# ------------------------------------------------------------------- R-SWA

H, HD, W = 10, 128, 128


def _fill(seq, f):
    out = np.zeros((H, seq, HD), f32)
    for r in range(seq):
        for d in range(HD):
            out[:, r, d] = f(r, d)
    return out


def _token(f):
    out = np.zeros((H, HD), f32)
    for d in range(HD):
        out[:, d] = f(d)
    return out


def _rswa_state(cap):
    return (np.zeros((H, cap, HD), f32), np.zeros((H, cap, HD), f32),
            np.zeros((H, W, HD), f32), np.zeros((H, W, HD), f32), np.zeros(2, np.int32))


def test_rswa_page_closed_forms():
    g = load_golden("rswa_closed_forms.txt")
    assert (int(g["num_heads"]), int(g["head_dim"]), int(g["ring_window"])) == (H, HD, W)
    scale = f32(1.0) / f32(math.sqrt(HD))
    e0 = lambda r, d: 1.0 if d == 0 else 0.0
    # single key
    rk, rv, gk, gv, cur = _rswa_state(8)
    rk[:, :1] = _fill(1, e0)
    rv[:, :1] = 7.0
    out = oracle.rswa_decode(_token(lambda d: 5.0 if d == 0 else 0.0), rk, rv, 1, gk, gv, 0, scale)
    assert np.all(np.abs(out - float(g["single_key_value"])) < float(g["single_key_tol"]))
    # equal scores
    rk, rv, gk, gv, cur = _rswa_state(8)
    rk[:, :2] = _fill(2, e0)
    rv[:, :2] = _fill(2, lambda r, d: 2.0 if r == 0 else 4.0)
    out = oracle.rswa_decode(_token(lambda d: 3.0 if d == 0 else 0.0), rk, rv, 2, gk, gv, 0, scale)
    assert np.all(np.abs(out - float(g["equal_scores_value"])) < float(g["equal_scores_tol"]))
    # write-then-attend (the query sees its own ring token)
    rk, rv, gk, gv, cur = _rswa_state(8)
    rk[:, :1] = _fill(1, lambda r, d: 1.0 if d == 1 else 0.0)
    rv[:, :1] = 1.0
    slot = oracle.rswa_write(gk, gv, _token(lambda d: 1.0 if d == 0 else 0.0),
                             _token(lambda d: 5.0), True, cur)
    assert slot == 0 and cur[0] == 1
    out = oracle.rswa_decode(_token(lambda d: 10.0 if d == 0 else 0.0), rk, rv, 1, gk, gv, cur[0], scale)
    approx = float(g["ring_entry_approx"])
    assert np.all(np.abs(out - approx) < 1e-3) and np.all(out > 3.0)
    w = math.exp(10.0 / math.sqrt(128.0))
    assert np.all(np.abs(out - (w * 5 + 1) / (w + 1)) < float(g["ring_entry_tol"]))


def test_rswa_online_fold_matches_two_pass():
    """[rswa] test online_matches_naive_softmax: the streaming fold (f32, page
    order) and the materialised two-pass definition agree within 1e-4."""
    g = load_golden("rswa_closed_forms.txt")
    m = 5
    keys = _fill(m, lambda r, d: float(r + 1) if d == 0 else 0.0)[0]
    vals = _fill(m, lambda r, d: r + d * 0.01)[0]
    q = np.zeros(HD, f32)
    q[0] = 0.5
    scale = f32(1.0) / f32(math.sqrt(HD))
    online = oracle.online_head(q, keys, vals, scale)
    rk, rv, gk, gv, _ = _rswa_state(16)
    rk[:, :m] = keys
    rv[:, :m] = vals
    two_pass = oracle.rswa_decode(np.tile(q, (H, 1)), rk, rv, m, gk, gv, 0, scale)[0]
    assert abs(online[0] - two_pass[0]) < float(g["online_vs_naive_tol"])
    assert np.max(np.abs(online - two_pass)) < 1e-5


def test_rswa_cursor_sequence():
    g = load_golden("ring_cursors.txt")
    rk, rv, gk, gv, cur = _rswa_state(4)
    for step in range(W):
        slot = oracle.rswa_write(gk, gv, _token(lambda d: float(step)), _token(lambda d: 0.0), True, cur)
        assert slot == step and cur[0] == step + 1
        # write_decode_step doc: during warm-up ring_pos tracks ring_len (mod W)
        assert cur[1] == (step + 1) % W
    assert cur[1] == int(g["warm_ring_pos_after_w"])
    slots, pos = [], []
    for _ in range(2):
        slots.append(oracle.rswa_write(gk, gv, _token(lambda d: 99.0), _token(lambda d: 99.0), True, cur))
        pos.append(int(cur[1]))
    assert slots == [int(s) for s in g["steady_slots"].split()]
    assert pos == [int(s) for s in g["steady_ring_pos"].split()]
    assert cur[0] == W and gk[0, 0, 0] == 99.0
    for expect in list(range(2, W)) + [0, 1]:
        assert oracle.rswa_write(gk, gv, _token(lambda d: 0.0), _token(lambda d: 0.0), True, cur) == expect
    assert cur[1] == 2


def test_rswa_errors():
    rk, rv, gk, gv, cur = _rswa_state(4)
    with pytest.raises(RuntimeError):
        oracle.rswa_write(gk, gv, _token(lambda d: 1.0), _token(lambda d: 1.0), False, cur)
    assert cur.tolist() == [0, 0]
    with pytest.raises(RuntimeError):
        oracle.rswa_decode(_token(lambda d: 1.0), rk, rv, None, gk, gv, 0, f32(0.1))
    with pytest.raises(RuntimeError):
        oracle.rswa_decode(_token(lambda d: 1.0), rk, rv, 0, gk, gv, 0, f32(0.1))


def rope(x, pos, base=10000.0):
    """Standard pairwise rotary embedding of the last axis at absolute position pos
    (test harness only: the pages leave RoPE to the caller)."""
    hd = x.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    th = pos * base ** (-2.0 * i / hd)
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., 0::2].astype(np.float64), x[..., 1::2].astype(np.float64)
    out = np.empty(x.shape, np.float64)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out.astype(f32)


def test_rswa_steady_state_is_prefix_plus_last_w_with_absolute_rope():
    """R-SWA module doc: after the ring wraps, decode equals brute-force attention
    over prefix ++ the last W generated rows (in logical order), with RoPE at
    the TRUE absolute position.  A slot-indexed RoPE must fail (teeth)."""
    m, steps = 37, 500
    prefix_k = synthetic.normal((H, m, HD), 81)
    prefix_v = synthetic.normal((H, m, HD), 82)
    gen_k = synthetic.normal((steps, H, HD), 83)
    gen_v = synthetic.normal((steps, H, HD), 84)
    q_raw = synthetic.normal((H, HD), 85)
    scale = f32(1.0) / f32(math.sqrt(HD))
    pk = np.stack([rope(prefix_k[:, r], r) for r in range(m)], axis=1)
    outs = {}
    for variant in ("absolute", "slot"):
        rk, rv, gk, gv, cur = _rswa_state(m)
        rk[:] = pk
        rv[:] = prefix_v
        for t in range(steps):
            slot_next = cur[0] if cur[0] < W else cur[1]
            pos = m + t if variant == "absolute" else m + slot_next
            oracle.rswa_write(gk, gv, rope(gen_k[t], pos), gen_v[t], True, cur)
        assert cur.tolist() == [W, steps % W] == [128, 116]
        qpos = m + steps - 1
        outs[variant] = oracle.rswa_decode(rope(q_raw, qpos), rk, rv, m, gk, gv, cur[0], scale)
    # brute force, logical order, absolute positions
    from scipy.special import softmax

    keep = range(steps - W, steps)
    ref = np.zeros((H, HD))
    for h in range(H):
        K = np.concatenate([pk[h], np.stack([rope(gen_k[t, h], m + t) for t in keep])]).astype(np.float64)
        V = np.concatenate([prefix_v[h], gen_v[list(keep), h]]).astype(np.float64)
        w = softmax(np.float64(scale) * (K @ rope(q_raw, m + steps - 1)[h].astype(np.float64)))
        ref[h] = w @ V
    assert np.allclose(outs["absolute"], ref, rtol=1e-10, atol=1e-12)
    assert np.max(np.abs(outs["slot"] - ref)) > 1e-3


# ------------------------------------------------- R-SWA int8 mirror (NEXT-2)

def _mirror(rk, rv, gk, gv):
    """The int8 mirror of the four f32 regions, one quantize_row_i8 per row."""
    rk8, rks = oracle.rswa_mirror(rk)
    rv8, rvs = oracle.rswa_mirror(rv)
    gk8, gks = oracle.rswa_mirror(gk)
    gv8, gvs = oracle.rswa_mirror(gv)
    return rk8, rks, rv8, rvs, gk8, gks, gv8, gvs


def _decode_i8(q, mir, pl, rl, scale):
    rk8, rks, rv8, rvs, gk8, gks, gv8, gvs = mir
    return oracle.rswa_decode_i8(q, rk8, rks, rv8, rvs, pl, gk8, gks, gv8, gvs, rl, scale)


def test_rswa_i8_lossless_rows_equal_the_f32_decode():
    """[rswa] decode_attention_int8: rows whose absmax is 127 and whose other
    entries are small integers quantise losslessly (scale 1, codes = values),
    so the int8 decode must equal the f32 definition (rswa_decode) over the
    same rows, reference and ring alike, up to f64 rounding."""
    rng = np.random.default_rng(11)
    m, n_ring = 9, 5

    def rows(shape):
        x = rng.integers(-3, 4, size=shape).astype(f32)
        x[..., 0] = 127.0
        return x

    rk, rv, gk, gv, cur = _rswa_state(16)
    rk[:, :m], rv[:, :m] = rows((H, m, HD)), rows((H, m, HD))
    for _ in range(n_ring):
        oracle.rswa_write(gk, gv, rows((H, HD)), rows((H, HD)), True, cur)
    q = rows((H, HD))
    q[:, 0] = -127.0  # the anchor may sit at either sign
    mir = _mirror(rk, rv, gk, gv)
    for codes, scales, src, n in ((mir[0], mir[1], rk, m), (mir[4], mir[5], gk, n_ring)):
        assert np.all(scales[:, :n] == f32(1.0))
        assert np.array_equal(codes[:, :n].astype(f32), src[:, :n])
    scale = f32(1e-3)
    got = _decode_i8(q, mir, m, cur[0], scale)
    ref = oracle.rswa_decode(q, rk, rv, m, gk, gv, cur[0], scale)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # the scores carry real spread (not a one-hot or uniform softmax)
    assert np.ptp(ref) > 1.0


def test_rswa_i8_dot_reaches_the_page_bound():
    """[rswa] quantize_row_i8: q = 1 and K = +-2 quantise to codes +-127 on all
    128 channels, so the i32 dot is exactly +-127*127*128 (the page's bound).
    Two keys with V rows 3 and -1 give out = -1 + 4 sigmoid(delta) with
    delta = 2 dot qscale kscale scale; solving for the dot recovers the bound."""
    g = load_golden("rswa_i8.txt")
    bound = int(g["qk_bound"])
    assert bound == 127 * 127 * int(g["head_dim"])
    rk, rv, gk, gv, _ = _rswa_state(16)
    rk[:, 0], rk[:, 1] = 2.0, -2.0
    rv[:, 0], rv[:, 1] = 3.0, -1.0
    q = np.ones((H, HD), f32)
    mir = _mirror(rk, rv, gk, gv)
    assert np.all(mir[0][:, 0] == 127) and np.all(mir[0][:, 1] == -127)
    scale = f32(1.0 / 4096.0)
    out = _decode_i8(q, mir, 2, 0, scale)
    qscale = float(f32(1.0) / f32(127.0))
    kscale = float(f32(2.0) / f32(127.0))
    v0 = 127.0 * float(f32(3.0) / f32(127.0))
    v1 = -127.0 * float(f32(1.0) / f32(127.0))
    sig = (out - v1) / (v0 - v1)
    delta = np.log(sig / (1.0 - sig))
    dot = delta / (2.0 * qscale * kscale * float(scale))
    assert np.all(np.abs(dot - bound) < 1e-3)


def test_rswa_i8_single_key_returns_the_dequantised_row():
    """One key: the softmax weight is 1, so out = V codes * V scale exactly, and
    round-to-nearest keeps it within half a step (plus the division's rounding)
    of the f32 row."""
    rk, rv, gk, gv, _ = _rswa_state(16)
    rk[:, 0] = synthetic.normal((H, HD), 91)
    rv[:, 0] = synthetic.normal((H, HD), 92)
    q = synthetic.normal((H, HD), 93)
    mir = _mirror(rk, rv, gk, gv)
    out = _decode_i8(q, mir, 1, 0, f32(0.1))
    deq = mir[2][:, 0].astype(np.float64) * mir[3][:, 0, None].astype(np.float64)
    assert np.array_equal(out, deq)
    step = mir[3][:, 0, None].astype(np.float64)
    assert np.all(np.abs(deq - rv[:, 0]) <= step * (0.5 + 1e-6))


def test_rswa_i8_zero_query_averages_reference_and_ring():
    """A zero query quantises to codes 0 with scale 1.0 (the page's zero-row
    rule), every score is 0, and the output is the plain mean of the
    dequantised V rows over the reference rows and the ring rows."""
    g = load_golden("rswa_i8.txt")
    q0, s0 = oracle.quantize_row_i8(np.zeros(HD, f32))
    assert np.all(q0 == 0) and s0 == f32(float(g["zero_row_scale"]))
    rk, rv, gk, gv, cur = _rswa_state(16)
    rk[:, :4] = synthetic.normal((H, 4, HD), 94)
    rv[:, :4] = synthetic.normal((H, 4, HD), 95)
    for t in range(3):
        oracle.rswa_write(gk, gv, synthetic.normal((H, HD), 96 + t), synthetic.normal((H, HD), 99 + t),
                          True, cur)
    mir = _mirror(rk, rv, gk, gv)
    out = _decode_i8(np.zeros((H, HD), f32), mir, 4, cur[0], f32(0.3))
    deq_ref = mir[2][:, :4].astype(np.float64) * mir[3][:, :4, None]
    deq_ring = mir[6][:, :3].astype(np.float64) * mir[7][:, :3, None]
    mean = np.concatenate([deq_ref, deq_ring], axis=1).mean(axis=1)
    assert np.allclose(out, mean, rtol=1e-12, atol=1e-12)


def test_rswa_i8_errors():
    rk, rv, gk, gv, _ = _rswa_state(4)
    mir = _mirror(rk, rv, gk, gv)
    with pytest.raises(RuntimeError):
        _decode_i8(np.ones((H, HD), f32), mir, None, 0, f32(0.1))
    with pytest.raises(RuntimeError):
        _decode_i8(np.ones((H, HD), f32), mir, 0, 0, f32(0.1))


def test_rswa_i8_ring_rows_use_their_own_scales():
    """Two ring keys of magnitudes 2 and -4 both quantise to codes +-127 and
    differ only in their row scales (2/127, 4/127); with q = 1 the scores are
    +-127*127*128 * qscale * kscale_r * scale, a closed form that fails if a
    ring row reads another row's scale."""
    rk, rv, gk, gv, cur = _rswa_state(16)
    k_rows = [np.full((H, HD), 2.0, f32), np.full((H, HD), -4.0, f32)]
    v_rows = [np.full((H, HD), 3.0, f32), np.full((H, HD), -1.0, f32)]
    for kr, vr in zip(k_rows, v_rows):
        oracle.rswa_write(gk, gv, kr, vr, True, cur)
    mir = _mirror(rk, rv, gk, gv)
    assert np.all(mir[4][:, 0] == 127) and np.all(mir[4][:, 1] == -127)
    scale = f32(1.0 / 2048.0)
    out = _decode_i8(np.ones((H, HD), f32), mir, 0, cur[0], scale)
    qs = float(f32(1.0) / f32(127.0))
    s0 = 2064512 * qs * float(f32(2.0) / f32(127.0)) * float(scale)
    s1 = -2064512 * qs * float(f32(4.0) / f32(127.0)) * float(scale)
    v0 = 127.0 * float(f32(3.0) / f32(127.0))
    v1 = -127.0 * float(f32(1.0) / f32(127.0))
    m = max(s0, s1)
    w0, w1 = math.exp(s0 - m), math.exp(s1 - m)
    assert np.allclose(out, (w0 * v0 + w1 * v1) / (w0 + w1), rtol=1e-12, atol=1e-12)


# --------------------------------------------------- Born eviction (NEXT-3)

def _ramp_cache(mode, n_kv, hd, rows, seed=0, alive=None):
    c = oracle.OracleSeqCache(mode, n_kv, hd, rows + 8, alive=alive)
    rng = np.random.default_rng(seed)
    for _ in range(rows):
        c.append(rng.normal(size=(n_kv, hd)).astype(f32), rng.normal(size=(n_kv, hd)).astype(f32))
        c.freeze_if_due()
    return c


def _snapshot(c):
    return {n: None if getattr(c, n) is None else getattr(c, n).copy() for n in ("k", "v", "kq", "ks", "vq", "vs")}


def test_born_page_example_keeps_sink_mass_and_recents():
    """[cortiq] born_eviction_keeps_high_mass_position, through KvCache::evict's
    recent = max(keep_last / 2, 1)."""
    g = load_golden("born_eviction.txt")
    n, keep = int(g["positions"]), int(g["keep_last"])
    c = oracle.OracleSeqCache(oracle.F32, 1, 2, 16)
    for pos in range(n):
        c.append(np.full((1, 2), pos, f32), np.full((1, 2), pos + 100.0, f32))
    imp = np.full(16, f32(float(g["light_mass"])), f32)
    imp[int(g["heavy_position"])] = f32(float(g["heavy_mass"]))
    kept = c.evict_born(keep, int(g["sink"]), max(keep // 2, 1), imp)
    expect = [float(x) for x in g["kept_keys"].split()]
    assert kept == keep == c.seq_len and c.head_rows[0] == keep
    assert c.k[0, :keep, 0].tolist() == expect
    assert c.v[0, :keep, 0].tolist() == [x + 100.0 for x in expect]
    assert imp[:keep].tolist() == [float(imp_v) for imp_v in
                                   np.array([0.05, 5.0, 0.05, 0.05], f32)]


@pytest.mark.parametrize("mode", [oracle.Q8K, oracle.Q8V])
def test_born_mixed_modes_gather_every_storage(mode):
    """[cortiq] born_eviction_mixed_modes_stay_consistent: K and V live in
    different storages in q8k / q8v; both are gathered, memory shrinks below
    half, and the kept V rows are the heavy tail's."""
    g = load_golden("born_eviction.txt")
    n = int(g["mixed_appends"])
    c = oracle.OracleSeqCache(mode, 1, 4, n)
    for p in range(n):
        c.append(np.full((1, 4), p * 0.01, f32), np.full((1, 4), float(p), f32))
        c.freeze_if_due()
    imp = np.arange(n, dtype=f32)
    before = c.memory_bytes()
    keep = int(g["mixed_keep"])
    assert c.evict_born(keep, int(g["mixed_sink"]), int(g["mixed_recent"]), imp) == keep
    assert c.head_rows[0] == keep and c.memory_bytes() < before / 2
    out = c.attend_group(np.ones((1, 4), f32), 0, f32(1.0))
    assert out[0, 0] > float(g["mixed_out_min"])
    # sinks 0..3, the 8 heaviest middle rows 64..71, the recents 72..79
    assert imp[:keep].tolist() == list(range(4)) + list(range(64, 80))


def test_born_is_a_no_op_at_or_under_budget():
    c = _ramp_cache(oracle.Q8, 2, 64, 70, seed=1)
    snap, imp = _snapshot(c), np.arange(78, dtype=f32)
    assert c.evict_born(70, 4, 8, imp.copy()) == 70 and c.evict_born(100, 4, 8, imp) == 70
    for k, v in snap.items():
        assert v is None or np.array_equal(getattr(c, k), v)


@pytest.mark.parametrize("mode", [oracle.F32, oracle.Q8, oracle.Q8K, oracle.Q8V])
def test_born_gathers_kept_rows_of_every_storage(mode):
    """Equal mass everywhere: ties keep the lowest middle positions (the page's
    stable sort), so the kept set is [0, s) + [s, s + budget) + the recents;
    every storage of every live head (a dead head stores nothing) holds the
    pre-eviction rows at those positions, in order, and imp follows them."""
    c = _ramp_cache(mode, 3, 64, 150, seed=2, alive=[1, 0, 1])
    snap = _snapshot(c)
    imp = np.full(158, 0.25, f32)
    imp[150:] = 99.0  # beyond the stored rows: never read
    keep, sink, recent = 40, 3, 10
    assert c.evict_born(keep, sink, recent, imp) == keep
    kept = list(range(sink)) + list(range(sink, sink + keep - sink - recent)) + list(range(140, 150))
    assert len(kept) == keep and np.all(imp[:keep] == f32(0.25))
    assert np.all(imp[keep:150] == 0.0) and np.all(imp[150:] == f32(99.0))  # dropped rows cleared
    for name, before in snap.items():
        if before is None:
            continue
        for h in (0, 2):
            assert np.array_equal(getattr(c, name)[h, :keep], before[h, kept]), (name, h)
    assert c.head_rows.tolist() == [keep, 0, keep]


def test_born_mass_order_and_clamps():
    """Increasing mass keeps the sinks and the last rows; sink >= keep_last
    keeps the first keep_last rows only; sink + recent > keep_last clamps the
    recents; the middle picks follow the mass, not the position."""
    def run(keep, sink, recent, imp_fn, n=60):
        c = oracle.OracleSeqCache(oracle.F32, 1, 32, n + 4)
        for p in range(n):
            c.append(np.full((1, 32), p, f32), np.full((1, 32), p, f32))
        imp = np.array([imp_fn(p) for p in range(n + 4)], f32)
        c.evict_born(keep, sink, recent, imp)
        return c.k[0, :keep, 0].astype(int).tolist()

    assert run(12, 2, 3, lambda p: p) == [0, 1] + list(range(50, 60))
    assert run(12, 20, 3, lambda p: p) == list(range(12))
    assert run(12, 5, 30, lambda p: p) == list(range(5)) + list(range(53, 60))
    # mass peaks at positions 30, 10, 20 (in that order of mass), budget 3
    peaks = {30: 9.0, 10: 8.0, 20: 7.0, 40: 1.0}
    assert run(8, 2, 3, lambda p: peaks.get(p, 0.0)) == [0, 1, 10, 20, 30, 57, 58, 59]
    # a tie at the threshold goes to the lower position
    ties = {25: 5.0, 15: 3.0, 35: 3.0, 45: 3.0}
    assert run(7, 2, 3, lambda p: ties.get(p, 0.0)) == [0, 1, 15, 25, 57, 58, 59]


def test_truncate_last_page_example_and_resume():
    """[cortiq] truncate_rolls_back_speculative_positions; then an append lands at
    the freed position, its mass starts from zero, and dropping more rows than
    are stored empties the sequence."""
    g = load_golden("born_eviction.txt")
    c = oracle.OracleSeqCache(oracle.F32, 2, 4, 16)
    for pos in range(int(g["trunc_appends"])):
        c.append(np.full((2, 4), pos, f32), np.full((2, 4), pos, f32))
    imp = np.arange(16, dtype=f32) + 1
    assert c.truncate_last(int(g["trunc_drop"]), imp) == int(g["trunc_left"]) == c.seq_len
    assert c.head_rows.tolist() == [3, 3] and c.k[0, 2, 0] == 2.0
    assert imp[:3].tolist() == [1, 2, 3] and imp[3:5].tolist() == [0, 0] and imp[5] == 6
    c.append(np.full((2, 4), 9.0, f32), np.full((2, 4), 9.0, f32))
    assert c.seq_len == 4 and c.k[1, 3, 0] == 9.0
    out = c.attend_group(np.zeros((1, 4), f32), 0, f32(1.0))
    assert np.allclose(out[0], (0 + 1 + 2 + 9) / 4.0)  # the dropped rows are gone
    assert c.truncate_last(10, imp) == 0 and c.head_rows.tolist() == [0, 0]


# ------------------------------------------------ verify / upto (NEXT-4)

def test_upto_equals_a_truncated_cache_and_limits():
    """[cortiq] attend_group_upto's upto: attending rows [0, upto) equals attending
    a copy truncated to upto rows (truncate_last is pinned on its own); upto at
    or above the stored rows changes nothing; upto 0 gives zeros; upto 1 returns
    the first row's dequantised value."""
    c = _ramp_cache(oracle.Q8, 2, 64, 120, seed=5)
    t = _ramp_cache(oracle.Q8, 2, 64, 120, seed=5)
    q = synthetic.normal((3, 64), 6)
    sc = f32(0.125)
    for u in (119, 90, 64, 2):
        t.truncate_last(t.seq_len - u)
        for first, cap_, sk in ((0, 0.0, None), (u // 2, 1.5, np.array([0.3, -1.0, 2.0], f32))):
            got = c.attend_group_ex(q, 1, sc, first, cap_, sk, None, u)
            ref = t.attend_group_ex(q, 1, sc, first, cap_, sk, None)
            assert np.array_equal(got, ref), (u, first)
    base = c.attend_group_ex(q, 0, sc)
    assert np.array_equal(c.attend_group_ex(q, 0, sc, upto=120), base)
    assert np.array_equal(c.attend_group_ex(q, 0, sc, upto=10 ** 6), base)
    assert not c.attend_group_ex(q, 0, sc, upto=0).any()
    one = c.attend_group_ex(q, 0, sc, upto=1)
    assert np.allclose(one, np.tile(c.row(0, 0, True), (3, 1)), rtol=1e-14, atol=0)


def test_verify_equals_sequential_decodes():
    """Query-batched verify of K = 4 drafts (causal among them) equals decoding
    after each draft's append in turn, with a window counted back from each
    query's position, soft-capping and sinks."""
    n_kv, hd, n_q, K = 2, 64, 6, 4
    c_seq = _ramp_cache(oracle.F32, n_kv, hd, 70, seed=7)
    c_bat = _ramp_cache(oracle.F32, n_kv, hd, 70, seed=7)
    drafts = [(synthetic.normal((n_kv, hd), 20 + i), synthetic.normal((n_kv, hd), 30 + i)) for i in range(K)]
    q = synthetic.normal((K, n_q, hd), 40)
    sinks = synthetic.normal((n_q,), 41)
    sc = f32(0.125)
    seq = []
    for k in range(K):
        c_seq.append(*drafts[k])
        seq.append(c_seq.decode_ex(q[k], n_q, sc, window=33, softcap=2.0, sinks=sinks))
    for d in drafts:
        c_bat.append(*d)
    bat = c_bat.decode_verify(q, n_q, K, sc, window=33, softcap=2.0, sinks=sinks)
    assert np.allclose(bat, np.stack(seq), rtol=1e-13, atol=1e-15)
    # K = 1 is the plain decode
    assert np.array_equal(c_bat.decode_verify(q[3:], n_q, 1, sc)[0], c_bat.decode(q[3], n_q, sc))


def test_rswa_verify_is_brute_force_over_the_last_w_rows():
    """[rswa] verify_attention: query i sees the reference rows and the last W
    rows of (live ring in logical order ++ drafts 0..i), in a warm ring (no
    overwrite), a ring that fills during the drafts, and a full ring (each
    draft evicts the oldest row); the caller's ring and cursors stay untouched.
    Brute force: scipy softmax over the explicit key list."""
    from scipy.special import softmax

    m, K = 11, 5
    scale = f32(1.0) / f32(math.sqrt(HD))
    for n_gen in (40, 125, 300):
        rk, rv, gk, gv, cur = _rswa_state(16)
        rk[:, :m] = synthetic.normal((H, m, HD), 110)
        rv[:, :m] = synthetic.normal((H, m, HD), 111)
        gen_k = synthetic.normal((n_gen, H, HD), 112)
        gen_v = synthetic.normal((n_gen, H, HD), 113)
        for t in range(n_gen):
            oracle.rswa_write(gk, gv, gen_k[t], gen_v[t], True, cur)
        dq = synthetic.normal((K, H, HD), 114)
        dk = synthetic.normal((K, H, HD), 115)
        dv = synthetic.normal((K, H, HD), 116)
        snap = (gk.copy(), gv.copy(), cur.copy())
        got = oracle.rswa_verify(dq, dk, dv, rk, rv, m, gk, gv, cur, scale)
        assert np.array_equal(gk, snap[0]) and np.array_equal(gv, snap[1]) and np.array_equal(cur, snap[2])
        for i in range(K):
            keys_k = np.concatenate([gen_k, dk[:i + 1]])[-W:]
            keys_v = np.concatenate([gen_v, dv[:i + 1]])[-W:]
            for h in range(H):
                Kh = np.concatenate([rk[h, :m], keys_k[:, h]]).astype(np.float64)
                Vh = np.concatenate([rv[h, :m], keys_v[:, h]]).astype(np.float64)
                w = softmax(np.float64(scale) * (Kh @ dq[i, h].astype(np.float64)))
                assert np.allclose(got[i, h], w @ Vh, rtol=1e-11, atol=1e-13), (n_gen, i, h)


def test_rswa_verify_int8_on_lossless_rows_equals_f32():
    """The int8 verify (drafts mirrored as write_decode_step mirrors them) equals
    the f32 verify on rows that quantise losslessly (absmax 127, small integers)."""
    rng = np.random.default_rng(12)

    def rows(shape):
        x = rng.integers(-3, 4, size=shape).astype(f32)
        x[..., 0] = 127.0
        return x

    rk, rv, gk, gv, cur = _rswa_state(16)
    rk[:, :6], rv[:, :6] = rows((H, 6, HD)), rows((H, 6, HD))
    for _ in range(126):
        oracle.rswa_write(gk, gv, rows((H, HD)), rows((H, HD)), True, cur)
    dq, dk, dv = rows((4, H, HD)), rows((4, H, HD)), rows((4, H, HD))
    args = (dq, dk, dv, rk, rv, 6, gk, gv, cur, f32(1e-3))
    assert np.allclose(oracle.rswa_verify(*args, int8=True), oracle.rswa_verify(*args), rtol=1e-12, atol=1e-12)
