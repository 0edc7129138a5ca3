// kvd_split_h16.cuh -- the q8_2f tensor-core decode for groups of 9..16 query
// heads (GQA fan-out up to 16), in the register layout where the heads are
// the MMA M dimension.
//
// Same work split, TMA ring, partial slots and precision scheme as the warp
// kernel in kvd_split_mma.cuh; only the fragment layout differs.  With 16
// heads the m16 rows of an MMA are exactly the group's heads, so:
//   scores  S^T[h][row] = 2^-E_h sum_g ks[row][g] (t1_h + t2_h)_g . K_g[row]
//           with A = the query terms (registers, built once per unit),
//           B = K codes straight from ldmatrix of the K tile, N = four n8
//           tiles of rows; the two query terms chain as K steps into one f32
//           accumulator per 32-channel group, scaled by ks[row][g] after.
//   softmax lane (gl4, t4) holds heads gl4 and gl4 + 8 for rows 2*t4, 2*t4+1
//           of every n8 tile: the row maximum needs two shuffles per head.
//   weights the f16 terms of w = 2^(S - max) * vs[row] * 2^Ew are packed
//           directly into the A fragments of the value MMA (the score
//           accumulator layout of two n8 tiles is the A layout of one k16
//           step), so they never leave registers.
//   values  out[h][ch] = sum_row P[h][row] V[row][ch]: B = V codes from
//           ldmatrix.trans (even and odd channels of a 16-channel chunk as two
//           n8 tiles), fresh f32 accumulators per tile folded into the
//           running sum with one IEEE FMA per element.
#pragma once

#include "kvd_split_mma.cuh"

namespace kvd {

struct H16Cfg {
    static constexpr int BAR_OFF = kStages * kStageBytes;
    static constexpr int SMEM = BAR_OFF + kStages * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // room to align the base to 1024
};

// OPT: the call has a window or a softcap; IMP: the call accumulates imp
// (per-row scores are stored).  Both are compiled out of the common path.
template <bool OPT, bool IMP>
__global__ void __launch_bounds__(32, 8) split_h16_kernel(WarpArgs wa, LayerSrc src,
                                                            const __grid_constant__ MmaMaps maps) {
    using C = H16Cfg;
    extern __shared__ __align__(128) char smem_raw[];
    const SplitArgs &a = wa.a;
    const int lane = threadIdx.x;
    const int gl4 = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::BAR_OFF);
    const int64_t T = wa.T, G = wa.G, c = blockIdx.x;
    const int64_t x_begin = c * T / G, x_end = (c + 1) * T / G;
    // launched as a dependent of the kernel before (the append of a decode
    // step): wait for it, then let the run merge be scheduled
    pdl_wait();
    pdl_trigger();
    if (x_begin >= x_end) return;

    TileCursor cur;
    if (!cursor_locate(cur, x_begin, src, wa.n_seq, a.window, a.K, lane, a.err)) return;
    TileCursor prod = cur;
    if (cur.tl % kBlockTiles == 0) {
        // the slot just below this worker's first run belongs to no run
        const int64_t gap = cur.bq + int64_t(cur.gl) * blocks_of(cur.Tb) + cur.tl / kBlockTiles + c - 1;
        if (gap >= 0 && lane < a.hpk) {
            a.pm[gap * a.hpk + lane] = -INFINITY;
            a.pl[gap * a.hpk + lane] = 0.0f;
        }
    }
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    int64_t issued = 0;
    bool prod_ok = true;
    {
        const int64_t first = x_end - x_begin < kStages ? x_end - x_begin : int64_t(kStages);
        for (int64_t i = 0; i < first && prod_ok; ++i) {
            if (lane == 0) issue_tile(prod, &maps.kq, &maps.vq, src, sm + (i % kStages) * kStageBytes,
                                      &bar[i % kStages]);
            ++issued;
            if (x_begin + issued < x_end) prod_ok = cursor_next(prod, src, wa.n_seq, a.window, a.K, a.err);
        }
    }

    // K tile (ldmatrix, B of the scores): matrix mi covers rows nt*8 .. +7 of
    // chunk 4*half + mi, row rr; 128-byte swizzle by the row's low bits (= rr).
    // V tile (ldmatrix.trans, B of the values): row 8*mi + rr of chunk cc.
    const uint32_t kv_row = uint32_t(rr) * 128;
    const uint32_t v_lane = uint32_t(8 * mi + rr) * 128;
    const int ha = gl4, hb = gl4 + 8;  // this lane's heads

    uint32_t qa[8][2][4];  // query A fragments [chunk][term][reg]
    float qexp_a = 1.0f, qexp_b = 1.0f;
    int q_b = -1, q_gl = -1;

    int64_t x = x_begin, i = 0;
    bool ok = true;
    while (x < x_end) {
        int64_t run_len = x_end - x;
        if (run_len > cur.Tb - cur.tl) run_len = cur.Tb - cur.tl;
        if (run_len > kBlockTiles - cur.tl % kBlockTiles) run_len = kBlockTiles - cur.tl % kBlockTiles;
        const int64_t slot = cur.bq + int64_t(cur.gl) * blocks_of(cur.Tb) + cur.tl / kBlockTiles + c;
        const int64_t unit = int64_t(cur.b) * src.n_live + cur.gl;
        const bool unit_end = cur.tl + run_len == cur.Tb;
        if (cur.tl == 0 && lane == 0) wa.unit_slots[2 * unit] = slot;
        if (cur.b != q_b || cur.gl != q_gl) {
            // q * kcol * scale * log2e * 2^E_h = t1 + t2 (f16) for heads ha and
            // hb at channels 16*chunk + 4*t4 .. + 3: A rows gl4 (ha), gl4 + 8
            // (hb), k indices 2*t4, 2*t4+1 <- channels 4*t4, 4*t4+1 and
            // 2*t4+8, 2*t4+9 <- channels 4*t4+2, 4*t4+3 (the order of B).
            q_b = cur.b;
            q_gl = cur.gl;
            const int g = src.live[cur.gl];
            // M row e: query head e of the group, or for a verify of K drafts
            // draft e / hg, head e % hg ([n_seq][K][n_q][128])
            const int hg = a.K > 1 ? a.hg : a.hpk;
            const float *qg = a.q + (int64_t(cur.b) * a.K * a.n_q + int64_t(g) * hg) * 128;
            const float *qa_row = qg + (int64_t(ha / hg) * a.n_q + ha % hg) * 128;
            const float *qb_row = qg + (int64_t(hb / hg) * a.n_q + hb % hg) * 128;
            const float *kc = src.kcol + (int64_t(cur.b) * src.n_live + cur.gl) * 128;
            // two passes over the (cached) query rows: the heads' maxima
            // first, then the scaled terms, so no copy of q stays live
            auto xq = [&](int ch, float (&xa)[4], float (&xb)[4]) {
                const int d = 16 * ch + 4 * t4;
                const float4 kv = *reinterpret_cast<const float4 *>(kc + d);
                float4 qv = make_float4(0.0f, 0.0f, 0.0f, 0.0f), qw = qv;
                if (ha < a.hpk) qv = *reinterpret_cast<const float4 *>(qa_row + d);
                if (hb < a.hpk) qw = *reinterpret_cast<const float4 *>(qb_row + d);
                xa[0] = qv.x * kv.x * a.qscale;
                xa[1] = qv.y * kv.y * a.qscale;
                xa[2] = qv.z * kv.z * a.qscale;
                xa[3] = qv.w * kv.w * a.qscale;
                xb[0] = qw.x * kv.x * a.qscale;
                xb[1] = qw.y * kv.y * a.qscale;
                xb[2] = qw.z * kv.z * a.qscale;
                xb[3] = qw.w * kv.w * a.qscale;
            };
            float mxa = 0.0f, mxb = 0.0f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float xa[4], xb[4];
                xq(ch, xa, xb);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    mxa = fmaxf(mxa, fabsf(xa[j]));
                    mxb = fmaxf(mxb, fabsf(xb[j]));
                }
            }
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            const int Ea = mxa > 0.0f ? min(14 - exponent_of(mxa), 100) : 0;
            const int Eb = mxb > 0.0f ? min(14 - exponent_of(mxb), 100) : 0;
            const float sa = pow2i(Ea), sb = pow2i(Eb);
            qexp_a = pow2i(-Ea);
            qexp_b = pow2i(-Eb);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float xa[4], xb[4];
                xq(ch, xa, xb);
                float ah[4], al[4], bh[4], bl[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ah[j] = xa[j] * sa;
                    al[j] = ah[j] - __half2float(__float2half_rn(ah[j]));
                    bh[j] = xb[j] * sb;
                    bl[j] = bh[j] - __half2float(__float2half_rn(bh[j]));
                }
                qa[ch][0][0] = pack_half2(ah[0], ah[1]);
                qa[ch][0][1] = pack_half2(bh[0], bh[1]);
                qa[ch][0][2] = pack_half2(ah[2], ah[3]);
                qa[ch][0][3] = pack_half2(bh[2], bh[3]);
                qa[ch][1][0] = pack_half2(al[0], al[1]);
                qa[ch][1][1] = pack_half2(bl[0], bl[1]);
                qa[ch][1][2] = pack_half2(al[2], al[3]);
                qa[ch][1][3] = pack_half2(bl[2], bl[3]);
            }
        }
        float ma = -INFINITY, mb = -INFINITY, la = 0.0f, lb = 0.0f;
        float acc[8][2][4];  // [chunk][even/odd channels][frag]
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[cc][e][j] = 0.0f;
        int ew_prev = 0;

        for (int64_t k = 0; k < run_len; ++k, ++i, ++x) {
            const int stg = int(i % kStages);
            char *st = sm + stg * kStageBytes;
            if (__any_sync(0xffffffffu, !mbar_wait_bounded(&bar[stg], uint32_t(i / kStages) & 1u))) {
                ok = false;
                break;
            }
            const int row0 = cur.f0 + cur.tl * kWR;  // unit row of the tile's row 0
            const int n_valid = min(kWR, cur.Lb - row0);
            const int r_lo = cur.lo - row0;  // rows before it are outside the window
            const uint32_t kbase = smem_addr(st + kStK);
            const float *ks_s = reinterpret_cast<const float *>(st + kStKs);
            const float *vs_s = reinterpret_cast<const float *>(st + kStVs);

            // ------------------------------------------------ scores
            // sreg[nt][j]: j = 0, 1 -> head ha, rows nt*8 + 2*t4 + {0, 1};
            //              j = 2, 3 -> head hb, same rows
            float sreg[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int r0 = nt * 8 + 2 * t4;
                const float4 k0 = *reinterpret_cast<const float4 *>(&ks_s[r0 * 4]);
                const float4 k1 = *reinterpret_cast<const float4 *>(&ks_s[(r0 + 1) * 4]);
                const float ks0[4] = {k0.x, k0.y, k0.z, k0.w};
                const float ks1[4] = {k1.x, k1.y, k1.z, k1.w};
                float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                const uint32_t rowaddr = kbase + uint32_t(nt * 8) * 128 + kv_row;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t u[4];  // chunk 4*half + j, row nt*8 + gl4, channels 4*t4 .. + 3
                    ldsm_x4(rowaddr + (uint32_t((4 * half + mi) ^ rr) << 4), u);
                    // groups 2*half and 2*half + 1: two independent chains, interleaved
                    uint32_t bk[2][2][2];  // [gg][ks][b0/b1]
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t w = u[j] ^ 0x80808080u;
                        bk[j >> 1][j & 1][0] = codes_f16x2<0x4140>(w);
                        bk[j >> 1][j & 1][1] = codes_f16x2<0x4342>(w);
                    }
                    float dg[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                        for (int tm = 0; tm < 2; ++tm)
#pragma unroll
                            for (int gg = 0; gg < 2; ++gg) {
                                const int ch = 4 * half + 2 * gg + ks;
                                mma_f16(dg[gg], qa[ch][tm][0], qa[ch][tm][1], qa[ch][tm][2], qa[ch][tm][3],
                                        bk[gg][ks][0], bk[gg][ks][1]);
                            }
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg) {
                        const int g = 2 * half + gg;
                        sacc[0] = fmaf(ks0[g], dg[gg][0], sacc[0]);
                        sacc[1] = fmaf(ks1[g], dg[gg][1], sacc[1]);
                        sacc[2] = fmaf(ks0[g], dg[gg][2], sacc[2]);
                        sacc[3] = fmaf(ks1[g], dg[gg][3], sacc[3]);
                    }
                }
                sreg[nt][0] = sacc[0] * qexp_a;
                sreg[nt][1] = sacc[1] * qexp_a;
                sreg[nt][2] = sacc[2] * qexp_b;
                sreg[nt][3] = sacc[3] * qexp_b;
                if (OPT && a.softcap2 > 0.0f) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) sreg[nt][j] = softcap_log2(sreg[nt][j], a.softcap2);
                }
            }
            // rows outside [r_lo, n_valid) (a partial last tile, or rows before
            // the window in the first one) drop out; full tiles skip the masks.
            // A verify bounds each M row by its own query's limit and window:
            // rows [lo_a, hi_a) for ha, [lo_b, hi_b) for hb (tile rows).
            bool full = (!OPT || r_lo <= 0) && n_valid == kWR;
            int lo_a = r_lo, hi_a = n_valid, lo_b = r_lo, hi_b = n_valid;
            if (OPT && a.K > 1) {
                const int hg = a.hg;
                const int upto_a = cur.Lb - (a.K - 1 - ha / hg), upto_b = cur.Lb - (a.K - 1 - hb / hg);
                lo_a = int(first_visible(upto_a, a.window)) - row0;
                lo_b = int(first_visible(upto_b, a.window)) - row0;
                hi_a = min(upto_a - row0, n_valid);
                hi_b = min(upto_b - row0, n_valid);
                full = full && __all_sync(0xffffffffu, lo_a <= 0 && lo_b <= 0 && hi_a >= kWR && hi_b >= kWR);
            }
            if (!full) {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int r0 = nt * 8 + 2 * t4;
                    if (!(r0 >= lo_a && r0 < hi_a)) sreg[nt][0] = -INFINITY;
                    if (!(r0 + 1 >= lo_a && r0 + 1 < hi_a)) sreg[nt][1] = -INFINITY;
                    if (!(r0 >= lo_b && r0 < hi_b)) sreg[nt][2] = -INFINITY;
                    if (!(r0 + 1 >= lo_b && r0 + 1 < hi_b)) sreg[nt][3] = -INFINITY;
                }
            }
            if (IMP) {
                // per-row log2 scores for the imp pass: [hpk][cap] per unit
                float *sp = a.scores + cur.rbase * a.hpk + row0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = hh ? hb : ha;
                    if (h < a.hpk) {
                        float *sh = sp + int64_t(h) * cur.cap;
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
                            const int r0 = nt * 8 + 2 * t4;
                            if (r0 >= r_lo && r0 + 1 < n_valid) {
                                *reinterpret_cast<float2 *>(sh + r0) =
                                    make_float2(sreg[nt][2 * hh], sreg[nt][2 * hh + 1]);
                            } else {
                                if (r0 >= r_lo && r0 < n_valid) sh[r0] = sreg[nt][2 * hh];
                                if (r0 + 1 >= r_lo && r0 + 1 < n_valid) sh[r0 + 1] = sreg[nt][2 * hh + 1];
                            }
                        }
                    }
                }
            }

            // ------------------------------------------------ softmax
            float vsr[4][2];
            float vmax = 0.0f, ta = -INFINITY, tb = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int r0 = nt * 8 + 2 * t4;
                const float2 vv = *reinterpret_cast<const float2 *>(&vs_s[r0]);
                vsr[nt][0] = vv.x;
                vsr[nt][1] = vv.y;
                if (!full) {
                    if (!(r0 >= r_lo && r0 < n_valid)) vsr[nt][0] = 0.0f;
                    if (!(r0 + 1 >= r_lo && r0 + 1 < n_valid)) vsr[nt][1] = 0.0f;
                }
                vmax = fmaxf(vmax, fmaxf(vsr[nt][0], vsr[nt][1]));
                ta = fmaxf(ta, fmaxf(sreg[nt][0], sreg[nt][1]));
                tb = fmaxf(tb, fmaxf(sreg[nt][2], sreg[nt][3]));
            }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
                ta = fmaxf(ta, __shfl_xor_sync(0xffffffffu, ta, off));
                tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, off));
            }
            // (the t4 lanes of any gl4 cover all 32 rows: every lane has the same vmax)
            const int ew = vmax > 0.0f ? min(14 - exponent_of(vmax), 100) : 0;
            const float wsc = pow2i(ew);
            // the change of Ew is an exact power of two (the approximate exp2
            // is not exact even at integers, and these factors compound over a run)
            const float dsc = pow2_wide(ew - ew_prev);
            ew_prev = ew;
            const float mna = fmaxf(ma, ta), mnb = fmaxf(mb, tb);
            // exactly 1 while the maximum holds; 0 before the first tile (m = -inf)
            const float ala = mna == ma ? 1.0f : fast_exp2(ma - mna);
            const float alb = mnb == mb ? 1.0f : fast_exp2(mb - mnb);
            const float fa_a = ala * dsc, fa_b = alb * dsc;
            la *= ala;
            lb *= alb;
            ma = mna;
            mb = mnb;
            // weights -> f16 terms in the A layout of the value MMA: k16 step
            // kk covers score tiles 2kk (a0, a1) and 2kk + 1 (a2, a3)
            // a verify row that has seen no visible row yet keeps weight 0
            const float mza = OPT && ma == -INFINITY ? 0.0f : ma, mzb = OPT && mb == -INFINITY ? 0.0f : mb;
            uint32_t pa[2][2][4];  // [kk][term][reg]
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const float e0 = fast_exp2(sreg[nt][0] - mza), e1 = fast_exp2(sreg[nt][1] - mza);
                const float e2 = fast_exp2(sreg[nt][2] - mzb), e3 = fast_exp2(sreg[nt][3] - mzb);
                la += e0 + e1;
                lb += e2 + e3;
                const float v0 = vsr[nt][0] * wsc, v1 = vsr[nt][1] * wsc;
                const float w0 = e0 * v0, w1 = e1 * v1, w2 = e2 * v0, w3 = e3 * v1;
                const uint32_t ta1 = pack_half2(w0, w1), tb1 = pack_half2(w2, w3);
                const float2 ba = __half22float2(*reinterpret_cast<const __half2 *>(&ta1));
                const float2 bb = __half22float2(*reinterpret_cast<const __half2 *>(&tb1));
                const int kk = nt >> 1, hi = (nt & 1) * 2;
                pa[kk][0][hi] = ta1;
                pa[kk][0][hi + 1] = tb1;
                pa[kk][1][hi] = pack_half2(w0 - ba.x, w1 - ba.y);
                pa[kk][1][hi + 1] = pack_half2(w2 - bb.x, w3 - bb.y);
            }

            // ------------------------------------------------ values
            const uint32_t vaddr = smem_addr(st + kStV) + v_lane;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t xv[4];  // rows 0-7, 8-15, 16-23, 24-31 of chunk cc
                ldsm_x4_t(vaddr + (uint32_t(cc ^ rr) << 4), xv);
                uint32_t bv[2][2][2];  // [even/odd][kk][b0/b1]
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t w = xv[2 * kk + j] ^ 0x80808080u;
                        bv[0][kk][j] = codes_f16x2<0x4240>(w);
                        bv[1][kk][j] = codes_f16x2<0x4341>(w);
                    }
                // even and odd channels: two independent chains, interleaved
                float d[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int tm = 0; tm < 2; ++tm)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            mma_f16(d[e], pa[kk][tm][0], pa[kk][tm][1], pa[kk][tm][2], pa[kk][tm][3], bv[e][kk][0],
                                    bv[e][kk][1]);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    acc[cc][e][0] = fmaf(acc[cc][e][0], fa_a, d[e][0]);
                    acc[cc][e][1] = fmaf(acc[cc][e][1], fa_a, d[e][1]);
                    acc[cc][e][2] = fmaf(acc[cc][e][2], fa_b, d[e][2]);
                    acc[cc][e][3] = fmaf(acc[cc][e][3], fa_b, d[e][3]);
                }
            }
            __syncwarp();  // every lane is done with this stage
            if (x_begin + issued < x_end && prod_ok) {
                if (lane == 0) {
                    fence_proxy_async();
                    issue_tile(prod, &maps.kq, &maps.vq, src, st, &bar[stg]);
                }
                ++issued;
                if (x_begin + issued < x_end) prod_ok = cursor_next(prod, src, wa.n_seq, a.window, a.K, a.err);
            }
            if (x + 1 < x_end && !cursor_next(cur, src, wa.n_seq, a.window, a.K, a.err)) {
                ok = false;
                ++i;
                break;
            }
        }
        if (!ok) break;

        // ------------------------------------------------ run partial
        if (unit_end && lane == 0) wa.unit_slots[2 * unit + 1] = slot;
        const int64_t p0 = slot * a.hpk;
        const float unscale = pow2i(-ew_prev);
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            la += __shfl_xor_sync(0xffffffffu, la, off);
            lb += __shfl_xor_sync(0xffffffffu, lb, off);
        }
        // head ha: channels 16*cc + 4*t4 + {0,1,2,3} = (even d0, odd d0, even d1, odd d1)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int h = hh ? hb : ha;
            if (h < a.hpk) {
                if (t4 == 0) {
                    a.pm[p0 + h] = hh ? mb : ma;
                    a.pl[p0 + h] = hh ? lb : la;
                }
                float *dst = a.pacc + (p0 + h) * 128 + 4 * t4;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<float4 *>(dst + 16 * cc) =
                        make_float4(acc[cc][0][2 * hh] * unscale, acc[cc][1][2 * hh] * unscale,
                                    acc[cc][0][2 * hh + 1] * unscale, acc[cc][1][2 * hh + 1] * unscale);
            }
        }
    }

    if (!ok && lane == 0) {
        set_error(a.err, kErrTimeout);
        for (int64_t j = i; j < issued; ++j)
            (void)mbar_wait_bounded(&bar[j % kStages], uint32_t(j / kStages) & 1u, 100000000ull);
    }
}

inline cudaError_t launch_split_h16(const WarpArgs &wa, const LayerSrc &s, const MmaMaps &maps,
                                    cudaStream_t st) {
    const bool opt = wa.a.window > 0 || wa.a.softcap2 > 0.0f || wa.a.K > 1, imp = wa.a.scores != nullptr;
    auto kern = opt ? (imp ? split_h16_kernel<true, true> : split_h16_kernel<true, false>)
                    : (imp ? split_h16_kernel<false, true> : split_h16_kernel<false, false>);
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), H16Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(unsigned(wa.G)), dim3(32), H16Cfg::SMEM_ALLOC, st, wa, s, maps);
}

inline int64_t split_h16_workers() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    auto kern = split_h16_kernel<false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, H16Cfg::SMEM_ALLOC) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 32, H16Cfg::SMEM_ALLOC) != cudaSuccess)
        return 0;
    return int64_t(sms) * occ;
}

}  // namespace kvd
