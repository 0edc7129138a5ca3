// kvd_split_mma.cuh -- split-KV decode over the q8_2f cache (int8 K and V,
// head_dim 128) on the tensor cores (warp-level mma.sync, f16 in, f32 out).
//
// Why: with int8 rows the CUDA-core kernel spends ~84 instructions per cached
// row (int8->f32 conversions, hpk x 128 FMAs per pass, warp reductions) and is
// issue-bound far below the HBM roofline at GQA fan-out 4..16.  Here both
// contractions run as f16 MMAs with f32 accumulation; the CUDA cores only turn
// each int8 code into an exact f16 once (a byte splice and one HSUB2 per pair),
// shared by every query head of the group.  (The legacy int8 mma.sync path is
// far slower than f16 on this GPU, so the codes go through f16.)
//
// Per tile of 128 cached rows:
//   scores  warps split the rows (32 each, two m16 blocks):
//           S[row][h] = 2^-E_h * sum_g ks[row][g] * K_g . (t1_h + t2_h)_g
//           K codes are exact in f16; q * kcol * scale * log2(e) * 2^E_h is
//           split into two f16 terms t1 + t2 (22 significant bits, E_h puts the
//           head's largest term near 2^14); m16n8k16 MMAs accumulate each
//           32-channel group in f32 so its scale ks[row][g] applies after.  The
//           channel order inside a k16 step is permuted identically in A and B
//           so a lane's four consecutive codes feed its fragment directly.
//           The per-warp maximum of each head is reduced in registers.
//   softmax online over tiles in the log2 domain (running max per head; every
//           thread derives the same maxima from the per-warp values).
//   weights w = 2^(S - max) * vs[row] * 2^Ew (Ew puts the tile's largest V
//           scale near 2^14) split into two f16 terms, written to shared
//           memory as the A operand [term][k16 step][head][position].
//   values  warps split the 128 channels (32 each); V codes become the f16 B
//           operand straight from ldmatrix.trans; m16n8k16 MMAs with M = the
//           group's heads accumulate into f32 registers across all tiles (the
//           accumulator is rescaled by the softmax correction and the change
//           of Ew between tiles).
// K and V code tiles arrive by TMA tensor copies with the 128-byte swizzle
// (conflict-free ldmatrix); scales by 1-D bulk copies; a ring of kMmaSlots
// slots alternates K and V segments.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "kvd_decode_kernels.cuh"

namespace kvd {

constexpr int kMmaTR = 128;        // rows per tile
constexpr int kMmaSlots = 3;       // ring slots (K, V alternate)
constexpr int kMmaTile = 16384;    // bytes of one 128 x 128 code tile
constexpr int kMmaKsOff = 16384;   // K scales within a K segment
constexpr int kMmaVsOff = 18432;   // V scales within a K segment
constexpr int kMmaSlot = 19456;    // bytes per slot (multiple of 1024)
constexpr int kMmaAw = 2 * 8 * 16 * 32;  // weights [term][k16 step][16 heads][16 f16]

template <int HPK>
struct MmaCfg {
    static constexpr int HPKP = HPK < 4 ? 4 : HPK;          // heads padded for the layouts
    static constexpr int NT = HPKP / 8 > 0 ? HPKP / 8 : 1;  // score n8 tiles
    static constexpr int S_OFF = kMmaSlots * kMmaSlot;       // q staging [HPKP][128] f32
    static constexpr int AW_OFF = S_OFF + HPKP * 128 * 4;
    static constexpr int MISC_OFF = AW_OFF + kMmaAw;
    // misc: bars[kMmaSlots], red[kWarps][HPKP], vred[kWarps]
    static constexpr int SMEM = MISC_OFF + kMmaSlots * 8 + kWarps * HPKP * 4 + kWarps * 4;
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // room to align the base to 1024
    static constexpr int MIN_CTAS = HPK >= 16 ? 2 : 3;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A(16x16 f16, row) * B(16x8 f16, col), f32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Exact f16 of two int8 codes picked from a word: bias to unsigned, splice each
// byte under the f16 exponent of 1024 (giving 1024 + code + 128), subtract 1152.
// sel picks the two bytes (0x4140: bytes 0,1; 0x4342: 2,3; 0x4240: 0,2; 0x4341: 1,3).
template <uint32_t SEL>
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t biased) {
    const uint32_t a = __byte_perm(biased, 0x64646464u, SEL);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 x = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    return *reinterpret_cast<const uint32_t *>(&x);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// exponent e with x in [2^(e-1), 2^e), x > 0
__device__ __forceinline__ int exponent_of(float x) {
    int e;
    frexpf(x, &e);
    return e;
}

struct MmaMaps {
    CUtensorMap kq, vq;
};

template <int HPK>
__device__ __forceinline__ void mma_issue(const ChunkInfo &ci, const CUtensorMap *kmap,
                                          const CUtensorMap *vmap, int64_t row_base, char *sm,
                                          uint64_t *bar, int j) {
    const int slot = j % kMmaSlots;
    const int t = j >> 1;
    const int row0 = t * kMmaTR;
    const int nt = min(kMmaTR, ci.n - row0);
    const int rows = (nt + kRowAlign - 1) / kRowAlign * kRowAlign;
    char *dst = sm + slot * kMmaSlot;
    if ((j & 1) == 0) {
        mbar_arrive_expect_tx(&bar[slot], uint32_t(kMmaTile + rows * 16 + rows * 4));
        tma_load_2d(dst, kmap, 0, int(row_base + row0), &bar[slot]);
        bulk_g2s(dst + kMmaKsOff, ci.ks + int64_t(row0) * 16, uint32_t(rows) * 16, &bar[slot]);
        bulk_g2s(dst + kMmaVsOff, ci.vs + int64_t(row0) * 4, uint32_t(rows) * 4, &bar[slot]);
    } else {
        mbar_arrive_expect_tx(&bar[slot], uint32_t(kMmaTile));
        tma_load_2d(dst, vmap, 0, int(row_base + row0), &bar[slot]);
    }
}

// Byte offset of weight (term, position p, head h) in the A operand area: 16 x
// 16 f16 blocks per (term, k16 step), the two 8-position halves of a head's
// row swapped on heads 4..7 and 12..15 so ldmatrix rows hit distinct banks.
__device__ __forceinline__ int aw_offset(int term, int p, int h) {
    const int ks = p >> 4, k = p & 15;
    return ((term * 8 + ks) * 16 + h) * 32 + (((k >> 3) ^ ((h >> 2) & 1)) << 4) + (k & 7) * 2;
}

// One CTA: one chunk of ci.n rows starting at storage row `row_base` of one
// (sequence, live group).  Writes the partial (max, sum, acc) of each head.
template <int HPK>
__device__ void split_mma_body(const ChunkInfo &ci, int64_t row_base, const SplitArgs &a,
                               const CUtensorMap *kmap, const CUtensorMap *vmap, char *smem_raw) {
    using C = MmaCfg<HPK>;
    constexpr int HPKP = C::HPKP, NT = C::NT;
    // align to 1024 by offsetting the shared array itself, so every derived
    // pointer stays a known shared-memory pointer (plain LDS/STS)
    char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gl4 = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix index, row in matrix
    char *Aw = sm + C::AW_OFF;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::MISC_OFF);
    float *red = reinterpret_cast<float *>(bar + kMmaSlots);
    float *vred = red + kWarps * HPKP;

    const int n = ci.n;
    const int ntiles = (n + kMmaTR - 1) / kMmaTR;
    const int nseg = 2 * ntiles;

    if (tid == 0) {
        for (int s = 0; s < kMmaSlots; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int j = 0; j < min(kMmaSlots, nseg); ++j) mma_issue<HPK>(ci, kmap, vmap, row_base, sm, bar, j);

    // ---- query terms: q * kcol * scale * log2e * 2^E_h = t1 + t2 (f16),
    //      staged through the staging area
    float *qf = reinterpret_cast<float *>(sm + C::S_OFF);
    for (int i = tid; i < HPKP * 128; i += kThreads) {
        const int h = i >> 7, d = i & 127;
        qf[i] = h < a.hpk ? ci.q[h * 128 + d] * ci.kcol[d] * a.qscale : 0.0f;
    }
    __syncthreads();
    if (tid < HPKP) {
        float mx = 0.0f;
        for (int d = 0; d < 128; ++d) mx = fmaxf(mx, fabsf(qf[tid * 128 + d]));
        red[tid] = mx > 0.0f ? float(14 - exponent_of(mx)) : 0.0f;
    }
    __syncthreads();
    uint32_t bq[4][2][NT][2][2];  // [group][k16 step][n-tile][term][reg]
    float qexp[NT][2];            // 2^-E of the heads in this lane's score columns
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = nt * 8 + 2 * t4 + c;
            qexp[nt][c] = h < HPKP ? exp2f(-red[h]) : 0.0f;
        }
        const int hb = nt * 8 + gl4;  // the B column this lane feeds
        const float sc = hb < HPKP ? exp2f(red[hb]) : 0.0f;
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int c0 = 32 * g + 16 * ks + 4 * t4;
                float x[4], r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[i] = hb < HPKP ? qf[hb * 128 + c0 + i] * sc : 0.0f;
                    r[i] = x[i] - __half2float(__float2half_rn(x[i]));
                }
                bq[g][ks][nt][0][0] = pack_half2(x[0], x[1]);
                bq[g][ks][nt][0][1] = pack_half2(x[2], x[3]);
                bq[g][ks][nt][1][0] = pack_half2(r[0], r[1]);
                bq[g][ks][nt][1][1] = pack_half2(r[2], r[3]);
            }
    }
    __syncthreads();  // staging read before anything reuses it

    // Lane-constant shared-memory offsets.  K tile (ldmatrix, scores): row
    // warp*32 + mb*16 + rr + 8*(mi&1), 16-byte chunk 2g + (mi>>1), swizzled by
    // the row's low 3 bits (= rr).  V tile (ldmatrix.trans): position 16ks +
    // 8*(mi&1) + rr, chunk 2*warp + (mi>>1).  Weights: head row rr + 8*(mi&1),
    // half mi>>1, swapped on heads 4..7 / 12..15.
    const uint32_t k_lane = uint32_t(warp * 32 + rr + 8 * (mi & 1)) * 128;
    uint32_t k_chunk[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) k_chunk[g] = uint32_t(((2 * g + (mi >> 1)) ^ rr) << 4);
    const uint32_t v_lane = uint32_t(8 * (mi & 1) + rr) * 128 + uint32_t(((2 * warp + (mi >> 1)) ^ rr) << 4);
    const int am = rr + 8 * (mi & 1);
    const uint32_t aw_lane = uint32_t(am * 32 + (((mi >> 1) ^ ((am >> 2) & 1)) << 4));
    const uint32_t aw_base = smem_addr(Aw) + aw_lane;
    // where this lane writes the weight terms of its score values: head h =
    // nt*8 + 2*t4 + c, position warp*32 + mb*16 + gl4 + 8*rw (k16 step warp*2 + mb)
    int wofs[2][NT][2][2];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int rw = 0; rw < 2; ++rw) {
                    const int h = nt * 8 + 2 * t4 + c;
                    wofs[mb][nt][c][rw] =
                        ((warp * 2 + mb) * 16 + h) * 32 + ((rw ^ ((h >> 2) & 1)) << 4) + gl4 * 2;
                }

    // running state: maxima and sums of this lane's score-column heads
    // (nt*8 + 2*t4 + c) and maxima of its P.V heads (gl4, gl4 + 8); every lane
    // derives identical maxima from the per-warp values in red
    float mcol[NT][2], lcol[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mcol[nt][0] = mcol[nt][1] = -INFINITY, lcol[nt][0] = lcol[nt][1] = 0.0f;
    float m_a = -INFINITY, m_b = -INFINITY;
    int ew_prev = 0;
    float acc[4][4];  // [n-tile: block 0 even, 0 odd, 1 even, 1 odd][frag]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = 0.0f;
    bool ok = true;

    for (int t = 0; t < ntiles; ++t) {
        const int row0 = t * kMmaTR;
        const int nt_rows = min(kMmaTR, n - row0);
        int j = 2 * t;
        int slot = j % kMmaSlots;
        if (__syncthreads_or(!mbar_wait_bounded(&bar[slot], (j / kMmaSlots) & 1))) {
            ok = false;
            break;
        }
        // the previous tile's V slot is drained (every thread passed the barrier)
        if (tid == 0 && t > 0 && j - 1 + kMmaSlots < nseg)
            mma_issue<HPK>(ci, kmap, vmap, row_base, sm, bar, j - 1 + kMmaSlots);
        const char *kseg = sm + slot * kMmaSlot;
        const uint32_t kaddr = smem_addr(kseg) + k_lane;
        const float *ks_s = reinterpret_cast<const float *>(kseg + kMmaKsOff);
        const float *vs_s = reinterpret_cast<const float *>(kseg + kMmaVsOff);
        // ------------------------------------------------ scores (f16 MMA)
        float sreg[2][NT][2][2];  // [m block][n-tile][column][row gl4 / gl4 + 8]
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
            const int r0 = warp * 32 + mb * 16;
            float sacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.0f;
            const float4 ksA = *reinterpret_cast<const float4 *>(&ks_s[(r0 + gl4) * 4]);
            const float4 ksB = *reinterpret_cast<const float4 *>(&ks_s[(r0 + gl4 + 8) * 4]);
            const float kA[4] = {ksA.x, ksA.y, ksA.z, ksA.w};
            const float kB[4] = {ksB.x, ksB.y, ksB.z, ksB.w};
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                uint32_t w[4];
                ldsm_x4(kaddr + mb * 2048 + k_chunk[g], w);
                // row gl4 / gl4 + 8, channels 4t..4t+3 of k16 step 0 and 1
                const uint32_t u0 = w[0] ^ 0x80808080u, u1 = w[1] ^ 0x80808080u;
                const uint32_t u2 = w[2] ^ 0x80808080u, u3 = w[3] ^ 0x80808080u;
                const uint32_t a00 = codes_f16x2<0x4140>(u0), a02 = codes_f16x2<0x4342>(u0);
                const uint32_t a01 = codes_f16x2<0x4140>(u1), a03 = codes_f16x2<0x4342>(u1);
                const uint32_t a10 = codes_f16x2<0x4140>(u2), a12 = codes_f16x2<0x4342>(u2);
                const uint32_t a11 = codes_f16x2<0x4140>(u3), a13 = codes_f16x2<0x4342>(u3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float dg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int tm = 0; tm < 2; ++tm) {
                        mma_f16(dg, a00, a01, a02, a03, bq[g][0][nt][tm][0], bq[g][0][nt][tm][1]);
                        mma_f16(dg, a10, a11, a12, a13, bq[g][1][nt][tm][0], bq[g][1][nt][tm][1]);
                    }
                    sacc[nt][0] = fmaf(kA[g], dg[0], sacc[nt][0]);
                    sacc[nt][1] = fmaf(kA[g], dg[1], sacc[nt][1]);
                    sacc[nt][2] = fmaf(kB[g], dg[2], sacc[nt][2]);
                    sacc[nt][3] = fmaf(kB[g], dg[3], sacc[nt][3]);
                }
            }
            const int ra = r0 + gl4, rb = r0 + gl4 + 8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    sreg[mb][nt][c][0] = ra < nt_rows ? sacc[nt][c] * qexp[nt][c] : -INFINITY;
                    sreg[mb][nt][c][1] = rb < nt_rows ? sacc[nt][2 + c] * qexp[nt][c] : -INFINITY;
                }
            if (a.scores != nullptr) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int h = nt * 8 + 2 * t4 + c;
                        if (h < a.hpk) {
                            float *sp = a.scores + ci.score0 + h * ci.score_ld + row0;
                            if (ra < nt_rows) sp[ra] = sreg[mb][nt][c][0];
                            if (rb < nt_rows) sp[rb] = sreg[mb][nt][c][1];
                        }
                    }
            }
        }
        // per-warp maxima of every head and of the V row scales
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float m = fmaxf(fmaxf(sreg[0][nt][c][0], sreg[0][nt][c][1]),
                                fmaxf(sreg[1][nt][c][0], sreg[1][nt][c][1]));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                const int h = nt * 8 + 2 * t4 + c;
                if (gl4 == 0 && h < HPKP) red[warp * HPKP + h] = m;
            }
        {
            float v = tid < nt_rows ? vs_s[tid] : 0.0f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) vred[warp] = v;
        }
        __syncthreads();
        // -------------------------- new maxima (identical in every thread)
        float vmax = vred[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) vmax = fmaxf(vmax, vred[w]);
        const int ew = vmax > 0.0f ? 14 - exponent_of(vmax) : 0;
        const float wscale = exp2f(float(ew));
        // Heads past HPKP (padding lanes) read a clamped head: harmless, and
        // it keeps every lane on the same path.  Tile maxima are finite (each
        // tile has a valid row), so exp2(old - new) is 0 on the first tile.
        auto tile_max = [&](int h) {
            h = min(h, HPKP - 1);
            float m = red[h];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) m = fmaxf(m, red[w * HPKP + h]);
            return m;
        };
        const float mna = fmaxf(m_a, tile_max(gl4));
        const float al_a = exp2f(m_a - mna);
        m_a = mna;
        const float mnb = fmaxf(m_b, tile_max(gl4 + 8));
        const float al_b = exp2f(m_b - mnb);
        m_b = mnb;
        // ------------------- weights from the score registers -> f16 terms
        float vsw[2][2];  // V row scale * 2^ew of this lane's rows (0 past the tile)
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int rw = 0; rw < 2; ++rw) {
                const int p = warp * 32 + mb * 16 + gl4 + 8 * rw;
                vsw[mb][rw] = p < nt_rows ? vs_s[p] * wscale : 0.0f;
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                // padding columns (heads >= HPKP when HPKP is 4) compute like
                // the others and write weight rows the value pass never reads
                const int h = nt * 8 + 2 * t4 + c;
                const float mn = fmaxf(mcol[nt][c], tile_max(h));
                lcol[nt][c] *= exp2f(mcol[nt][c] - mn);
                mcol[nt][c] = mn;
                const float live = h < a.hpk ? 1.0f : 0.0f;
#pragma unroll
                for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                    for (int rw = 0; rw < 2; ++rw) {
                        // rows past the tile hold -inf scores: e = 0
                        const float e = live * exp2f(sreg[mb][nt][c][rw] - mn);
                        lcol[nt][c] += e;
                        const float w = e * vsw[mb][rw];
                        const __half t1 = __float2half_rn(w);
                        const __half t2 = __float2half_rn(w - __half2float(t1));
                        *reinterpret_cast<__half *>(Aw + wofs[mb][nt][c][rw]) = t1;
                        *reinterpret_cast<__half *>(Aw + 8 * 16 * 32 + wofs[mb][nt][c][rw]) = t2;
                    }
            }
        __syncthreads();  // weights visible; K slot drained
        if (tid == 0 && j + kMmaSlots < nseg) mma_issue<HPK>(ci, kmap, vmap, row_base, sm, bar, j + kMmaSlots);
        // ------------------------------------------------ P.V (f16 MMA)
        j = 2 * t + 1;
        slot = j % kMmaSlots;
        if (__syncthreads_or(!mbar_wait_bounded(&bar[slot], (j / kMmaSlots) & 1))) {
            ok = false;
            break;
        }
        // This tile's P.V goes into fresh MMA accumulators (16 chained MMAs
        // each); it is folded into the running sum with IEEE FMAs below, so the
        // tensor cores' accumulation rounding never compounds across tiles.
        float dacc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) dacc[i][c] = 0.0f;
        const uint32_t vaddr = smem_addr(sm + slot * kMmaSlot) + v_lane;
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            // V: matrices (positions +0..7, +8..15) x (channel chunks 2w, 2w + 1)
            uint32_t x[4];
            ldsm_x4_t(vaddr + ks * 2048, x);
            uint32_t b[4][2];  // [n-tile][reg]
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                const uint32_t lo = x[2 * blk] ^ 0x80808080u, hi = x[2 * blk + 1] ^ 0x80808080u;
                b[2 * blk][0] = codes_f16x2<0x4240>(lo);
                b[2 * blk][1] = codes_f16x2<0x4240>(hi);
                b[2 * blk + 1][0] = codes_f16x2<0x4341>(lo);
                b[2 * blk + 1][1] = codes_f16x2<0x4341>(hi);
            }
#pragma unroll
            for (int term = 0; term < 2; ++term) {
                uint32_t af[4];
                ldsm_x4(aw_base + (term * 8 + ks) * 512, af);
#pragma unroll
                for (int q = 0; q < 4; ++q) mma_f16(dacc[q], af[0], af[1], af[2], af[3], b[q][0], b[q][1]);
            }
        }
        {
            // acc holds sum * 2^ew: rescale by the softmax correction and the
            // change of weight exponent, then add this tile
            const float fa = al_a * exp2f(float(ew - ew_prev));
            const float fb = al_b * exp2f(float(ew - ew_prev));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[i][0] = fmaf(acc[i][0], fa, dacc[i][0]);
                acc[i][1] = fmaf(acc[i][1], fa, dacc[i][1]);
                acc[i][2] = fmaf(acc[i][2], fb, dacc[i][2]);
                acc[i][3] = fmaf(acc[i][3], fb, dacc[i][3]);
            }
            ew_prev = ew;
        }
    }

    if (!ok) {
        if (tid == 0) {
            set_error(a.err, kErrTimeout);
            for (int s = 0; s < kMmaSlots; ++s) (void)mbar_wait_bounded(&bar[s], 0, 100000000ull);
            for (int s = 0; s < kMmaSlots; ++s) (void)mbar_wait_bounded(&bar[s], 1, 100000000ull);
        }
        return;
    }

    // ------------------------------------------------------------ partials
    // sums: reduce each column head over the lanes sharing it, then the warps
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float l = lcol[nt][c];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            lcol[nt][c] = l;
        }
    __syncthreads();  // every warp is past its last read of red
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = nt * 8 + 2 * t4 + c;
            if (gl4 == 0 && h < HPKP) red[warp * HPKP + h] = lcol[nt][c];
        }
    __syncthreads();
    if (warp == 0 && gl4 == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int h = nt * 8 + 2 * t4 + c;
                if (h < a.hpk) {
                    float l = red[h];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) l += red[w * HPKP + h];
                    a.pm[ci.pidx0 + h] = mcol[nt][c];
                    a.pl[ci.pidx0 + h] = l;
                }
            }
    }
    // lane (gl4, t4) of warp w holds heads gl4 and gl4 + 8 at channels
    // 32w + 16 blk + 4 t4 + {0, 2} (even tile) and + {1, 3} (odd tile)
    const float unscale = exp2f(-float(ew_prev));
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = gl4 + 8 * hh;
        if (h < a.hpk) {
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                float *dst = a.pacc + (ci.pidx0 + h) * 128 + 32 * warp + 16 * blk + 4 * t4;
                const float *e = acc[2 * blk];
                const float *o = acc[2 * blk + 1];
                *reinterpret_cast<float4 *>(dst) =
                    make_float4(e[2 * hh] * unscale, o[2 * hh] * unscale, e[2 * hh + 1] * unscale,
                                o[2 * hh + 1] * unscale);
            }
        }
    }
}

template <int HPK>
__global__ void __launch_bounds__(kThreads, MmaCfg<HPK>::MIN_CTAS)
    split_mma_kernel(SplitArgs a, LayerSrc src, const __grid_constant__ MmaMaps maps) {
    extern __shared__ __align__(128) char smem[];
    const int b = blockIdx.z, gl = blockIdx.y, c = blockIdx.x;
    const int L = src.seq_len[b];
    const int64_t r0 = int64_t(c) * a.chunk;
    if (r0 >= L) return;
    const int64_t cap = src.cap[b];
    if (L > cap) {
        if (threadIdx.x == 0) set_error(a.err, kErrBounds);
        return;
    }
    const int64_t row = src.row_base[b] + int64_t(gl) * cap + r0;
    ChunkInfo ci;
    ci.k = nullptr;
    ci.v = nullptr;
    ci.ks = reinterpret_cast<const char *>(src.ks + row * 4);
    ci.vs = reinterpret_cast<const char *>(src.vs + row);
    ci.n = int(a.chunk < L - r0 ? int64_t(a.chunk) : L - r0);
    ci.pidx0 = ((int64_t(b) * a.n_grp + gl) * a.nc_max + c) * a.hpk;
    const int g = src.live[gl];
    ci.q = a.q + (int64_t(b) * a.n_q + int64_t(g) * a.hpk) * 128;
    ci.kcol = src.kcol + (int64_t(b) * src.n_live + gl) * 128;
    ci.score0 = (src.row_base[b] + int64_t(gl) * cap) * a.hpk + r0;
    ci.score_ld = cap;
    split_mma_body<HPK>(ci, row, a, &maps.kq, &maps.vq, smem);
}

template <int HPK>
cudaError_t launch_split_mma(const SplitArgs &a, const LayerSrc &s, const MmaMaps &maps, dim3 grid,
                             cudaStream_t st) {
    using C = MmaCfg<HPK>;
    auto kern = split_mma_kernel<HPK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM_ALLOC, st>>>(a, s, maps);
    return cudaGetLastError();
}

}  // namespace kvd
