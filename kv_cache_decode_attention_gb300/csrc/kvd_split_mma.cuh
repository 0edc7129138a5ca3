// kvd_split_mma.cuh -- split-KV decode over the q8_2f cache (int8 K and V,
// head_dim 128) on the tensor cores.
//
// Why: with int8 rows, the CUDA-core kernel spends ~84 instructions per
// cached row on int8->f32 conversions, hpk x 128 FMAs per pass and the warp
// reductions; at GQA fan-out 4..16 that is issue-bound far below the HBM
// roofline.  Here both contractions go through mma.sync, and the only
// per-element CUDA-core work left is a 4-instruction int8->f16 conversion of
// the K codes.
//
// Score (per tile of 128 rows, each warp 32 rows = two m16 blocks):
//   S[row][h] = 2^-E_h * sum_g ks[row][g] * (K_g f16) . (q_g t1 + q_g t2)
//   K codes are exact in f16; q * kcol * scale * log2(e) * 2^E_h is split
//   into two f16 terms t1 + t2 (22 significant bits; E_h puts each head's
//   largest term near 2^14); m16n8k16 MMAs accumulate in f32 per 32-channel
//   group so the group scale ks[row][g] applies after.  The channel order
//   inside a k16 step is permuted consistently in A and B so that one lane's
//   four consecutive int8 codes feed its fragment directly.
// Softmax: online over tiles, running max per head, in the log2 domain.
// Value (the same tile): w = 2^(S - max) * vs[row] is quantised to a 24-bit
//   unsigned fixed point relative to the tile's largest vs (exact byte digits
//   w = d0 + 256 d1 + 65536 d2, relative error <= 2^-24 of the largest
//   weight); m16n8k32 u8 x s8 MMAs with int32 accumulation give
//   sum_p d_j[h][p] V[p][c] exactly; the three digit sums are combined in
//   f32 once per tile and folded into the running accumulator.  Warps split
//   the 128 channels (32 each), so no cross-warp reduction is needed.
// Data movement: K and V code tiles arrive by TMA tensor copies with the
// 128-byte swizzle (conflict-free ldmatrix), scales by 1-D bulk copies, into
// a ring of kMmaSlots slots alternating K and V segments.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "kvd_decode_kernels.cuh"

namespace kvd {

constexpr int kMmaTR = 128;        // rows per tile
constexpr int kMmaSlots = 4;       // ring slots (K, V alternate)
constexpr int kMmaTile = 16384;    // bytes of one 128 x 128 code tile
constexpr int kMmaKsOff = 16384;   // K scales within a K segment
constexpr int kMmaVsOff = 18432;   // V scales within a K segment
constexpr int kMmaSlot = 19456;    // bytes per slot (multiple of 1024)

template <int HPK>
struct MmaCfg {
    static constexpr int HPKP = HPK < 4 ? 4 : HPK;   // heads padded for the layouts
    static constexpr int NT = HPKP / 8 > 0 ? HPKP / 8 : 1;  // score n8 tiles
    static constexpr int MT = (3 * HPKP + 15) / 16;  // PV m16 tiles (3 digits x heads)
    static constexpr int MROWS = 16 * MT;
    static constexpr int S_OFF = kMmaSlots * kMmaSlot;           // scores [TR][HPKP] f32
    static constexpr int A_OFF = S_OFF + kMmaTR * HPKP * 4;      // digits [8][MROWS][16]
    static constexpr int MISC_OFF = A_OFF + 8 * MROWS * 16;
    // misc: bars[kMmaSlots], red[kWarps][HPKP], mrun[HPKP], alpha[HPKP], vred[kWarps], u
    static constexpr int SMEM = MISC_OFF + kMmaSlots * 8 + (kWarps + 2) * HPKP * 4 + kWarps * 4 + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // room to align the base to 1024
    static_assert(kWarps * HPKP * 128 * 4 <= kMmaSlots * kMmaSlot, "acc staging must fit");
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

// D += A(16x32 u8, row) * B(32x8 s8, col), s32 accumulate.
__device__ __forceinline__ void mma_u8s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four int8 codes -> two exact f16 pairs (codes 0,1 and codes 2,3): bias the
// bytes to unsigned, splice them under the f16 exponent of 1024, subtract 1152.
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 x = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 y = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&x);
    hi = *reinterpret_cast<const uint32_t *>(&y);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
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

// One CTA: one chunk of ci.n rows starting at storage row `row_base` of one
// (sequence, live group).  Writes the partial (max, sum, acc) of each head.
template <int HPK>
__device__ void split_mma_body(const ChunkInfo &ci, int64_t row_base, const SplitArgs &a,
                               const CUtensorMap *kmap, const CUtensorMap *vmap, char *smem_raw) {
    using C = MmaCfg<HPK>;
    constexpr int HPKP = C::HPKP, NT = C::NT, MT = C::MT, MROWS = C::MROWS;
    char *sm = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gl4 = lane >> 2, t4 = lane & 3;
    float *S = reinterpret_cast<float *>(sm + C::S_OFF);
    char *A = sm + C::A_OFF;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::MISC_OFF);
    float *red = reinterpret_cast<float *>(bar + kMmaSlots);
    float *mrun = red + kWarps * HPKP;
    float *alpha = mrun + HPKP;
    float *vred = alpha + HPKP;
    float *ushared = vred + kWarps;

    const int n = ci.n;
    const int ntiles = (n + kMmaTR - 1) / kMmaTR;
    const int nseg = 2 * ntiles;

    if (tid == 0) {
        for (int s = 0; s < kMmaSlots; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    if (tid < HPKP) mrun[tid] = -INFINITY;
    __syncthreads();
    if (tid == 0)
        for (int j = 0; j < min(kMmaSlots, nseg); ++j) mma_issue<HPK>(ci, kmap, vmap, row_base, sm, bar, j);

    // ---- query terms: q * kcol * scale * log2e * 2^E_h = t1 + t2 (f16)
    // staging [HPKP][128] in the score area (exactly that size, free until the
    // first tile's scores)
    float *qf = S;
    static_assert(kMmaTR == 128, "the score area doubles as the q staging area");
    for (int i = tid; i < HPKP * 128; i += kThreads) {
        const int h = i >> 7, d = i & 127;
        qf[i] = h < a.hpk ? ci.q[h * 128 + d] * ci.kcol[d] * a.qscale : 0.0f;
    }
    __syncthreads();
    if (tid < HPKP) {
        float mx = 0.0f;
        for (int d = 0; d < 128; ++d) mx = fmaxf(mx, fabsf(qf[tid * 128 + d]));
        int e2 = 0;
        if (mx > 0.0f) {
            int ex;
            frexpf(mx, &ex);  // mx in [2^(ex-1), 2^ex)
            e2 = 14 - ex;
        }
        alpha[tid] = float(e2);  // exponent scratch, overwritten in the tile loop
    }
    __syncthreads();
    // B fragments: [group][k16 step][n-tile][term][2]
    uint32_t bq[4][2][NT][2][2];
    float qexp[NT][2];  // 2^-E of the heads this lane's score columns hold
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = nt * 8 + 2 * t4 + c;
            qexp[nt][c] = h < HPKP ? exp2f(-alpha[h]) : 0.0f;
        }
        const int hb = nt * 8 + gl4;  // the B column this lane feeds
        const float sc = hb < HPKP ? exp2f(alpha[hb]) : 0.0f;
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int c0 = 32 * g + 16 * ks + 4 * t4;
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] = hb < HPKP ? qf[hb * 128 + c0 + i] * sc : 0.0f;
                float r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) r[i] = x[i] - __half2float(__float2half_rn(x[i]));
                bq[g][ks][nt][0][0] = pack_half2(x[0], x[1]);
                bq[g][ks][nt][0][1] = pack_half2(x[2], x[3]);
                bq[g][ks][nt][1][0] = pack_half2(r[0], r[1]);
                bq[g][ks][nt][1][1] = pack_half2(r[2], r[3]);
            }
    }
    __syncthreads();  // qf staging read before the scores overwrite it

    // PV accumulators: this lane's heads x 8 channels (2 blocks x 4)
    constexpr int NH = HPKP >= 16 ? 2 : 1;  // heads per lane after the digit combine
    float acc[NH][8];
#pragma unroll
    for (int i = 0; i < NH; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[i][c] = 0.0f;
    float lsum = 0.0f;
    bool ok = true;

    const uint32_t A_base = smem_addr(A);
    for (int t = 0; t < ntiles && ok; ++t) {
        const int row0 = t * kMmaTR;
        const int nt_rows = min(kMmaTR, n - row0);
        int j = 2 * t;
        int slot = j % kMmaSlots;
        if (__syncthreads_or(!mbar_wait_bounded(&bar[slot], (j / kMmaSlots) & 1))) {
            ok = false;
            break;
        }
        const char *kseg = sm + slot * kMmaSlot;
        const uint32_t kbase = smem_addr(kseg);
        const float *ks_s = reinterpret_cast<const float *>(kseg + kMmaKsOff);
        const float *vs_s = reinterpret_cast<const float *>(kseg + kMmaVsOff);
        // ------------------------------------------------ scores (f16 MMA)
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
            const int mi = lane >> 3, rr = lane & 7;
            const int lrow = r0 + rr + 8 * (mi & 1);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int chunk = 2 * g + (mi >> 1);
                uint32_t w[4];
                ldsm_x4(kbase + lrow * 128 + ((chunk ^ (lrow & 7)) << 4), w);
                uint32_t a00, a02, a01, a03, a10, a12, a11, a13;
                codes_to_f16(w[0], a00, a02);  // row gl4,   channels 4t..4t+3 (k step 0)
                codes_to_f16(w[1], a01, a03);  // row gl4+8
                codes_to_f16(w[2], a10, a12);  // row gl4,   k step 1
                codes_to_f16(w[3], a11, a13);  // row gl4+8
                float dg[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) dg[nt][i] = 0.0f;
#pragma unroll
                    for (int tm = 0; tm < 2; ++tm) {
                        mma_f16(dg[nt], a00, a01, a02, a03, bq[g][0][nt][tm][0], bq[g][0][nt][tm][1]);
                        mma_f16(dg[nt], a10, a11, a12, a13, bq[g][1][nt][tm][0], bq[g][1][nt][tm][1]);
                    }
                    sacc[nt][0] = fmaf(kA[g], dg[nt][0], sacc[nt][0]);
                    sacc[nt][1] = fmaf(kA[g], dg[nt][1], sacc[nt][1]);
                    sacc[nt][2] = fmaf(kB[g], dg[nt][2], sacc[nt][2]);
                    sacc[nt][3] = fmaf(kB[g], dg[nt][3], sacc[nt][3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int h = nt * 8 + 2 * t4 + c;
                    if (h < HPKP) {
                        const int ra = r0 + gl4, rb = r0 + gl4 + 8;
                        const float sa = ra < nt_rows ? sacc[nt][c] * qexp[nt][c] : -INFINITY;
                        const float sb = rb < nt_rows ? sacc[nt][2 + c] * qexp[nt][c] : -INFINITY;
                        S[ra * HPKP + h] = sa;
                        S[rb * HPKP + h] = sb;
                        if (a.scores != nullptr && h < a.hpk) {
                            if (ra < nt_rows) a.scores[ci.score0 + int64_t(row0 + ra) * a.hpk + h] = sa;
                            if (rb < nt_rows) a.scores[ci.score0 + int64_t(row0 + rb) * a.hpk + h] = sb;
                        }
                    }
                }
            }
        }
        // largest V row scale of the tile (rows < nt_rows)
        {
            float v = tid < nt_rows ? vs_s[tid] : 0.0f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) vred[warp] = v;
        }
        __syncthreads();
        // ------------------------------------------------ tile max, rescale
        {
            const int h = tid % HPKP;
            float mx = -INFINITY;
            for (int r = tid / HPKP; r < nt_rows; r += kThreads / HPKP) mx = fmaxf(mx, S[r * HPKP + h]);
#pragma unroll
            for (int off = HPKP; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane < HPKP) red[warp * HPKP + lane] = mx;
        }
        __syncthreads();
        if (tid < HPKP) {
            float mx = red[tid];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red[w * HPKP + tid]);
            const float mo = mrun[tid];
            const float mn = fmaxf(mo, mx);
            alpha[tid] = (mo == -INFINITY) ? 0.0f : exp2f(mo - mn);
            mrun[tid] = mn;
        }
        if (tid == 0) {
            float vm = vred[0];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) vm = fmaxf(vm, vred[w]);
            ushared[0] = vm > 0.0f ? vm * (1.0f / 16777215.0f) : 1.0f;
        }
        __syncthreads();
        // ------------------------------- weights -> 24-bit unsigned digits
        {
            const int h = tid % HPKP;
            const float mn = mrun[h];
            const float inv_u = 1.0f / ushared[0];
            lsum *= alpha[h];
            for (int qd = tid / HPKP; qd < 32; qd += kThreads / HPKP) {
                const int kb = qd >> 3, half = (qd >> 2) & 1, tq = qd & 3;
                const int pbase = 32 * kb + 16 * half + 2 * tq;
                uint32_t qv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int p = pbase + (i & 1) + 8 * (i >> 1);
                    float wv = 0.0f;
                    if (h < a.hpk && p < nt_rows) {
                        const float e = exp2f(S[p * HPKP + h] - mn);
                        lsum += e;
                        wv = e * vs_s[p] * inv_u;
                    }
                    qv[i] = min(__float2uint_rn(wv), 0xFFFFFFu);
                }
                const uint32_t lo0 = __byte_perm(qv[0], qv[1], 0x0040);
                const uint32_t hi0 = __byte_perm(qv[2], qv[3], 0x0040);
                const uint32_t lo1 = __byte_perm(qv[0], qv[1], 0x0051);
                const uint32_t hi1 = __byte_perm(qv[2], qv[3], 0x0051);
                const uint32_t lo2 = __byte_perm(qv[0], qv[1], 0x0062);
                const uint32_t hi2 = __byte_perm(qv[2], qv[3], 0x0062);
                const int kc = 2 * kb + half;
                char *dst = A + (kc * MROWS) * 16 + 4 * tq;
                *reinterpret_cast<uint32_t *>(dst + (0 * HPKP + h) * 16) = __byte_perm(lo0, hi0, 0x5410);
                *reinterpret_cast<uint32_t *>(dst + (1 * HPKP + h) * 16) = __byte_perm(lo1, hi1, 0x5410);
                *reinterpret_cast<uint32_t *>(dst + (2 * HPKP + h) * 16) = __byte_perm(lo2, hi2, 0x5410);
            }
        }
        __syncthreads();  // digits visible; K slot drained
        if (tid == 0 && j + kMmaSlots < nseg) mma_issue<HPK>(ci, kmap, vmap, row_base, sm, bar, j + kMmaSlots);
        // ------------------------------------------------ P.V (u8 x s8 MMA)
        j = 2 * t + 1;
        slot = j % kMmaSlots;
        if (__syncthreads_or(!mbar_wait_bounded(&bar[slot], (j / kMmaSlots) & 1))) {
            ok = false;
            break;
        }
        const uint32_t vbase = smem_addr(sm + slot * kMmaSlot);
        int dv[MT][4][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int i = 0; i < 4; ++i) dv[mt][q4][i] = 0;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            uint32_t af[MT][4];
            {
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int m = 16 * mt + rr + 8 * (mi & 1);
                    const int kc = 2 * kb + (mi >> 1);
                    ldsm_x4(A_base + (kc * MROWS + m) * 16, af[mt]);
                }
            }
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int cc = 2 * warp + cb;  // 16-channel chunk of the row
                const int pos = 32 * kb + 8 * (lane >> 3) + (lane & 7);
                uint32_t x[4];
                ldsm_x4_t(vbase + pos * 128 + ((cc ^ (pos & 7)) << 4), x);
                const uint32_t be0 = __byte_perm(x[0], x[1], 0x6420);
                const uint32_t be1 = __byte_perm(x[2], x[3], 0x6420);
                const uint32_t bo0 = __byte_perm(x[0], x[1], 0x7531);
                const uint32_t bo1 = __byte_perm(x[2], x[3], 0x7531);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    mma_u8s8(dv[mt][2 * cb], af[mt], be0, be1);
                    mma_u8s8(dv[mt][2 * cb + 1], af[mt], bo0, bo1);
                }
            }
        }
        // digits -> f32, fold into the running accumulator:
        // acc = acc * alpha + u * (d0 + 256 d1 + 65536 d2)
        {
            const float u = ushared[0];
            if (HPKP == 4) {
                // rows: g<4 -> (digit 0, head g) and (digit 2, head g); g>=4 -> digit 1 of head g-4
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int d1 = __shfl_xor_sync(0xffffffffu, dv[0][q4][c], 16);
                        if (gl4 < 4) {
                            const int lo = d1 * 256 + dv[0][q4][c];
                            const float val = fmaf(float(dv[0][q4][2 + c]), 65536.0f, float(lo));
                            const int ch = (q4 >> 1) * 4 + 2 * c + (q4 & 1);
                            acc[0][ch] = fmaf(acc[0][ch], alpha[gl4], u * val);
                        }
                    }
            } else if (HPKP == 8) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int lo = dv[0][q4][2 + c] * 256 + dv[0][q4][c];
                        const float val = fmaf(float(dv[1][q4][c]), 65536.0f, float(lo));
                        const int ch = (q4 >> 1) * 4 + 2 * c + (q4 & 1);
                        acc[0][ch] = fmaf(acc[0][ch], alpha[gl4], u * val);
                    }
            } else {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int lo = dv[1][q4][2 * hh + c] * 256 + dv[0][q4][2 * hh + c];
                            const float val = fmaf(float(dv[2][q4][2 * hh + c]), 65536.0f, float(lo));
                            const int ch = (q4 >> 1) * 4 + 2 * c + (q4 & 1);
                            acc[hh][ch] = fmaf(acc[hh][ch], alpha[gl4 + 8 * hh], u * val);
                        }
            }
        }
        __syncthreads();  // V slot drained, alpha/u no longer needed
        if (tid == 0 && j + kMmaSlots < nseg) mma_issue<HPK>(ci, kmap, vmap, row_base, sm, bar, j + kMmaSlots);
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
    {
        const int h = tid % HPKP;
        float l = lsum;
#pragma unroll
        for (int off = HPKP; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane < HPKP) red[warp * HPKP + lane] = l;
    }
    __syncthreads();
    if (tid < a.hpk) {
        float l = red[tid];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) l += red[w * HPKP + tid];
        a.pm[ci.pidx0 + tid] = mrun[tid];
        a.pl[ci.pidx0 + tid] = l;
    }
    // lane (gl4, t4) of warp w holds channels 32w + 16cb + 4t4 + {0..3} of
    // head gl4 (+8 for the second head when HPKP == 16)
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        const int h = gl4 + 8 * hh;
        const bool mine = (HPKP == 4 ? gl4 < 4 : true) && h < a.hpk;
        if (mine) {
            float *dst = a.pacc + (ci.pidx0 + h) * 128 + 32 * warp + 4 * t4;
            *reinterpret_cast<float4 *>(dst) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
            *reinterpret_cast<float4 *>(dst + 16) =
                make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
        }
    }
}

template <int HPK>
__global__ void __launch_bounds__(kThreads, 2)
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
    ci.score0 = row * a.hpk;
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
