// kvd_decode_kernels.cuh -- split-KV decode attention kernels (templates).
//
// One CTA owns one chunk of consecutive cached rows of one (sequence, KV
// group) and every query head of that group (GQA: each K and V row is read
// once for all hpk heads, as cortiq attend_group reads it).  The chunk is
// streamed through shared memory in tiles by 1-D bulk asynchronous copies
// (TMA bulk engine, mbarrier completion) into a ring of kNSeg slots that
// alternates K tiles (with their scales) and V tiles.  Per tile:
//   score pass  lanes split the channels of a row; each lane forms partial
//               dots for RB rows x HPK heads and one butterfly
//               reduce-scatter over the warp leaves one complete score per
//               lane (dequantisation fused in: int8 codes x per-32-channel
//               scale, field and softmax scale folded into q once);
//   softmax     running max per head, rescale of the running sum and
//               accumulator by exp2(old - new) (the online recurrence of
//               rswa fold, applied per tile);
//   value pass  each warp walks rows, lanes own channels, accumulators in
//               registers; V codes are weighted by exp * row scale.
// The CTA writes its (max, sum, accumulator) partial per head; a second
// kernel merges the chunks of a sequence by log-sum-exp and applies the V
// field.  Scores are kept in the log2 domain (q is pre-scaled by log2(e)).
#pragma once

#include <math.h>

#include "kvd_internal.cuh"

namespace kvd {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kNSeg = 4;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int ce_max(int a, int b) { return a > b ? a : b; }
constexpr int ce_min(int a, int b) { return a < b ? a : b; }
constexpr int ce_log2(int x) { return x <= 1 ? 0 : 1 + ce_log2(x / 2); }
constexpr int ce_round(int x, int a) { return (x + a - 1) / a * a; }

// Tile geometry for a head dim and storage mode.  KI8: int8 K codes with
// one scale per row (the R-SWA int8 mirror) instead of one per 32 channels.
template <int HD, bool KQ, bool VQ, bool KI8 = false>
struct TileCfg {
    static constexpr int NG = HD / kKGroup;
    static constexpr int NKS = KI8 ? 1 : NG;  // K scales per row
    static constexpr int CPL = HD / 32;  // channels per lane
    static constexpr int KROW = KQ ? HD : 4 * HD;
    static constexpr int VROW = VQ ? HD : 4 * HD;
    static constexpr int TR = ce_min(256, 16384 / ce_max(KROW, VROW));  // rows per tile
    static constexpr int KS_OFF = TR * KROW;
    static constexpr int VS_OFF = KS_OFF + (KQ ? TR * NKS * 4 : 0);
    static constexpr int KSEG = VS_OFF + (VQ ? TR * 4 : 0);
    static constexpr int VSEG = TR * VROW;
    // Ring slots alternate K segments (even slots) and V segments (odd slots),
    // each sized for its own segment: with one int8 component (q8k, q8v) the
    // ring is ~40 KB instead of 64 KB, so four CTAs fit an SM instead of three.
    static constexpr int KSLOT = ce_round(KSEG, 128);
    static constexpr int VSLOT = ce_round(VSEG, 128);
    static constexpr int RING = 2 * (KSLOT + VSLOT);
    static_assert(kNSeg == 4, "segment j goes to slot j % 4: K in slots 0 and 2, V in 1 and 3");
    static __host__ __device__ constexpr int slot_off(int slot) { return (slot >> 1) * (KSLOT + VSLOT) + (slot & 1) * KSLOT; }
};

template <int HD, int HPK, bool KQ, bool VQ, bool KI8 = false>
struct SplitCfg : TileCfg<HD, KQ, VQ, KI8> {
    using T = TileCfg<HD, KQ, VQ, KI8>;
    static constexpr int RPW = T::TR / kWarps;             // score rows per warp per tile
    static constexpr int RB = ce_min(32 / HPK, RPW);       // rows per reduce batch
    static constexpr int E = RB * HPK;                     // entries per reduce (<= 32)
    static constexpr int LOGE = ce_log2(E);
    static constexpr int SC_OFF = T::RING;                 // scores/weights [TR][HPK]
    static constexpr int MISC_OFF = SC_OFF + T::TR * HPK * 4;
    // misc: kNSeg mbarriers, red[kWarps][HPK], mrun[HPK], alpha[HPK], flag
    static constexpr int SMEM = MISC_OFF + kNSeg * 8 + (kWarps + 2) * HPK * 4 + 16;
    static_assert(kWarps * HPK * HD * 4 <= T::RING, "accumulator reduction must fit");
    static_assert((1 << LOGE) == E, "reduce entries must be a power of two");
};

// First visible row of a sequence holding L rows under a sliding window of
// `window` rows (0 = no window): cortiq attend_group_upto's `first` when the
// caller passes stored - window.  Always <= L - 1 for L >= 1.
__host__ __device__ __forceinline__ int64_t first_visible(int64_t L, int64_t window) {
    return window > 0 && L > window ? L - window : 0;
}

// Softcap in the log2 domain: scores s2 = s * log2(e) are capped as
// c2 * tanh(s2 / c2) with c2 = softcap * log2(e), the same as capping s.
__device__ __forceinline__ float softcap_log2(float s2, float c2) { return c2 * tanhf(s2 / c2); }

// Arguments common to every split launch.
struct SplitArgs {
    const float *q;        // [.., n_q, HD] query rows
    int32_t n_q, hpk;      // query heads per sequence/stream; heads per KV group
    float qscale;          // softmax scale * log2(e)
    int32_t chunk;         // rows per chunk (multiple of every tile height)
    int32_t nc_max;        // chunk slots per (sequence, group) in the partials
    int32_t n_grp;         // groups per sequence in the partials (live heads / R-SWA heads)
    float *pm, *pl, *pacc; // partial max, sum, accumulator
    float *scores;         // per-row log2 scores for the imp pass, or null
    uint32_t *err;
    int64_t window = 0;      // sliding window in rows (0 = none)
    float softcap2 = 0.0f;   // softcap * log2(e) (0 = none)
    // Query-batched verify of K draft rows (K = 1: a plain decode): the group's
    // hpk = K * hg query rows are e = k * hg + h (draft k, head h of the hg
    // heads per KV group), query k sees rows [first_k, upto_k) with upto_k =
    // L - (K - 1 - k) and first_k the window's start counted back from upto_k.
    int32_t K = 1;
    int32_t hg = 0;
};

// Rows the earliest query of a verify sees at most: L - (K - 1), at least 0.
__host__ __device__ __forceinline__ int64_t verify_len(int64_t L, int32_t K) {
    return L - (K - 1) > 0 ? L - (K - 1) : 0;
}

// Where one CTA's chunk lives.
struct ChunkInfo {
    const char *k, *v, *ks, *vs;  // global address of the chunk's first row
    int n;                        // rows in the chunk (>= 1)
    int lo;                       // rows of the chunk before the first visible one
    int L, r0;                    // the sequence's rows and the chunk's first row (verify)
    int64_t pidx0;                // partial index of the group's head 0
    const float *q;               // query of the group's head 0
    const float *kcol;            // K field of the group, or null
    int64_t score0;               // scores index of the chunk's row 0, head 0 (or -1)
    int64_t score_ld;             // scores stride between heads (rows of the region)
};

// Butterfly reduce-scatter of E partial sums held by every lane: after it,
// lane l holds in v[0] the full warp sum of entry l >> (5 - LOGE).  T: float,
// or int for exact integer partials.
template <int E, int LOGE, typename T>
__device__ __forceinline__ T reduce_scatter(T (&v)[E], int lane) {
#pragma unroll
    for (int s = 0; s < LOGE; ++s) {
        const int off = 16 >> s;
        const int half = (E >> s) >> 1;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const T send = upper ? v[i] : v[i + half];
            const T keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int s = LOGE; s < 5; ++s) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> s);
    return v[0];
}

// Load CPL consecutive channels of a row (lane's share) as f32.  PERM: int8
// codes convert by byte permutes and float subtracts (full-rate pipes)
// rather than int-to-float conversions (a quarter-rate pipe); the value pass
// uses it, where each code feeds few FMAs.
template <int CPL, bool Q, bool PERM = false>
__device__ __forceinline__ void load_lane(const char *row, int lane, float (&x)[CPL]) {
    if (Q && PERM) {
        // code + 128 (the byte XOR 0x80) as the low mantissa byte of 2^23:
        // the float 2^23 + 128 + code, exact; one subtract leaves the code
        const uint32_t w = (CPL == 4 ? reinterpret_cast<const uint32_t *>(row)[lane]
                                     : uint32_t(reinterpret_cast<const uint16_t *>(row)[lane])) ^
                           0x80808080u;
#pragma unroll
        for (int j = 0; j < CPL; ++j)
            x[j] = __uint_as_float(__byte_perm(w, 0x4b000000u, 0x7650u | uint32_t(j))) - 8388736.0f;
    } else if (Q) {
        if (CPL == 4) {
            const uint32_t w = reinterpret_cast<const uint32_t *>(row)[lane];
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = float(int8_t((w >> (8 * j)) & 0xffu));
        } else {
            const uint32_t w = reinterpret_cast<const uint16_t *>(row)[lane];
#pragma unroll
            for (int j = 0; j < CPL; ++j) x[j] = float(int8_t((w >> (8 * j)) & 0xffu));
        }
    } else {
        if (CPL == 4) {
            const float4 f = reinterpret_cast<const float4 *>(row)[lane];
            x[0] = f.x;
            x[1] = f.y;
            x[2] = f.z;
            x[3] = f.w;
        } else {
            const float2 f = reinterpret_cast<const float2 *>(row)[lane];
            x[0] = f.x;
            x[1] = f.y;
        }
    }
}

template <int HD, int HPK, bool KQ, bool VQ, bool KI8>
__device__ __forceinline__ void issue_segment(const ChunkInfo &ci, char *smem, uint64_t *bar,
                                              int j) {
    using C = SplitCfg<HD, HPK, KQ, VQ, KI8>;
    const int slot = j % kNSeg;
    const int t = j >> 1;
    const int row0 = t * C::TR;
    const int nt = min(C::TR, ci.n - row0);
    const int rows = (nt + kRowAlign - 1) / kRowAlign * kRowAlign;
    char *dst = smem + C::slot_off(slot);
    if ((j & 1) == 0) {
        uint32_t bytes = uint32_t(rows) * C::KROW;
        if (KQ) bytes += uint32_t(rows) * C::NKS * 4;
        if (VQ) bytes += uint32_t(rows) * 4;
        mbar_arrive_expect_tx(&bar[slot], bytes);
        bulk_g2s(dst, ci.k + int64_t(row0) * C::KROW, uint32_t(rows) * C::KROW, &bar[slot]);
        if (KQ)
            bulk_g2s(dst + C::KS_OFF, ci.ks + int64_t(row0) * C::NKS * 4, uint32_t(rows) * C::NKS * 4,
                     &bar[slot]);
        if (VQ)
            bulk_g2s(dst + C::VS_OFF, ci.vs + int64_t(row0) * 4, uint32_t(rows) * 4, &bar[slot]);
    } else {
        const uint32_t bytes = uint32_t(rows) * C::VROW;
        mbar_arrive_expect_tx(&bar[slot], bytes);
        bulk_g2s(dst, ci.v + int64_t(row0) * C::VROW, bytes, &bar[slot]);
    }
}

// Quantise one f32 value against a row scale as rswa quantize_row_i8 does:
// IEEE division, round half to even, clamp to [-127, 127].
__device__ __forceinline__ int quant_code_i8(float x, float sc) {
    const float t = rintf(__fdiv_rn(x, sc));
    return int(fminf(fmaxf(t, -127.0f), 127.0f));
}

// OPT: the call has a window or a softcap (compiled out of the common path).
// KI8: the R-SWA int8 mirror (int8 K with one scale per row; several query
// rows only for a verify): each query row is quantised like a cache row and
// the QK dot is the exact integer dot of the codes, scaled by qscale *
// kscale[row] after.
template <int HD, int HPK, bool KQ, bool VQ, bool OPT, bool KI8 = false>
__device__ void split_body(const ChunkInfo &ci, const SplitArgs &a, char *smem) {
    using C = SplitCfg<HD, HPK, KQ, VQ, KI8>;
    static_assert(!KI8 || KQ, "the int8 mirror has int8 K");
    constexpr int CPL = C::CPL, TR = C::TR;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *sc = reinterpret_cast<float *>(smem + C::SC_OFF);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::MISC_OFF);
    float *red = reinterpret_cast<float *>(bar + kNSeg);
    float *mrun = red + kWarps * HPK;
    float *alpha = mrun + HPK;

    const int n = ci.n;
    const int ntiles = (n + TR - 1) / TR;
    const int nseg = 2 * ntiles;

    if (tid == 0) {
        for (int s = 0; s < kNSeg; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    if (tid < HPK) mrun[tid] = -INFINITY;
    __syncthreads();
    if (tid == 0)
        for (int j = 0; j < min(kNSeg, nseg); ++j) issue_segment<HD, HPK, KQ, VQ, KI8>(ci, smem, bar, j);

    // Query of every head of the group for this lane's channels, with the
    // K field and the softmax scale (in log2 units) folded in.
    float qr[HPK][CPL];
    uint32_t qi[HPK];    // KI8: this lane's query codes per query row, packed bytes
    float qfac[HPK];     // KI8: qscale * softmax scale * log2(e) per query row
#pragma unroll
    for (int h = 0; h < HPK; ++h) {
        qi[h] = 0;
        qfac[h] = 0.0f;
        if (KI8 && h < a.hpk) {
            const int64_t qo = a.K > 1 ? int64_t(h / a.hg) * a.n_q * HD + int64_t(h % a.hg) * HD : int64_t(h) * HD;
            float x[CPL], mx = 0.0f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                x[j] = ci.q[qo + lane * CPL + j];
                mx = fmaxf(mx, fabsf(x[j]));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float sq = mx > 0.0f ? __fdiv_rn(mx, 127.0f) : 1.0f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) qi[h] |= (uint32_t(quant_code_i8(x[j], sq)) & 0xffu) << (8 * j);
            qfac[h] = sq * a.qscale;
        }
    }
#pragma unroll
    for (int h = 0; h < HPK; ++h) {
        // query row h: draft h / hg, head h % hg (h itself for a plain decode)
        const int64_t qo = a.K > 1 ? int64_t(h / a.hg) * a.n_q * HD + int64_t(h % a.hg) * HD : int64_t(h) * HD;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            float x = 0.0f;
            if (!KI8 && h < a.hpk) {
                x = ci.q[qo + lane * CPL + j];
                if (KQ) x *= ci.kcol[lane * CPL + j];
                x *= a.qscale;
            }
            qr[h][j] = x;
        }
    }
    float acc[HPK][CPL];
#pragma unroll
    for (int h = 0; h < HPK; ++h)
#pragma unroll
        for (int j = 0; j < CPL; ++j) acc[h][j] = 0.0f;
    float lsum = 0.0f;  // this thread's share of the running sum of head tid % HPK
    bool ok = true;

    for (int t = 0; t < ntiles && ok; ++t) {
        const int row0 = t * TR;
        const int nt = min(TR, n - row0);
        // ---------------------------------------------------- K tile
        int j = 2 * t;
        int slot = j % kNSeg;
        // Every thread waits; the give-up decision is made block-wide so that
        // no thread leaves the loop while others sit in a barrier.
        if (__syncthreads_or(!mbar_wait_bounded(&bar[slot], (j / kNSeg) & 1))) {
            ok = false;
            break;
        }
        const char *kseg = smem + C::slot_off(slot);
#pragma unroll 1
        for (int bt = 0; bt < C::RPW / C::RB; ++bt) {
            const int rbase = warp * C::RPW + bt * C::RB;
            float v[C::E];
            int vi[C::E];  // KI8: the codes' dot products, exact integers
#pragma unroll
            for (int r = 0; r < C::RB; ++r) {
                if (KI8) {
                    // exact: |partial| <= 4 * 127 * 127, the warp sum <= 128 * 127 * 127
                    const char *kr = kseg + (rbase + r) * C::KROW;
                    const uint32_t kw = CPL == 4 ? reinterpret_cast<const uint32_t *>(kr)[lane]
                                                 : uint32_t(reinterpret_cast<const uint16_t *>(kr)[lane]);
#pragma unroll
                    for (int h = 0; h < HPK; ++h) vi[r * HPK + h] = __dp4a(int(qi[h]), int(kw), 0);
                    continue;
                }
                float x[CPL];
                load_lane<CPL, KQ>(kseg + (rbase + r) * C::KROW, lane, x);
                float gs = 1.0f;
                if (KQ)
                    gs = reinterpret_cast<const float *>(kseg + C::KS_OFF)[(rbase + r) * C::NG +
                                                                           (lane * CPL) / kKGroup];
#pragma unroll
                for (int h = 0; h < HPK; ++h) {
                    float p = 0.0f;
#pragma unroll
                    for (int jj = 0; jj < CPL; ++jj) p = fmaf(qr[h][jj], x[jj], p);
                    v[r * HPK + h] = KQ ? p * gs : p;
                }
            }
            // KI8: reduced in integers, one conversion per row and query
            // (an integer below 2^24, so the float is the same either way)
            float s = KI8 ? float(reduce_scatter<C::E, C::LOGE>(vi, lane)) : reduce_scatter<C::E, C::LOGE>(v, lane);
            if ((lane & ((32 >> C::LOGE) - 1)) == 0) {
                const int e = lane >> (5 - C::LOGE);
                const int r = rbase + e / HPK, h = e % HPK;
                if (KI8) {
                    float qf = qfac[0];
#pragma unroll
                    for (int hh = 1; hh < HPK; ++hh)
                        if (h == hh) qf = qfac[hh];
                    s = s * reinterpret_cast<const float *>(kseg + C::KS_OFF)[r] * qf;
                }
                bool vis = r < nt && (!OPT || row0 + r >= ci.lo);
                if (OPT && a.K > 1 && vis) {
                    // verify: this query row's own causal limit and window
                    const int64_t upto = int64_t(ci.L) - (a.K - 1 - h / a.hg);
                    const int64_t row = int64_t(ci.r0) + row0 + r;
                    vis = row < upto && row >= first_visible(upto, a.window);
                }
                const float sv =
                    vis ? (OPT && a.softcap2 > 0.0f ? softcap_log2(s, a.softcap2) : s) : -INFINITY;
                sc[r * HPK + h] = sv;
                if (a.scores != nullptr && vis && h < a.hpk)
                    a.scores[ci.score0 + h * ci.score_ld + row0 + r] = sv;
            }
        }
        __syncthreads();
        // ------------------------------------------- tile max per head
        {
            const int h = tid % HPK;
            float mx = -INFINITY;
            for (int r = tid / HPK; r < nt; r += kThreads / HPK) mx = fmaxf(mx, sc[r * HPK + h]);
#pragma unroll
            for (int off = HPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane < HPK) red[warp * HPK + lane] = mx;
        }
        __syncthreads();
        if (tid < HPK) {
            float mx = red[tid];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red[w * HPK + tid]);
            const float mo = mrun[tid];
            const float mn = fmaxf(mo, mx);
            alpha[tid] = (mo == -INFINITY) ? 0.0f : exp2f(mo - mn);
            mrun[tid] = mn;
        }
        __syncthreads();
        // --------------------- weights exp2(s - max) (x V row scale), sums
        {
            const int h = tid % HPK;
            const float mn = mrun[h];
            lsum *= alpha[h];
            const float *vsr = reinterpret_cast<const float *>(kseg + C::VS_OFF);
            for (int r = tid / HPK; r < nt; r += kThreads / HPK) {
                // a head that has seen no visible row yet (verify) keeps weight 0
                const float e = mn == -INFINITY ? 0.0f : exp2f(sc[r * HPK + h] - mn);
                lsum += e;
                sc[r * HPK + h] = VQ ? e * vsr[r] : e;
            }
        }
        __syncthreads();  // K slot drained, weights visible
        if (tid == 0 && j + kNSeg < nseg) issue_segment<HD, HPK, KQ, VQ, KI8>(ci, smem, bar, j + kNSeg);
        // ---------------------------------------------------- V tile
        j = 2 * t + 1;
        slot = j % kNSeg;
        if (__syncthreads_or(!mbar_wait_bounded(&bar[slot], (j / kNSeg) & 1))) {
            ok = false;
            break;
        }
        const char *vseg = smem + C::slot_off(slot);
        // this tile's rows accumulate into fresh registers, folded into the
        // running (rescaled) sum once per tile: short rounding chains
        float tacc[HPK][CPL];
#pragma unroll
        for (int h = 0; h < HPK; ++h)
#pragma unroll
            for (int jj = 0; jj < CPL; ++jj) tacc[h][jj] = 0.0f;
        for (int r = warp; r < nt; r += kWarps) {
            float x[CPL];
            load_lane<CPL, VQ, true>(vseg + r * C::VROW, lane, x);
            float w[HPK];
            if (HPK % 4 == 0) {
#pragma unroll
                for (int h = 0; h < HPK; h += 4) {
                    const float4 w4 = *reinterpret_cast<const float4 *>(&sc[r * HPK + h]);
                    w[h] = w4.x;
                    w[h + 1] = w4.y;
                    w[h + 2] = w4.z;
                    w[h + 3] = w4.w;
                }
            } else {
#pragma unroll
                for (int h = 0; h < HPK; ++h) w[h] = sc[r * HPK + h];
            }
#pragma unroll
            for (int h = 0; h < HPK; ++h)
#pragma unroll
                for (int jj = 0; jj < CPL; ++jj) tacc[h][jj] = fmaf(w[h], x[jj], tacc[h][jj]);
        }
#pragma unroll
        for (int h = 0; h < HPK; ++h) {
            const float al = alpha[h];
#pragma unroll
            for (int jj = 0; jj < CPL; ++jj) acc[h][jj] = fmaf(acc[h][jj], al, tacc[h][jj]);
        }
        __syncthreads();  // V slot drained
        if (tid == 0 && j + kNSeg < nseg) issue_segment<HD, HPK, KQ, VQ, KI8>(ci, smem, bar, j + kNSeg);
    }

    if (!ok) {  // block-uniform (decided by __syncthreads_or above)
        // A copy never completed: record it, give the copies still in flight a
        // bounded chance to land (so none writes into a successor CTA's
        // shared memory), and leave without a partial.
        if (tid == 0) {
            set_error(a.err, kErrTimeout);
            for (int s = 0; s < kNSeg; ++s) (void)mbar_wait_bounded(&bar[s], 0, 100000000ull);
            for (int s = 0; s < kNSeg; ++s) (void)mbar_wait_bounded(&bar[s], 1, 100000000ull);
        }
        return;
    }

    // ------------------------------------------------------ partial out
    {
        float l = lsum;
#pragma unroll
        for (int off = HPK; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane < HPK) red[warp * HPK + lane] = l;
    }
    float *accs = reinterpret_cast<float *>(smem);  // [kWarps][HPK][HD], reuses the slots
#pragma unroll
    for (int h = 0; h < HPK; ++h)
#pragma unroll
        for (int jj = 0; jj < CPL; ++jj) accs[(warp * HPK + h) * HD + lane * CPL + jj] = acc[h][jj];
    __syncthreads();
    if (tid < a.hpk && tid < HPK) {
        float l = red[tid];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) l += red[w * HPK + tid];
        a.pm[ci.pidx0 + tid] = mrun[tid];
        a.pl[ci.pidx0 + tid] = l;
    }
    for (int i = tid; i < a.hpk * HD; i += kThreads) {
        const int h = i / HD, d = i % HD;
        float s = accs[h * HD + d];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) s += accs[(w * HPK + h) * HD + d];
        a.pacc[(ci.pidx0 + h) * HD + d] = s;
    }
}

// ---------------------------------------------------------------- layer

struct LayerSrc {
    const float *kf, *vf;
    const int8_t *kq, *vq;
    const float *ks, *vs, *kcol;
    const int64_t *row_base, *cap;
    const int32_t *seq_len, *live;
    int32_t n_live;
};

// Up to 4 heads per group the kernel fits 102 registers without spilling, so
// five CTAs share an SM where shared memory allows (the q8k and q8v rings);
// more heads per group need the larger register budget of two.
template <int HD, int HPK, bool KQ, bool VQ, bool OPT>
__global__ void __launch_bounds__(kThreads, HPK <= 4 ? 5 : 2) split_layer_kernel(SplitArgs a, LayerSrc src) {
    extern __shared__ __align__(128) char smem[];
    const int b = blockIdx.z, gl = blockIdx.y, c = blockIdx.x;
    const int L = src.seq_len[b];
    // chunks start at the first visible row (of the earliest query, for a
    // verify) rounded down to kRowAlign (the bulk copies' alignment); the rows
    // before it are masked in chunk 0
    const int64_t first = first_visible(verify_len(L, a.K), a.window);
    const int64_t f0 = first / kRowAlign * kRowAlign;
    const int64_t r0 = f0 + int64_t(c) * a.chunk;
    if (r0 >= L) return;
    const int64_t cap = src.cap[b];
    if (L > cap) {
        if (threadIdx.x == 0) set_error(a.err, kErrBounds);
        return;
    }
    const int64_t row = src.row_base[b] + int64_t(gl) * cap + r0;
    ChunkInfo ci;
    ci.lo = int(first - r0 > 0 ? first - r0 : 0);
    ci.L = L;
    ci.r0 = int(r0);
    ci.k = KQ ? reinterpret_cast<const char *>(src.kq + row * HD)
              : reinterpret_cast<const char *>(src.kf + row * HD);
    ci.v = VQ ? reinterpret_cast<const char *>(src.vq + row * HD)
              : reinterpret_cast<const char *>(src.vf + row * HD);
    ci.ks = KQ ? reinterpret_cast<const char *>(src.ks + row * (HD / kKGroup)) : nullptr;
    ci.vs = VQ ? reinterpret_cast<const char *>(src.vs + row) : nullptr;
    ci.n = int(a.chunk < L - r0 ? int64_t(a.chunk) : L - r0);
    ci.pidx0 = ((int64_t(b) * a.n_grp + gl) * a.nc_max + c) * a.hpk;
    const int g = src.live[gl];
    const int hg = a.K > 1 ? a.hg : a.hpk;  // query heads per KV group
    ci.q = a.q + (int64_t(b) * a.K * a.n_q + int64_t(g) * hg) * HD;
    ci.kcol = KQ ? src.kcol + (int64_t(b) * src.n_live + gl) * HD : nullptr;
    // scores region of (b, gl): [hpk][cap] starting at its first storage row * hpk
    ci.score0 = (src.row_base[b] + int64_t(gl) * cap) * a.hpk + r0;
    ci.score_ld = cap;
    split_body<HD, HPK, KQ, VQ, OPT>(ci, a, smem);
}

// ---------------------------------------------------------------- R-SWA

struct RswaTable {
    int32_t s0, n;                // first stream of the launch, streams in it
    int32_t prefill_len[kSlice];  // reference rows per stream
    int32_t ring_len[kSlice];     // ring rows per stream
};

struct RswaSrc {
    const float *ref_k, *ref_v, *ring_k, *ring_v;      // f32 regions
    const int8_t *ref_k8, *ref_v8, *ring_k8, *ring_v8;  // int8 mirror codes
    const float *ref_ks, *ref_vs, *ring_ks, *ring_vs;   // int8 mirror row scales
    int64_t ref_cap;
    int32_t W, H;
};

// I8: read the int8 mirror (rswa decode_attention_int8) instead of the f32
// regions (decode_attention_scalar_head).  HPK > 1 only for a verify: the
// a.K = a.hpk draft queries of a head share every row (q [B][K][H][HD]).
template <int HD, bool I8, int HPK = 1>
__global__ void __launch_bounds__(kThreads, 2) split_rswa_kernel(SplitArgs a, RswaSrc src,
                                                                 RswaTable tb) {
    extern __shared__ __align__(128) char smem[];
    const int si = blockIdx.z, h = blockIdx.y, c = blockIdx.x;
    if (si >= tb.n) return;
    const int s = tb.s0 + si;
    const int pl = tb.prefill_len[si], rl = tb.ring_len[si];
    const int ncp = (pl + a.chunk - 1) / a.chunk;
    const int ncr = (rl + a.chunk - 1) / a.chunk;
    ChunkInfo ci;
    const int64_t head = int64_t(s) * src.H + h;
    ci.ks = ci.vs = nullptr;
    if (c < ncp) {
        const int64_t row = head * src.ref_cap + int64_t(c) * a.chunk;
        if (I8) {
            ci.k = reinterpret_cast<const char *>(src.ref_k8 + row * HD);
            ci.v = reinterpret_cast<const char *>(src.ref_v8 + row * HD);
            ci.ks = reinterpret_cast<const char *>(src.ref_ks + row);
            ci.vs = reinterpret_cast<const char *>(src.ref_vs + row);
        } else {
            ci.k = reinterpret_cast<const char *>(src.ref_k + row * HD);
            ci.v = reinterpret_cast<const char *>(src.ref_v + row * HD);
        }
        ci.n = min(a.chunk, pl - c * a.chunk);
    } else if (c - ncp < ncr) {
        const int cr = c - ncp;
        const int64_t row = head * src.W + int64_t(cr) * a.chunk;
        if (I8) {
            ci.k = reinterpret_cast<const char *>(src.ring_k8 + row * HD);
            ci.v = reinterpret_cast<const char *>(src.ring_v8 + row * HD);
            ci.ks = reinterpret_cast<const char *>(src.ring_ks + row);
            ci.vs = reinterpret_cast<const char *>(src.ring_vs + row);
        } else {
            ci.k = reinterpret_cast<const char *>(src.ring_k + row * HD);
            ci.v = reinterpret_cast<const char *>(src.ring_v + row * HD);
        }
        ci.n = min(a.chunk, rl - cr * a.chunk);
    } else {
        return;
    }
    ci.lo = 0;
    ci.pidx0 = (head * a.nc_max + c) * a.hpk;
    ci.q = a.q + (int64_t(s) * a.K * src.H + h) * HD;
    ci.kcol = nullptr;
    ci.score0 = -1;
    ci.score_ld = 0;
    split_body<HD, HPK, I8, I8, false, I8>(ci, a, smem);
}

// ---------------------------------------------------------------- merge

struct MergeArgs {
    const float *pm, *pl, *pacc;
    float *out;     // [.., n_q, HD]
    float *ml;      // (max, sum) per (sequence, query head) for the imp pass, or null
    const float *sinks = nullptr;  // learned sink logit per query head [n_q], or null
    int64_t window = 0;            // sliding window in rows (0 = none)
    int32_t n_q, hpk, n_grp, nc_max, chunk;
};

// Log-sum-exp merge of the chunk partials of one (sequence, query head):
// out[d] = field[d] * sum_c acc_c[d] 2^(m_c - M) / sum_c l_c 2^(m_c - M).
// orow: output row (sequence-major); hh: the query row within its group's
// partials; h: the query head (for its sink).  A query that saw no row at all
// (a verify query whose limit precedes every row) outputs zeros.
template <int HD>
__device__ void merge_body(const MergeArgs &a, int b, int64_t orow, int hh, int h, int grp, int nc,
                           const float *vcol) {
    const int d = threadIdx.x;
    float *o = a.out + orow * HD;
    const int64_t p0 = (int64_t(b) * a.n_grp + grp) * a.nc_max * a.hpk + hh;
    float Mr = -INFINITY;
    for (int c = 0; grp >= 0 && c < nc; ++c) Mr = fmaxf(Mr, a.pm[p0 + int64_t(c) * a.hpk]);
    if (grp < 0 || nc == 0 || Mr == -INFINITY) {
        o[d] = 0.0f;
        if (a.ml && d == 0) {
            a.ml[orow * 2] = -INFINITY;
            a.ml[orow * 2 + 1] = 0.0f;
        }
        return;
    }
    // a learned sink joins the maximum and the sum; it has no value row
    const float z = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
    const float M = fmaxf(Mr, z);
    float Ls = a.sinks ? exp2f(z - M) : 0.0f, s = 0.0f;
    for (int c = 0; c < nc; ++c) {
        const int64_t p = p0 + int64_t(c) * a.hpk;
        const float f = exp2f(a.pm[p] - M);
        Ls = fmaf(a.pl[p], f, Ls);
        s = fmaf(a.pacc[p * HD + d], f, s);
    }
    float r = s / Ls;
    if (vcol) r *= vcol[d];
    o[d] = r;
    if (a.ml && d == 0) {
        a.ml[orow * 2] = M;
        a.ml[orow * 2 + 1] = Ls;
    }
}

struct MergeLayerSrc {
    const int32_t *seq_len, *slot;
    const float *vcol;  // [n_seq][n_live][HD] or null
    int32_t n_live;
};

template <int HD>
__global__ void __launch_bounds__(HD) merge_layer_kernel(MergeArgs a, MergeLayerSrc src) {
    pdl_trigger();  // launched after the split kernel finished: the imp pass may start
    const int h = blockIdx.x, b = blockIdx.y;
    const int L = src.seq_len[b];
    const int grp = src.slot[h / a.hpk];
    // chunks start at the first visible row rounded down to kRowAlign
    const int f0 = int(first_visible(L, a.window) / kRowAlign * kRowAlign);
    const int nc = (L - f0 + a.chunk - 1) / a.chunk;
    const float *vcol = (src.vcol && grp >= 0) ? src.vcol + (int64_t(b) * src.n_live + grp) * HD : nullptr;
    merge_body<HD>(a, b, int64_t(b) * a.n_q + h, h % a.hpk, h, grp, nc, vcol);
}

// Verify merge: grid (n_q, n_seq, K); a.hpk = K * hg partial rows per group,
// output [n_seq][K][n_q][HD].
template <int HD>
__global__ void __launch_bounds__(HD) merge_verify_kernel(MergeArgs a, MergeLayerSrc src, int32_t K, int32_t hg) {
    const int h = blockIdx.x, b = blockIdx.y, k = blockIdx.z;
    const int L = src.seq_len[b];
    const int grp = src.slot[h / hg];
    const int f0 = int(first_visible(verify_len(L, K), a.window) / kRowAlign * kRowAlign);
    const int nc = (L - f0 + a.chunk - 1) / a.chunk;
    const float *vcol = (src.vcol && grp >= 0) ? src.vcol + (int64_t(b) * src.n_live + grp) * HD : nullptr;
    merge_body<HD>(a, b, (int64_t(b) * K + k) * a.n_q + h, k * hg + h % hg, h, grp, nc, vcol);
}

template <int HD>
__global__ void __launch_bounds__(HD) merge_rswa_kernel(MergeArgs a, RswaTable tb) {
    const int h = blockIdx.x, si = blockIdx.y;
    if (si >= tb.n) return;
    const int s = tb.s0 + si;
    const int nc = (tb.prefill_len[si] + a.chunk - 1) / a.chunk +
                   (tb.ring_len[si] + a.chunk - 1) / a.chunk;
    merge_body<HD>(a, s, int64_t(s) * a.n_q + h, 0, h, h, nc, nullptr);
}

// R-SWA verify merge: grid (H, streams of the launch, K); chunk partials of
// the reference rows then one tail partial (ring + drafts) per query.
template <int HD>
__global__ void __launch_bounds__(HD) merge_rswa_verify_kernel(MergeArgs a, RswaTable tb, int32_t K) {
    const int h = blockIdx.x, si = blockIdx.y, i = blockIdx.z;
    if (si >= tb.n) return;
    const int s = tb.s0 + si;
    const int nc = (tb.prefill_len[si] + a.chunk - 1) / a.chunk + 1;
    merge_body<HD>(a, s, (int64_t(s) * K + i) * a.n_q + h, i, h, h, nc, nullptr);
}

// Host launcher for one instance (instantiated per storage mode in its own unit).
template <int HD, int HPK, bool KQ, bool VQ>
cudaError_t launch_split_layer_impl(const SplitArgs &a, const LayerSrc &s, dim3 grid,
                                    cudaStream_t st) {
    using C = SplitCfg<HD, HPK, KQ, VQ>;
    auto kern = (a.window > 0 || a.softcap2 > 0.0f || a.K > 1) ? split_layer_kernel<HD, HPK, KQ, VQ, true>
                                                                : split_layer_kernel<HD, HPK, KQ, VQ, false>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM, st>>>(a, s);
    return launch_status();
}

}  // namespace kvd
