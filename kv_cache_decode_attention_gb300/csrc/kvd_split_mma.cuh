// kvd_split_mma.cuh -- split-KV decode over the q8_2f cache (int8 K and V,
// head_dim 128) on the tensor cores (warp-level mma.sync, f16 in, f32 out).
// The same kernel, in its row-scale mode (ROWK), reads the reference block of
// the R-SWA int8 mirror for a query-batched verify (rswa verify_attention over
// decode_attention_int8): one K scale per row, int8 query codes.
//
// Why tensor cores: with int8 rows a CUDA-core kernel spends ~84 instructions
// per cached row (int8->f32 conversions, hpk x 128 FMAs per pass, warp
// reductions) and is issue-bound far below the HBM roofline at GQA fan-out
// 4..16.  Here both contractions run as f16 MMAs with f32 accumulation; the
// CUDA cores only turn each int8 code into an exact f16 once (a byte splice
// and one HSUB2 per pair), shared by every query head of the group.  (The
// legacy int8 mma.sync path is far slower than f16 on this GPU, so the codes
// go through f16.)
//
// Work split: a persistent grid of one-warp CTAs.  The cached rows of all
// (sequence, live group) units are cut into tiles of 32 rows and laid end to
// end; worker c owns the contiguous tile range [c T / G, (c+1) T / G), so
// every warp streams the same number of tiles whatever the length mix.  A
// worker keeps one online-softmax state per run -- a stretch of its range
// inside one unit and one block of kBlockTiles tiles -- and writes the run's
// (max, sum, accumulator) per head as one partial; a second kernel merges a
// unit's partials by log-sum-exp.  Partial slots need no table: the run of
// worker c starting in block j of unit u sits at slot NB(u) + j + c, where
// NB(u) counts the blocks of the units before u.  (Runs start at block starts
// and worker starts; moving to the next run start adds one to j or to c, so
// slots are distinct.  Where a worker starts exactly on a block start both
// grow and one slot is skipped; that worker marks it empty, so a unit's runs
// and markers fill the slot range from its first run to its last, which the
// workers holding those runs record for the merge.)
//
// Each warp owns a ring of kStages stages (K codes, V codes, K scales, V
// scales of one tile) filled by TMA: 2-D tensor copies with the 128-byte
// swizzle for the codes (conflict-free ldmatrix), 1-D bulk copies for the
// scales, one mbarrier per stage.  Per tile:
//   scores  S[row][h] = 2^-E_h sum_g ks[row][g] K_g . (t1_h + t2_h)_g with
//           M = the tile's rows (two m16 blocks), N = heads, K = channels.
//           K codes are exact in f16; q * kcol * scale * log2(e) * 2^E_h is
//           split into two f16 terms t1 + t2 (22 significant bits, E_h puts
//           the head's largest term near 2^14) whose MMAs chain into one f32
//           accumulator per 32-channel group, so ks[row][g] applies after.
//           Inside a k16 step the channel order is permuted identically in A
//           and B so a lane's four consecutive codes feed its fragment.
//   softmax online per warp in the log2 domain (running max per head).
//   weights w = 2^(S - max) * vs[row] * 2^Ew (Ew puts the tile's largest V
//           scale near 2^14), split into two f16 terms and written
//           transposed ([row][head]) to a 1 KB per-warp buffer.
//   values  out^T = V^T P^T: M = channels (eight m16 blocks, even channels of
//           a 16-channel chunk in rows 0..7, odd ones in rows 8..15, straight
//           from ldmatrix.trans of the V tile), N = heads, K = the tile's
//           rows; the two weight terms chain into fresh f32 accumulators that
//           are folded into the running sum with one IEEE FMA per element
//           (rescaled by the softmax correction and the change of Ew).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "kvd_decode_kernels.cuh"

namespace kvd {

constexpr int kWR = 32;             // rows per tile
constexpr int kBlockTiles = 64;     // tiles per partial block (2048 rows; bounds one f32 fold chain)
constexpr int kStages = 2;          // ring stages per warp
constexpr int kStK = 0;             // K codes [32][128], 128-byte swizzled
constexpr int kStV = 4096;          // V codes [32][128], 128-byte swizzled
constexpr int kStKs = 8192;         // K scales [32][4] f32
constexpr int kStVs = 8704;         // V scales [32] f32
constexpr int kStageBytes = 9216;   // multiple of 1024 (swizzle atom)
constexpr uint32_t kStageTx = 4096 + 4096 + 512 + 128;
constexpr uint32_t kStageTxRow = 4096 + 4096 + 128 + 128;  // one K scale per row

// PACK: groups of at most 4 query heads put both query terms (and both
// weight terms) side by side in the 8 columns of one n8 tile; larger groups
// (up to 8 heads) use the 8 columns for heads and chain the two terms.
template <bool PACK>
struct WarpCfg {
    static constexpr int P_OFF = kStages * kStageBytes;   // P^T [term][32 rows][8 columns] f16
    static constexpr int P_BYTES = PACK ? 512 : 1024;
    static constexpr int BAR_OFF = P_OFF + P_BYTES;
    static constexpr int SMEM = BAR_OFF + kStages * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // room to align the base to 1024
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Order this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (TMA) writes to it.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// D += A(16x16 f16, row) * B(16x8 f16, col), f32 accumulate.  Not volatile:
// it has no side effects, so the compiler may interleave independent chains.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
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

// 2^x by the hardware approximation (relative error a few ulp; results below
// the smallest normal flush to zero, which no weight here needs).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// e with x in [2^(e-1), 2^e) for a positive normal x.
__device__ __forceinline__ int exponent_of(float x) {
    return int((__float_as_uint(x) >> 23) & 0xffu) - 126;
}

// 2^e for -126 <= e <= 127.
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }

// 2^d for |d| <= 252 as the product of two normal powers of two: exact, and
// rounded like ldexpf(1, d) where the result leaves the normal range.
__device__ __forceinline__ float pow2_wide(int d) {
    const int d1 = d >> 1;
    return pow2i(d1) * pow2i(d - d1);
}

struct MmaMaps {
    CUtensorMap kq, vq;
};

struct WarpArgs {
    SplitArgs a;
    int64_t *unit_slots;  // [n_seq * n_live][2]: slot of each unit's first and last run
    int64_t T;            // tiles of all units
    int32_t G;            // workers (grid size), 1 <= G <= T
    int32_t n_seq;
};

// Number of workers whose range starts at or before global tile x.
__device__ __forceinline__ int64_t workers_started(int64_t x, int64_t T, int64_t G) {
    const int64_t c = ((x + 1) * G + T - 1) / T;
    return c < G ? c : G;
}

// Position of one tile in the unit order (sequence-major, live group, tile).
// A unit's tiles start at its first visible row rounded down to a tile (f0).
struct TileCursor {
    int b, gl, tl;   // sequence, live group, tile within the unit
    int Tb, Lb;      // tiles and rows of sequence b
    int f0, lo;      // row of tile 0, first visible row
    int64_t cap;     // region rows of sequence b
    int64_t rbase;   // storage row of the unit's row 0
    int64_t bq;      // partial blocks of the units of sequences before b
};

__device__ __forceinline__ int blocks_of(int tiles) { return (tiles + kBlockTiles - 1) / kBlockTiles; }

// Tiles of a sequence of L rows under a sliding window (0 = none); for a
// verify of K drafts they start at the earliest query's first row.
__host__ __device__ __forceinline__ int64_t tiles_of(int64_t L, int64_t window, int32_t K = 1) {
    const int64_t f0 = first_visible(verify_len(L, K), window) / kWR * kWR;
    return (L - f0 + kWR - 1) / kWR;
}

// Load sequence b's shape into the cursor; false (and an error bit) if its
// length exceeds its capacity.
__device__ __forceinline__ bool cursor_seq(TileCursor &c, const LayerSrc &src, int64_t window, int32_t K,
                                           uint32_t *err) {
    c.cap = src.cap[c.b];
    c.rbase = src.row_base[c.b];
    c.lo = int(first_visible(verify_len(c.Lb, K), window));
    c.f0 = c.lo / kWR * kWR;
    if (int64_t(c.Lb) > c.cap) {
        set_error(err, kErrBounds);
        return false;
    }
    return true;
}

// Advance to the next tile in the global order; false past the last sequence.
__device__ __forceinline__ bool cursor_next(TileCursor &c, const LayerSrc &src, int n_seq, int64_t window,
                                            int32_t K, uint32_t *err) {
    if (++c.tl < c.Tb) return true;
    c.tl = 0;
    if (++c.gl < src.n_live) {
        c.rbase += c.cap;
        return true;
    }
    c.gl = 0;
    c.bq += int64_t(src.n_live) * blocks_of(c.Tb);
    for (;;) {
        if (++c.b >= n_seq) return false;
        c.Lb = src.seq_len[c.b];
        c.Tb = int(tiles_of(c.Lb, window, K));
        if (c.Tb > 0) break;
    }
    return cursor_seq(c, src, window, K, err);
}

// Find global tile x: a warp-wide scan of the sequences' tile counts.
__device__ inline bool cursor_locate(TileCursor &c, int64_t x, const LayerSrc &src, int n_seq, int64_t window,
                                     int32_t K, int lane, uint32_t *err) {
    int64_t tp = 0, bq = 0;  // tiles and blocks of the sequences before `base`
    for (int base = 0; base < n_seq; base += 32) {
        const int i = base + lane;
        const int L = i < n_seq ? src.seq_len[i] : 0;
        const int Tb = int(tiles_of(L, window, K));
        int64_t ut = int64_t(src.n_live) * Tb, ub = int64_t(src.n_live) * blocks_of(Tb);
        // inclusive prefix over the lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t t = __shfl_up_sync(0xffffffffu, ut, off);
            const int64_t bb = __shfl_up_sync(0xffffffffu, ub, off);
            if (lane >= off) ut += t, ub += bb;
        }
        const int64_t tot_t = __shfl_sync(0xffffffffu, ut, 31);
        const int64_t tot_b = __shfl_sync(0xffffffffu, ub, 31);
        if (tp + tot_t > x) {
            // first lane whose inclusive prefix passes x
            const unsigned m = __ballot_sync(0xffffffffu, tp + ut > x);
            const int src_lane = __ffs(m) - 1;
            const int64_t ex_t = __shfl_sync(0xffffffffu, ut, src_lane) -
                                 int64_t(src.n_live) * __shfl_sync(0xffffffffu, Tb, src_lane);
            const int64_t ex_b = __shfl_sync(0xffffffffu, ub, src_lane) -
                                 int64_t(src.n_live) * blocks_of(__shfl_sync(0xffffffffu, Tb, src_lane));
            c.b = base + src_lane;
            c.Lb = __shfl_sync(0xffffffffu, L, src_lane);
            c.Tb = __shfl_sync(0xffffffffu, Tb, src_lane);
            c.bq = bq + ex_b;
            const int64_t r = x - (tp + ex_t);
            c.gl = int(r / c.Tb);
            c.tl = int(r % c.Tb);
            if (!cursor_seq(c, src, window, K, err)) return false;
            c.rbase += int64_t(c.gl) * c.cap;
            return true;
        }
        tp += tot_t;
        bq += tot_b;
    }
    set_error(err, kErrBounds);
    return false;
}

// ROWK: one K scale per row ([rows] f32) instead of one per 32 channels.
template <bool ROWK = false>
__device__ __forceinline__ void issue_tile(const TileCursor &c, const CUtensorMap *kmap,
                                           const CUtensorMap *vmap, const LayerSrc &src, char *stage,
                                           uint64_t *bar) {
    const int64_t row = c.rbase + c.f0 + int64_t(c.tl) * kWR;
    mbar_arrive_expect_tx(bar, ROWK ? kStageTxRow : kStageTx);
    tma_load_2d(stage + kStK, kmap, 0, int(row), bar);
    tma_load_2d(stage + kStV, vmap, 0, int(row), bar);
    if (ROWK) bulk_g2s(stage + kStKs, src.ks + row, 128, bar);
    else bulk_g2s(stage + kStKs, src.ks + row * 4, 512, bar);
    bulk_g2s(stage + kStVs, src.vs + row, 128, bar);
}

// OPT: the call has a window or a softcap; IMP: the call accumulates imp
// (per-row scores are stored).  Both are compiled out of the common path.
// ROWK: the R-SWA int8 mirror's reference block (rswa decode_attention_int8,
// query-batched for verify_attention): one K scale per row, no column field,
// and each query row quantised like a cache row, so the B operand is the
// query's int8 codes (exact in f16, one term) and the score is the exact
// integer dot times the row's K scale times qscale * softmax scale * log2(e).
// The group's a.hpk query rows are the K drafts of one head, read from
// q [stream][draft][head][128] (a.n_q heads); a.K stays 1 (every draft sees
// the whole block).
template <bool PACK, bool OPT, bool IMP, bool ROWK = false>
__global__ void __launch_bounds__(32, 12) split_warp_kernel(WarpArgs wa, LayerSrc src,
                                                        const __grid_constant__ MmaMaps maps) {
    using C = WarpCfg<PACK>;
    extern __shared__ __align__(128) char smem_raw[];
    const SplitArgs &a = wa.a;
    const int lane = threadIdx.x;
    const int gl4 = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix index, row in matrix
    // align to 1024 by offsetting the shared array itself, so every derived
    // pointer stays a known shared-memory pointer
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
        // This worker starts on a block start: the slot just below its first
        // run belongs to no run.  Mark it empty (max -inf) so that every unit's
        // runs fill a contiguous slot range.
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
    int64_t issued = 0;  // tiles issued so far (tile i goes to stage i % kStages)
    bool prod_ok = true;
    {
        const int64_t first = x_end - x_begin < kStages ? x_end - x_begin : int64_t(kStages);
        for (int64_t i = 0; i < first && prod_ok; ++i) {
            if (lane == 0) issue_tile<ROWK>(prod, &maps.kq, &maps.vq, src, sm + (i % kStages) * kStageBytes,
                                            &bar[i % kStages]);
            ++issued;
            if (x_begin + issued < x_end) prod_ok = cursor_next(prod, src, wa.n_seq, a.window, a.K, a.err);
        }
    }

    // Lane-constant shared-memory offsets.  K tile (ldmatrix): row
    // mb*16 + rr + 8*(mi&1), 16-byte chunk 2g + (mi>>1), swizzled by the row's
    // low 3 bits (= rr).  V tile (ldmatrix.trans): row 8*mi + rr, chunk cc.
    const uint32_t k_lane = uint32_t(rr + 8 * (mi & 1)) * 128;
    uint32_t k_chunk[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) k_chunk[g] = uint32_t(((2 * g + (mi >> 1)) ^ rr) << 4);
    const uint32_t v_lane = uint32_t(8 * mi + rr) * 128;
    const uint32_t p_base = smem_addr(sm + C::P_OFF);
    const uint32_t p_ld = p_base + uint32_t(8 * mi + rr) * 16;  // ldmatrix.trans rows of P^T
    const uint32_t p_st = p_base + uint32_t(t4) * 4;              // + row * 16

    // Score columns.  PACK: column n holds term n / 4 of head n % 4, so this
    // lane's columns 2*t4, 2*t4 + 1 are heads hc0 = (2*t4) % 4 and hc0 + 1
    // (the t1 part when t4 < 2, the t2 part otherwise); after the two parts
    // are added, lanes t4 and t4 ^ 2 hold the same scores.  Otherwise columns
    // are heads 2*t4, 2*t4 + 1.
    const int hc0 = PACK ? (2 * t4) & 3 : 2 * t4;
    const bool owner = !PACK || t4 < 2;  // writes scores and partials of its heads
    // B fragments of the query [chunk][term or -][reg]: the column this lane
    // feeds is gl4 (PACK: term gl4 / 4 of head gl4 % 4; else head gl4)
    uint32_t bq[8][(PACK || ROWK) ? 1 : 2][2];
    float qexp[2];
    int q_b = -1, q_gl = -1;

    int64_t x = x_begin, i = 0;  // global tile, worker-local tile count
    bool ok = true;
    while (x < x_end) {
        // ------------------------------------------------ run set-up
        int64_t run_len = x_end - x;
        if (run_len > cur.Tb - cur.tl) run_len = cur.Tb - cur.tl;
        if (run_len > kBlockTiles - cur.tl % kBlockTiles) run_len = kBlockTiles - cur.tl % kBlockTiles;
        const int64_t slot = cur.bq + int64_t(cur.gl) * blocks_of(cur.Tb) + cur.tl / kBlockTiles + c;
        const int64_t unit = int64_t(cur.b) * src.n_live + cur.gl;
        const bool unit_end = cur.tl + run_len == cur.Tb;
        if (cur.tl == 0 && lane == 0) wa.unit_slots[2 * unit] = slot;
        if (cur.b != q_b || cur.gl != q_gl) {
            // q * kcol * scale * log2e * 2^E_h = t1 + t2 (f16), channels
            // 16*chunk + 4*t4 .. + 3 of every chunk
            q_b = cur.b;
            q_gl = cur.gl;
            const int g = src.live[cur.gl];
            if constexpr (ROWK) {
                // draft hb of head g, quantised like a cache row (scale max|x| / 127,
                // 1 for a zero row; IEEE division, round half to even, clamp to
                // +-127): the codes are exact f16 values, the scale joins qexp
                const int hb = PACK ? gl4 & 3 : gl4;
                const float *qr = a.q + ((int64_t(cur.b) * a.hpk + hb) * a.n_q + g) * 128;
                float xq[8][4];
                float mx = 0.0f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float4 qv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (hb < a.hpk) qv = *reinterpret_cast<const float4 *>(qr + 16 * ch + 4 * t4);
                    xq[ch][0] = qv.x, xq[ch][1] = qv.y, xq[ch][2] = qv.z, xq[ch][3] = qv.w;
#pragma unroll
                    for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(xq[ch][j]));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float qs = mx > 0.0f ? __fdiv_rn(mx, 127.0f) : 1.0f;
                const bool empty = PACK && gl4 >= 4;  // the second term's columns stay zero
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float cd[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) cd[j] = float(quant_code_i8(xq[ch][j], qs));
                    bq[ch][0][0] = empty ? 0u : pack_half2(cd[0], cd[1]);
                    bq[ch][0][1] = empty ? 0u : pack_half2(cd[2], cd[3]);
                }
                const float qf = qs * a.qscale;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) qexp[cc] = __shfl_sync(0xffffffffu, qf, (hc0 + cc) * 4);
                __syncwarp();
            } else {
            const float *qg = a.q + (int64_t(cur.b) * a.n_q + int64_t(g) * a.hpk) * 128;
            const float *kc = src.kcol + (int64_t(cur.b) * src.n_live + cur.gl) * 128;
            const int hb = PACK ? gl4 & 3 : gl4;
            float xq[8][4];
            float mx = 0.0f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const int d = 16 * ch + 4 * t4;
                float4 qv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (hb < a.hpk) qv = *reinterpret_cast<const float4 *>(qg + hb * 128 + d);
                const float4 kv = *reinterpret_cast<const float4 *>(kc + d);
                xq[ch][0] = qv.x * kv.x * a.qscale;
                xq[ch][1] = qv.y * kv.y * a.qscale;
                xq[ch][2] = qv.z * kv.z * a.qscale;
                xq[ch][3] = qv.w * kv.w * a.qscale;
#pragma unroll
                for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(xq[ch][j]));
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const int E = mx > 0.0f ? min(14 - exponent_of(mx), 100) : 0;
            const float sc = pow2i(E);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float hi[4], lo[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    hi[j] = xq[ch][j] * sc;
                    lo[j] = hi[j] - __half2float(__float2half_rn(hi[j]));
                }
                if constexpr (PACK) {
                    const bool t2 = gl4 >= 4;
                    bq[ch][0][0] = t2 ? pack_half2(lo[0], lo[1]) : pack_half2(hi[0], hi[1]);
                    bq[ch][0][1] = t2 ? pack_half2(lo[2], lo[3]) : pack_half2(hi[2], hi[3]);
                } else {
                    bq[ch][0][0] = pack_half2(hi[0], hi[1]);
                    bq[ch][0][1] = pack_half2(hi[2], hi[3]);
                    bq[ch][(PACK || ROWK) ? 0 : 1][0] = pack_half2(lo[0], lo[1]);
                    bq[ch][(PACK || ROWK) ? 0 : 1][1] = pack_half2(lo[2], lo[3]);
                }
            }
            // 2^-E of the heads of this lane's score columns, held by the
            // lanes feeding them (gl4 = head)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) qexp[cc] = pow2i(-__shfl_sync(0xffffffffu, E, (hc0 + cc) * 4));
            __syncwarp();
            }
        }
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
        float acc[8][4];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[cc][j] = 0.0f;
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
            const uint32_t kaddr = smem_addr(st + kStK) + k_lane;
            const float *ks_s = reinterpret_cast<const float *>(st + kStKs);
            const float *vs_s = reinterpret_cast<const float *>(st + kStVs);

            // ------------------------------------------------ scores
            float sreg[2][2][2];  // [m block][column][row gl4 / gl4 + 8]
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
                float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float kA[4], kB[4];
                if constexpr (ROWK) {
                    kA[0] = ks_s[mb * 16 + gl4];
                    kB[0] = ks_s[mb * 16 + gl4 + 8];
                } else {
                    const float4 ksA = *reinterpret_cast<const float4 *>(&ks_s[(mb * 16 + gl4) * 4]);
                    const float4 ksB = *reinterpret_cast<const float4 *>(&ks_s[(mb * 16 + gl4 + 8) * 4]);
                    kA[0] = ksA.x, kA[1] = ksA.y, kA[2] = ksA.z, kA[3] = ksA.w;
                    kB[0] = ksB.x, kB[1] = ksB.y, kB[2] = ksB.z, kB[3] = ksB.w;
                }
                float di[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // ROWK: the integer dot over all channels
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t w[4];
                    ldsm_x4(kaddr + mb * 2048 + k_chunk[g], w);
                    const uint32_t u0 = w[0] ^ 0x80808080u, u1 = w[1] ^ 0x80808080u;
                    const uint32_t u2 = w[2] ^ 0x80808080u, u3 = w[3] ^ 0x80808080u;
                    const uint32_t a00 = codes_f16x2<0x4140>(u0), a02 = codes_f16x2<0x4342>(u0);
                    const uint32_t a01 = codes_f16x2<0x4140>(u1), a03 = codes_f16x2<0x4342>(u1);
                    const uint32_t a10 = codes_f16x2<0x4140>(u2), a12 = codes_f16x2<0x4342>(u2);
                    const uint32_t a11 = codes_f16x2<0x4140>(u3), a13 = codes_f16x2<0x4342>(u3);
                    if constexpr (ROWK) {
                        mma_f16(di, a00, a01, a02, a03, bq[2 * g][0][0], bq[2 * g][0][1]);
                        mma_f16(di, a10, a11, a12, a13, bq[2 * g + 1][0][0], bq[2 * g + 1][0][1]);
                    } else {
                        float dg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int tm = 0; tm < (PACK ? 1 : 2); ++tm) {
                            mma_f16(dg, a00, a01, a02, a03, bq[2 * g][tm][0], bq[2 * g][tm][1]);
                            mma_f16(dg, a10, a11, a12, a13, bq[2 * g + 1][tm][0], bq[2 * g + 1][tm][1]);
                        }
                        sacc[0] = fmaf(kA[g], dg[0], sacc[0]);
                        sacc[1] = fmaf(kA[g], dg[1], sacc[1]);
                        sacc[2] = fmaf(kB[g], dg[2], sacc[2]);
                        sacc[3] = fmaf(kB[g], dg[3], sacc[3]);
                    }
                }
                if constexpr (ROWK) {
                    // every partial sum is an integer below 2^24: exact in f32
                    sacc[0] = di[0] * kA[0];
                    sacc[1] = di[1] * kA[0];
                    sacc[2] = di[2] * kB[0];
                    sacc[3] = di[3] * kB[0];
                }
                if constexpr (PACK) {
                    // add the other term's part (columns 2*t4 ^ 4)
#pragma unroll
                    for (int j = 0; j < 4; ++j) sacc[j] += __shfl_xor_sync(0xffffffffu, sacc[j], 2);
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    float x0 = sacc[cc] * qexp[cc], x1 = sacc[2 + cc] * qexp[cc];
                    if (OPT && a.softcap2 > 0.0f) {
                        x0 = softcap_log2(x0, a.softcap2);
                        x1 = softcap_log2(x1, a.softcap2);
                    }
                    sreg[mb][cc][0] = x0;
                    sreg[mb][cc][1] = x1;
                }
            }
            // rows outside [r_lo, n_valid) (a partial last tile, or rows before
            // the window in the first one) drop out; full tiles skip the masks
            const bool full = (!OPT || r_lo <= 0) && n_valid == kWR;
            if (!full) {
#pragma unroll
                for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                    for (int rw = 0; rw < 2; ++rw) {
                        const int r = mb * 16 + gl4 + 8 * rw;
                        if (!(r >= r_lo && r < n_valid)) sreg[mb][0][rw] = sreg[mb][1][rw] = -INFINITY;
                    }
            }
            if (IMP && owner) {
                // per-row log2 scores for the imp pass: [hpk][cap] per unit
                float *sp = a.scores + cur.rbase * a.hpk + row0;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int h = hc0 + cc;
                    if (h < a.hpk) {
                        float *sh = sp + int64_t(h) * cur.cap;
#pragma unroll
                        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                            for (int rw = 0; rw < 2; ++rw) {
                                const int r = mb * 16 + gl4 + 8 * rw;
                                if (r >= r_lo && r < n_valid) sh[r] = sreg[mb][cc][rw];
                            }
                    }
                }
            }

            // ------------------------------------------------ softmax
            float vsr[2][2];
            float vmax = 0.0f;
#pragma unroll
            for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                for (int rw = 0; rw < 2; ++rw) {
                    const int r = mb * 16 + gl4 + 8 * rw;
                    vsr[mb][rw] = full || (r >= r_lo && r < n_valid) ? vs_s[r] : 0.0f;
                    vmax = fmaxf(vmax, vsr[mb][rw]);
                }
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 4));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 8));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 16));
            const int ew = vmax > 0.0f ? min(14 - exponent_of(vmax), 100) : 0;
            const float wsc = pow2i(ew);
            // the change of Ew is an exact power of two (the approximate exp2
            // is not exact even at integers, and these factors compound over a run)
            const float dsc = pow2_wide(ew - ew_prev);
            ew_prev = ew;
            float fa[2];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                float tmx = fmaxf(fmaxf(sreg[0][cc][0], sreg[0][cc][1]), fmaxf(sreg[1][cc][0], sreg[1][cc][1]));
                tmx = fmaxf(tmx, __shfl_xor_sync(0xffffffffu, tmx, 4));
                tmx = fmaxf(tmx, __shfl_xor_sync(0xffffffffu, tmx, 8));
                tmx = fmaxf(tmx, __shfl_xor_sync(0xffffffffu, tmx, 16));
                const float mn = fmaxf(m[cc], tmx);
                // exactly 1 while the maximum holds; 0 before the first tile (m = -inf)
                const float al = mn == m[cc] ? 1.0f : fast_exp2(m[cc] - mn);
                fa[cc] = al * dsc;
                l[cc] *= al;
                m[cc] = mn;
            }
#pragma unroll
            for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                for (int rw = 0; rw < 2; ++rw) {
                    // rows past the tile hold -inf scores and a zero scale
                    const float e0 = fast_exp2(sreg[mb][0][rw] - m[0]);
                    const float e1 = fast_exp2(sreg[mb][1][rw] - m[1]);
                    l[0] += e0;
                    l[1] += e1;
                    const float vw = vsr[mb][rw] * wsc;
                    const float w0 = e0 * vw, w1 = e1 * vw;
                    const uint32_t t1 = pack_half2(w0, w1);
                    const float2 back = __half22float2(*reinterpret_cast<const __half2 *>(&t1));
                    const uint32_t t2 = pack_half2(w0 - back.x, w1 - back.y);
                    const uint32_t row = uint32_t(mb * 16 + gl4 + 8 * rw) * 16;
                    if constexpr (PACK) {
                        sts32(p_st + row, t4 < 2 ? t1 : t2);  // column 2*t4: term t4 / 2
                    } else {
                        sts32(p_st + row, t1);
                        sts32(p_st + 512 + row, t2);
                    }
                }
            __syncwarp();
            uint32_t bp[PACK ? 1 : 2][4];  // P^T fragments [term][b0/b1 of k16 step 0, 1]
#pragma unroll
            for (int tm = 0; tm < (PACK ? 1 : 2); ++tm) ldsm_x4_t(p_ld + uint32_t(tm) * 512, bp[tm]);

            // ------------------------------------------------ values
            const uint32_t vaddr = smem_addr(st + kStV) + v_lane;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t xv[4];
                ldsm_x4_t(vaddr + (uint32_t((cc ^ rr)) << 4), xv);
                uint32_t af[2][4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint32_t lo = xv[2 * kk] ^ 0x80808080u, hi = xv[2 * kk + 1] ^ 0x80808080u;
                    af[kk][0] = codes_f16x2<0x4240>(lo);
                    af[kk][1] = codes_f16x2<0x4341>(lo);
                    af[kk][2] = codes_f16x2<0x4240>(hi);
                    af[kk][3] = codes_f16x2<0x4341>(hi);
                }
                float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int tm = 0; tm < (PACK ? 1 : 2); ++tm)
                        mma_f16(d, af[kk][0], af[kk][1], af[kk][2], af[kk][3], bp[tm][2 * kk], bp[tm][2 * kk + 1]);
                acc[cc][0] = fmaf(acc[cc][0], fa[0], d[0]);
                acc[cc][1] = fmaf(acc[cc][1], fa[1], d[1]);
                acc[cc][2] = fmaf(acc[cc][2], fa[0], d[2]);
                acc[cc][3] = fmaf(acc[cc][3], fa[1], d[3]);
            }
            __syncwarp();  // every lane is done with this stage and the P^T buffer
            // refill this stage with the tile kStages ahead
            if (x_begin + issued < x_end && prod_ok) {
                if (lane == 0) {
                    fence_proxy_async();
                    issue_tile<ROWK>(prod, &maps.kq, &maps.vq, src, st, &bar[stg]);
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
        if constexpr (PACK) {
            // add the t2 columns' sums (lanes t4 ^ 2) to the t1 columns'
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[cc][j] += __shfl_xor_sync(0xffffffffu, acc[cc][j], 2);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            float lv = l[cc];
            lv += __shfl_xor_sync(0xffffffffu, lv, 4);
            lv += __shfl_xor_sync(0xffffffffu, lv, 8);
            lv += __shfl_xor_sync(0xffffffffu, lv, 16);
            const int h = hc0 + cc;
            if (owner && h < a.hpk) {
                if (gl4 == 0) {
                    a.pm[p0 + h] = m[cc];
                    a.pl[p0 + h] = lv;
                }
                float *dst = a.pacc + (p0 + h) * 128 + 2 * gl4;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<float2 *>(dst + 16 * ch) =
                        make_float2(acc[ch][cc] * unscale, acc[ch][2 + cc] * unscale);
            }
        }
    }

    if (!ok) {
        // A copy never completed (or the sequences changed under the launch):
        // record it and give the copies still in flight a bounded chance to
        // land, so none writes into a successor CTA's shared memory.
        if (lane == 0) {
            set_error(a.err, kErrTimeout);
            for (int64_t j = i; j < issued; ++j)
                (void)mbar_wait_bounded(&bar[j % kStages], uint32_t(j / kStages) & 1u, 100000000ull);
        }
    }
}

template <bool PACK>
cudaError_t launch_split_warp(const WarpArgs &wa, const LayerSrc &s, const MmaMaps &maps,
                              cudaStream_t st) {
    using C = WarpCfg<PACK>;
    const bool opt = wa.a.window > 0 || wa.a.softcap2 > 0.0f, imp = wa.a.scores != nullptr;
    auto kern = opt ? (imp ? split_warp_kernel<PACK, true, true> : split_warp_kernel<PACK, true, false>)
                    : (imp ? split_warp_kernel<PACK, false, true> : split_warp_kernel<PACK, false, false>);
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(unsigned(wa.G)), dim3(32), C::SMEM_ALLOC, st, wa, s, maps);
}

// The R-SWA int8 mirror's reference block (no window, softcap or imp there).
template <bool PACK>
cudaError_t launch_split_warp_rowk(const WarpArgs &wa, const LayerSrc &s, const MmaMaps &maps,
                                   cudaStream_t st) {
    using C = WarpCfg<PACK>;
    auto kern = split_warp_kernel<PACK, false, false, true>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(unsigned(wa.G)), dim3(32), C::SMEM_ALLOC, st, wa, s, maps);
}

// Workers of one launch on the current device: SMs x resident CTAs per SM.
template <bool PACK, bool ROWK = false>
int64_t split_warp_workers() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    auto kern = split_warp_kernel<PACK, false, false, ROWK>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             WarpCfg<PACK>::SMEM_ALLOC) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 32, WarpCfg<PACK>::SMEM_ALLOC) !=
            cudaSuccess)
        return 0;
    return int64_t(sms) * occ;
}

}  // namespace kvd
