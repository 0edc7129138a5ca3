// kvd_split_h16_tc.cuh -- the q8_2f decode for groups of 9..16 query heads
// (GQA fan-out up to 16) on the fifth-generation tensor cores: tcgen05.mma
// with its accumulators in tensor memory (TMEM), operands staged by TMA.
//
// Same work split (balanced ranges of 32-row tiles over all (sequence, live
// group) units, one partial per run), partial slots, precision scheme and
// run merge as the warp kernels of kvd_split_mma.cuh; the per-tile work is
// reorganised around 128-row chunks (four TMA tiles of one run), one CTA per
// SM with specialised warps:
//
//   warps 0, 3 producers: walk the worker's tile range in chunk order; warp 0
//              writes one record per chunk (unit, rows, run slot and flags)
//              and loads the K codes and K scales by TMA (one 128-row 2-D
//              swizzled box and one 1-D scale copy) into a three-stage ring
//              that the rows free as soon as the K codes are converted; warp 3
//              loads the V codes and V scales into two buffers per set of row
//              warps (the V codes wait there until the set's previous chunk's
//              values are done); one mbarrier each;
//   warps 1-2  lane 0 of warp 1 + s issues every MMA of row set s (below), in
//              the set's order; warp 1 owns the TMEM allocation:
//                scores  S[row][(t, h)] = K_g[row] . t_{t,h,g}, one f32
//                        accumulator of 32 columns (both query terms t of the
//                        16 heads) per 32-channel group g: A = the chunk's K
//                        codes as exact f16 in TMEM (128 lanes = rows), B = the
//                        query terms in shared memory;
//                values  O_r[ch][(t, h)] = sum_row V[row][ch] w_t[row][h] over
//                        the 32 rows of tile r of the chunk: A = V^T (f16,
//                        shared memory), B = the two weight terms (shared
//                        memory), D = four 128 x 32 f32 accumulators in TMEM
//                        that reuse the score columns (the scores are read
//                        before the weights exist);
//              each group of MMAs is committed to an mbarrier;
//   warps 4-19 two sets of eight row warps; set s takes the chunks i with
//              i % 2 = s, so one set converts and weighs while the other
//              waits for its MMAs.  Thread = TMEM lane = row of the chunk (and
//              channel of the value accumulators): convert the K codes to f16
//              into TMEM and the V codes into shared memory, then the softmax
//              of its row and the weights, then add the chunk's four value
//              accumulators to per-thread f32 sums (IEEE FMAs; the tensor
//              core's own f32 chains stay two MMAs long).
//
// Softmax without a per-chunk maximum.  Each set keeps per head a running
// maximum m that moves only when a row's score exceeds it by more than
// kTcHeadroom (log2 units) or a row's V scale would overflow the f16 weight
// range; such a chunk (and a set's first chunk of every run) takes a
// block-wide maximum and rescales the set's sums as the online softmax does.
// Every other chunk computes w = 2^(s - m) * vs[row] * 2^E straight from its
// own row: the weights stay below 2^15 and keep 22 significant bits in two
// f16 terms, as in the warp kernels.  E (per set and run segment) puts the
// largest V scale seen near 2^(14 - kTcHeadroom).  When both sets hold part
// of a run, the set with the run's second-to-last chunk hands its (max, sum,
// accumulator) to the other through shared memory, which combines them by
// log-sum-exp and writes the run's partial.
//
// Every wait is bounded (2 s), polls a CTA-wide abort flag, and on failure
// sets the device error word; the roles then drain their copies and MMAs in
// flight (bounded again) and free the TMEM before the CTA exits.
#pragma once

#include "kvd_split_mma.cuh"

namespace kvd {

constexpr int kTcSub = 4;                                  // TMA tiles (32 rows) per chunk
constexpr int kTcRows = kTcSub * kWR;                      // 128 rows per chunk = TMEM lanes
constexpr int kTcStages = 3;                               // stages of the K ring (codes + scales)
constexpr int kTcKStage = kTcSub * 4096 + kTcSub * 512;   // 18432: K codes [4][32][128] swizzled, K scales [4][32][4]
constexpr int kTcVBuf = kTcSub * 4096;                     // V codes of a chunk [4][32][128] swizzled
constexpr int kTcMeta = 8;                                 // chunk records in flight
constexpr int kTcWarps = 20;                               // 2 producers, 2 MMA issuers, 2 x 8 row warps
constexpr int kTcSetThreads = 256;                         // row threads of a set
constexpr float kTcHeadroom = 8.0f;                        // log2 growth allowed before a rebase
constexpr uint32_t kTcCols = 512;                          // TMEM columns allocated (the whole SM)
// TMEM columns per set s: K f16 [64] at 64 s, scores [128] at 128 + 128 s, value accumulators
// [2][32] at 384 + 64 s
constexpr uint32_t kTmK = 0, kTmS = 128, kTmO = 384;

struct TcCfg {
    static constexpr int VR_OFF = kTcStages * kTcKStage;       // V codes [set][2][16 KB]
    static constexpr int VS_OFF = VR_OFF + 4 * kTcVBuf;        // V scales [set][2][128] f32
    static constexpr int V16_OFF = VS_OFF + 4 * 512;           // V^T f16 [set][32 KB]
    static constexpr int P_OFF = V16_OFF + 2 * 32768;          // weights f16 [set][8 KB]
    static constexpr int Q_OFF = P_OFF + 2 * 8192;             // query terms f16 [set][8 KB]
    static constexpr int X_OFF = Q_OFF + 2 * 8192;             // run hand-over: acc [16][128], m [16], l [16]
    static constexpr int META_OFF = X_OFF + 16 * 128 * 4 + 2 * 16 * 4;  // chunk records [kTcMeta][64]
    static constexpr int QEXP_OFF = META_OFF + kTcMeta * 64;   // 2^-E_h [set][16]
    static constexpr int RED_OFF = QEXP_OFF + 2 * 16 * 4;      // reduction scratch [set][role][4][12]
    static constexpr int BAR_OFF = RED_OFF + 2 * 2 * 4 * 12 * 4;  // mbarriers
    static constexpr int NBAR = 2 * kTcStages + 8 + 12;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;        // TMEM base, abort flag, set failure flags
    static constexpr int SMEM = MISC_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
};
static_assert(TcCfg::SMEM_ALLOC <= 227 * 1024, "shared memory");

// One chunk of a worker's range, written by the producer before its TMA.
struct TcChunk {
    int64_t rbase;    // storage row of the unit's row 0
    int64_t cap;      // rows of the unit's region (stride of the imp scores)
    int64_t slot;     // partial slot of the chunk's run
    int32_t b, gl;    // sequence, live group
    int32_t row0;     // unit row of the chunk's row 0
    int32_t Lb, lo;   // rows of the sequence, first visible row
    int32_t nsub;     // tiles of the chunk (rows of later tiles belong to no run here)
    int32_t flags;    // kTc* below
    int32_t xseq;     // hand-over number within the worker (kTcExport / kTcImport)
    int32_t pad;
};
static_assert(sizeof(TcChunk) <= 64, "chunk record");
// kTcSetStart: the set's first chunk of the run (fresh state); kTcExport: the
// set's last chunk of a run the other set finishes (hand its state over);
// kTcEmit: the run's last chunk (write the partial, after taking the other
// set's state when kTcImport); kTcLast: the worker's last chunk.
constexpr int32_t kTcSetStart = 1, kTcExport = 2, kTcEmit = 4, kTcImport = 8, kTcLast = 16;

// ------------------------------------------------------------ tcgen05 PTX

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: lbo / sbo = byte strides between
// 8 x 16-byte core matrices adjacent along K / along M or N.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: f16 A and B, f32 D, M x N, A and B
// K-major (0) or M/N-major (1).
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) | (uint32_t(N >> 3) << 17) |
           (uint32_t(M >> 4) << 24);
}

// D (+)= A B with A in TMEM.
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// D (+)= A B with A in shared memory.
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_pin8(uint32_t (&r)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) asm volatile("" : "+r"(r[k]));
}

// After tmem_wait_ld: tie the loaded registers to a point after the wait, so
// no use of them is scheduled before it.
__device__ __forceinline__ void tmem_pin(uint32_t (&r)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) asm volatile("" : "+r"(r[k]));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barriers of one set's 256 row threads: id 1 + 2 set (sync), 2 + 2 set (reduction).
__device__ __forceinline__ void set_sync(int set) { asm volatile("bar.sync %0, 256;" ::"r"(1 + 2 * set) : "memory"); }
__device__ __forceinline__ bool set_any(int set, bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred q, %2, 256, q;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(p)), "r"(2 + 2 * set)
        : "memory");
    return r != 0;
}

// mbarrier wait bounded in time that also gives up once another role has
// aborted (the flag in shared memory).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, const volatile int *abort_flag) {
    // the thread sleeps in the barrier (up to the hint) instead of spinning,
    // which leaves the issue slots to the warps with work; the clock and the
    // abort flag are looked at every 16 tries only
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((n & 15u) == 0 && (*abort_flag || global_ns() - t0 > 2000000000ull)) return false;
    }
}

// tc_wait with one outcome for the whole warp (what follows is warp-collective).
__device__ __forceinline__ bool tc_wait_warp(uint64_t *bar, uint32_t parity, const volatile int *abort_flag) {
    return __all_sync(0xffffffffu, tc_wait(bar, parity, abort_flag));
}

// A chunk (128 storage rows from `row`, the first nsub * 32 of them in the
// run) in two copies per side: the codes as one 128-row box (rows past the
// run are loaded too and masked; rows past the buffer read as zeros), the
// scales of the run's rows as one bulk copy.
__device__ __forceinline__ void issue_k_chunk(int64_t row, int nsub, const CUtensorMap *kmap, const LayerSrc &src,
                                              char *kst, uint64_t *bar) {
    mbar_arrive_expect_tx(bar, uint32_t(kTcRows * 128 + nsub * 512));
    tma_load_2d(kst, kmap, 0, int(row), bar);
    bulk_g2s(kst + kTcSub * 4096, src.ks + row * 4, uint32_t(nsub * 512), bar);
}
__device__ __forceinline__ void issue_v_chunk(int64_t row, int nsub, const CUtensorMap *vmap, const LayerSrc &src,
                                              char *vbuf, char *vsb, uint64_t *bar) {
    mbar_arrive_expect_tx(bar, uint32_t(kTcRows * 128 + nsub * 128));
    tma_load_2d(vbuf, vmap, 0, int(row), bar);
    bulk_g2s(vsb, src.vs + row, uint32_t(nsub * 128), bar);
}

// Four int8 codes (one word) -> two f16x2 words, exact.
__device__ __forceinline__ void codes4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    w ^= 0x80808080u;
    lo = codes_f16x2<0x4140>(w);
    hi = codes_f16x2<0x4342>(w);
}

// OPT: window / softcap / verify limits; IMP: per-row scores stored for the imp pass.
template <bool OPT, bool IMP>
__global__ void __launch_bounds__(kTcWarps * 32, 1) split_h16_tc_kernel(WarpArgs wa, LayerSrc src,
                                                                         const __grid_constant__ MmaMaps maps) {
    using C = TcCfg;
    extern __shared__ __align__(128) char smem_raw[];
    char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const SplitArgs &a = wa.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    TcChunk *meta = reinterpret_cast<TcChunk *>(sm + C::META_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::BAR_OFF);
    // K ring: full / empty per stage; V buffers: vrfull / vrempty [set][2]
    uint64_t *full = bars, *empty = bars + kTcStages, *vrfull = bars + 2 * kTcStages, *vrempty = vrfull + 4;
    // per set s: kfull[s] (K in TMEM), sfull[s] (scores), vfull[s] (V^T), pfull[s]
    // (weights), ofull[s] (value accumulators); xfull / xempty: the run hand-over
    uint64_t *kfull = bars + 2 * kTcStages + 8, *sfull = kfull + 2, *vfull = kfull + 4, *pfull = kfull + 6,
             *ofull = kfull + 8, *xfull = kfull + 10, *xempty = kfull + 11;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::MISC_OFF + 4);
    volatile int *set_fail = reinterpret_cast<volatile int *>(sm + C::MISC_OFF + 8);  // [2]

    const int64_t T = wa.T, G = wa.G, c = blockIdx.x;
    const int64_t x_begin = c * T / G, x_end = (c + 1) * T / G;
    if (threadIdx.x == 0) {
        // full: the producer's expect-tx; sfull / ofull: one MMA commit; kfull /
        // vfull: a set's K / V warps; empty, pfull, xfull, xempty: a whole set
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTcSetThreads);
        }
        for (int v = 0; v < 4; ++v) {
            mbar_init(&vrfull[v], 1);
            mbar_init(&vrempty[v], kTcSetThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&kfull[b], kTcRows);
            mbar_init(&sfull[b], 1);
            mbar_init(&vfull[b], kTcRows);
            mbar_init(&pfull[b], kTcSetThreads);
            mbar_init(&ofull[b], 1);
        }
        mbar_init(xfull, kTcSetThreads);
        mbar_init(xempty, kTcSetThreads);
        *abort_flag = 0;
        set_fail[0] = 0;
        set_fail[1] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTcCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // launched as a dependent of the kernel before (the append of a decode
    // step): wait for it, then let the run merge be scheduled
    pdl_wait();
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (x_begin < x_end) {
        if (warp == 0 || warp == 3) {
            // ---------------------------------------------------- producers
            // warp 0 loads the K codes and scales into the ring and writes the
            // chunk records (and the unit slot table); warp 3 loads the V codes
            // and scales into the sets' buffers.  Each walks the whole range in
            // chunk order (so no wait runs more than one phase ahead); lane 0
            // issues.
            const bool kside = warp == 0;
            TileCursor cur;
            bool ok = cursor_locate(cur, x_begin, src, wa.n_seq, a.window, a.K, lane, a.err);
            if (kside && ok && cur.tl % kBlockTiles == 0) {
                // the slot just below this worker's first run belongs to no run
                const int64_t gap = cur.bq + int64_t(cur.gl) * blocks_of(cur.Tb) + cur.tl / kBlockTiles + c - 1;
                if (gap >= 0 && lane < a.hpk) {
                    a.pm[gap * a.hpk + lane] = -INFINITY;
                    a.pl[gap * a.hpk + lane] = 0.0f;
                }
            }
            if (lane == 0) {
                int64_t x = x_begin, i = 0;
                int32_t xseq = 0;
                while (ok && x < x_end) {
                    int64_t run_len = x_end - x;
                    if (run_len > cur.Tb - cur.tl) run_len = cur.Tb - cur.tl;
                    if (run_len > kBlockTiles - cur.tl % kBlockTiles) run_len = kBlockTiles - cur.tl % kBlockTiles;
                    const int64_t slot = cur.bq + int64_t(cur.gl) * blocks_of(cur.Tb) + cur.tl / kBlockTiles + c;
                    const int64_t unit = int64_t(cur.b) * src.n_live + cur.gl;
                    const bool unit_end = cur.tl + run_len == cur.Tb;
                    if (kside && cur.tl == 0) wa.unit_slots[2 * unit] = slot;
                    const int n_ch = int((run_len + kTcSub - 1) / kTcSub);
                    const int32_t xs = xseq;
                    if (n_ch >= 2) ++xseq;
                    for (int kc = 0; kc < n_ch && ok; ++kc, ++i) {
                        const int64_t k = int64_t(kc) * kTcSub;
                        const int nsub = int(run_len - k < kTcSub ? run_len - k : kTcSub);
                        const int64_t row = cur.rbase + cur.f0 + int64_t(cur.tl) * kWR;
                        if (kside) {
                            const int s = int(i % kTcStages);
                            if (i >= kTcStages && !tc_wait(&empty[s], uint32_t(i / kTcStages + 1) & 1u, abort_flag)) {
                                ok = false;
                                break;
                            }
                            TcChunk &m = meta[i % kTcMeta];
                            m.rbase = cur.rbase;
                            m.cap = cur.cap;
                            m.slot = slot;
                            m.b = cur.b;
                            m.gl = cur.gl;
                            m.row0 = cur.f0 + cur.tl * kWR;
                            m.Lb = cur.Lb;
                            m.lo = cur.lo;
                            m.nsub = nsub;
                            m.flags = (kc <= 1 ? kTcSetStart : 0) | (n_ch >= 2 && kc == n_ch - 2 ? kTcExport : 0) |
                                      (kc == n_ch - 1 ? kTcEmit : 0) | (n_ch >= 2 && kc == n_ch - 1 ? kTcImport : 0) |
                                      (x + nsub >= x_end ? kTcLast : 0);
                            m.xseq = xs;
                            if (unit_end && kc == n_ch - 1) wa.unit_slots[2 * unit + 1] = slot;
                            issue_k_chunk(row, nsub, &maps.kq, src, sm + s * kTcKStage, &full[s]);
                        } else {
                            // the set's V buffer of chunk i: free once the set has
                            // converted the V codes of chunk i - 4
                            const int vb = int(i & 1) * 2 + int((i >> 1) & 1);
                            if (i >= 4 && !tc_wait(&vrempty[vb], uint32_t((i >> 2) + 1) & 1u, abort_flag)) {
                                ok = false;
                                break;
                            }
                            issue_v_chunk(row, nsub, &maps.vq, src, sm + C::VR_OFF + vb * kTcVBuf, sm + C::VS_OFF + vb * 512,
                                          &vrfull[vb]);
                        }
                        for (int j = 0; j < nsub; ++j) {
                            ++x;
                            if (x < x_end && !cursor_next(cur, src, wa.n_seq, a.window, a.K, a.err)) {
                                ok = false;
                                break;
                            }
                        }
                    }
                }
                // one record past the last chunk tells the set waiting on it to stop
                if (ok && kside) {
                    const int s = int(i % kTcStages);
                    if (i >= kTcStages && !tc_wait(&empty[s], uint32_t(i / kTcStages + 1) & 1u, abort_flag)) ok = false;
                    if (ok) {
                        meta[i % kTcMeta].flags = kTcLast | kTcEmit | kTcExport | kTcImport | kTcSetStart;
                        meta[i % kTcMeta].nsub = -1;
                        mbar_arrive(&full[s]);
                    }
                }
                if (!ok) {
                    set_error(a.err, kErrTimeout);
                    *abort_flag = 1;
                    // copies in flight land before the CTA leaves
                    if (kside) {
                        for (int64_t j = i > kTcStages ? i - kTcStages : 0; j < i; ++j)
                            (void)mbar_wait_bounded(&full[j % kTcStages], uint32_t(j / kTcStages) & 1u, 100000000ull);
                    } else {
                        for (int64_t j = i > 4 ? i - 4 : 0; j < i; ++j)
                            (void)mbar_wait_bounded(&vrfull[int(j & 1) * 2 + int((j >> 1) & 1)], uint32_t(j >> 2) & 1u,
                                                    100000000ull);
                    }
                }
            }
            __syncwarp();
        } else if (warp <= 2) {
            // ---------------------------------------------------- MMA issuers
            // warp 1 + s serves row set s, in the set's own order: scores once
            // its K codes are in TMEM, values once its V^T and weights are in
            if (lane == 0) {
                const int set = warp - 1;
                const uint32_t id_v = umma_idesc(128, 32, 1, 1), id_s = umma_idesc(128, 32, 0, 0);
                const uint32_t qb = smem_addr(sm + C::Q_OFF) + 8192u * set;
                const uint32_t vb = smem_addr(sm + C::V16_OFF) + 32768u * set;
                const uint32_t pb = smem_addr(sm + C::P_OFF) + 8192u * set;
                const uint32_t kt = tmem + kTmK + 64u * set, sd = tmem + kTmS + 128u * set,
                               od = tmem + kTmO + 64u * set;
                uint64_t *last_bar = nullptr;
                uint32_t last_par = 0;
                bool ok = true;
                for (int64_t i = set;; i += 2) {
                    const uint32_t par = uint32_t(i >> 1) & 1u;
                    if (!tc_wait(&kfull[set], par, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const TcChunk &m = meta[i % kTcMeta];
                    if (m.nsub < 0) break;  // the set reached the record past the last chunk
                    const bool last = (m.flags & kTcLast) != 0;
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            umma_ts(sd + uint32_t(32 * g), kt + uint32_t(16 * g + 8 * j),
                                    umma_desc(qb + uint32_t(4 * g + 2 * j) * 128u, 128, 2048), id_s, j ? 1u : 0u);
                    umma_commit(&sfull[set]);
                    last_bar = &sfull[set];
                    last_par = par;
                    if (!tc_wait(&vfull[set], par, abort_flag) || !tc_wait(&pfull[set], par, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // one accumulator per 64 rows of the chunk (four-MMA f32 chains)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t k8 = uint32_t(2 * (4 * hh + kk));
                            umma_ss(od + uint32_t(32 * hh), umma_desc(vb + k8 * 128u, 128, 2048),
                                    umma_desc(pb + k8 * 128u, 128, 2048), id_v, kk ? 1u : 0u);
                        }
                    umma_commit(&ofull[set]);
                    last_bar = &ofull[set];
                    if (last) break;
                }
                if (!ok) {
                    set_error(a.err, kErrTimeout);
                    *abort_flag = 1;
                }
                // every MMA issued has completed before the TMEM is freed
                if (last_bar != nullptr) (void)mbar_wait_bounded(last_bar, last_par, 100000000ull);
            }
            __syncwarp();
        } else {
            // ---------------------------------------------------- row warps
            // set s (8 warps) takes the chunks i with i % 2 == s; per TMEM lane
            // quarter one K warp (K codes, heads 0-7) and one V warp (V codes,
            // heads 8-15) share the quarter's 32 rows
            const int set = (warp - 4) >> 3;
            const int role = ((warp - 4) >> 2) & 1;
            const int hb = 8 * role;                 // this warp's first head
            const int q = warp & 3;                  // TMEM lane quarter
            const int rt = 32 * q + lane;            // row of the chunk = TMEM lane = channel
            const uint32_t tl = tmem + (uint32_t(32 * q) << 16);
            const uint32_t kt = tl + kTmK + 64u * set, so = tl + kTmS + 128u * set, oo = tl + kTmO + 64u * set;
            const int st_sub = rt >> 5, rr = lane;   // tile of the chunk, row in the tile
            char *v16 = sm + C::V16_OFF + set * 32768;
            char *pbuf = sm + C::P_OFF + set * 8192;
            char *qb = sm + C::Q_OFF + set * 8192;
            float *qexp = reinterpret_cast<float *>(sm + C::QEXP_OFF) + set * 16;
            float *red = reinterpret_cast<float *>(sm + C::RED_OFF) + (set * 2 + role) * 48;  // [4][12]
            float *xacc = reinterpret_cast<float *>(sm + C::X_OFF), *xm = xacc + 16 * 128, *xl = xm + 16;
            bool fail = false;

            // query terms of a unit (K warps): thread -> head h = rt / 8, channels
            // 16 (rt % 8) .. + 15; B of the scores, K-major: (n = 16 t + h, channel
            // c) at (n/8)*2048 + (c/8)*128 + (n%8)*16 + (c%8)*2
            auto prep_query = [&](const TcChunk &m) {
                const int h = rt >> 3, cb = rt & 7;
                const int g = src.live[m.gl];
                const int hg = a.K > 1 ? a.hg : a.hpk;
                const float *qg = a.q + (int64_t(m.b) * a.K * a.n_q + int64_t(g) * hg) * 128;
                const float *qrow = qg + (int64_t(h / hg) * a.n_q + h % hg) * 128 + 16 * cb;
                const float *kc = src.kcol + (int64_t(m.b) * src.n_live + m.gl) * 128 + 16 * cb;
                float x[16];
                float mx = 0.0f;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 kv = *reinterpret_cast<const float4 *>(kc + 4 * k4);
                    float4 qv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (h < a.hpk) qv = *reinterpret_cast<const float4 *>(qrow + 4 * k4);
                    x[4 * k4 + 0] = qv.x * kv.x * a.qscale;
                    x[4 * k4 + 1] = qv.y * kv.y * a.qscale;
                    x[4 * k4 + 2] = qv.z * kv.z * a.qscale;
                    x[4 * k4 + 3] = qv.w * kv.w * a.qscale;
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) mx = fmaxf(mx, fabsf(x[k]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                const int E = mx > 0.0f ? min(14 - exponent_of(mx), 100) : 0;
                const float sc = pow2i(E);
                uint32_t t1[8], t2[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float a0 = x[2 * k] * sc, a1 = x[2 * k + 1] * sc;
                    t1[k] = pack_half2(a0, a1);
                    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&t1[k]));
                    t2[k] = pack_half2(a0 - b.x, a1 - b.y);
                }
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t *w = t ? &t2[4 * half] : &t1[4 * half];
                        *reinterpret_cast<uint4 *>(qb + (2 * t + (h >> 3)) * 2048 + (2 * cb + half) * 128 + (h & 7) * 16) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                if (cb == 0) qexp[h] = pow2i(-E);
            };
            // K codes of row rt -> f16 into TMEM (64 columns: channels 2j, 2j + 1 in column j)
            auto convert_k = [&](int s) {
                const char *krow = sm + s * kTcKStage + st_sub * 4096 + rr * 128;
#pragma unroll 1
                for (int jj = 0; jj < 4; ++jj) {
                    uint32_t w[16];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int j = 2 * jj + h2;
                        const uint4 u = *reinterpret_cast<const uint4 *>(krow + ((j ^ (rr & 7)) << 4));
                        codes4(u.x, w[8 * h2 + 0], w[8 * h2 + 1]);
                        codes4(u.y, w[8 * h2 + 2], w[8 * h2 + 3]);
                        codes4(u.z, w[8 * h2 + 4], w[8 * h2 + 5]);
                        codes4(u.w, w[8 * h2 + 6], w[8 * h2 + 7]);
                    }
                    tmem_st16(kt + uint32_t(16 * jj), w);
                }
                tmem_wait_st();
            };
            // V codes of row rt -> f16 V^T (A of the values, M/N-major, no swizzle):
            // (channel c, row r) at (c/8)*2048 + r*16 + (c%8)*2
            auto convert_v = [&](int vb) {
                const char *vrow = sm + C::VR_OFF + vb * kTcVBuf + st_sub * 4096 + rr * 128;
                char *dst = v16 + rt * 16;
#pragma unroll 2
                for (int j = 0; j < 8; ++j) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(vrow + ((j ^ (rr & 7)) << 4));
                    uint32_t w[8];
                    codes4(u.x, w[0], w[1]);
                    codes4(u.y, w[2], w[3]);
                    codes4(u.z, w[4], w[5]);
                    codes4(u.w, w[6], w[7]);
                    *reinterpret_cast<uint4 *>(dst + (2 * j) * 2048) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(dst + (2 * j + 1) * 2048) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            };
            // sums over the set's 128 rows, per head of this warp, in every thread
            auto rows_sum = [&](const float (&v)[8], float (&out)[8]) {
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    float t = v[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
                    out[h] = t;
                }
                if (lane == 0)
#pragma unroll
                    for (int h = 0; h < 8; ++h) red[q * 12 + h] = out[h];
                set_sync(set);
#pragma unroll
                for (int h = 0; h < 8; ++h) out[h] = (red[h] + red[12 + h]) + (red[24 + h] + red[36 + h]);
                set_sync(set);
            };

            float m_run[8], l_part[8], acc[8];
            float qx[8];         // 2^-E_h of this warp's heads, for the unit of the chunk in the softmax
            bool q_new = false;  // a new unit came in: reload qx at the next softmax
            int E = 0;
            int pb = -1, pgl = -1;
            float ksr[4] = {0.0f, 0.0f, 0.0f, 0.0f}, vsr = 0.0f;  // this row's scales, chunk in the softmax

            auto load_scales = [&](int s, int vb) {
                const float4 k4 =
                    *reinterpret_cast<const float4 *>(sm + s * kTcKStage + kTcSub * 4096 + st_sub * 512 + rr * 16);
                ksr[0] = k4.x;
                ksr[1] = k4.y;
                ksr[2] = k4.z;
                ksr[3] = k4.w;
                vsr = *reinterpret_cast<const float *>(sm + C::VS_OFF + vb * 512 + st_sub * 128 + rr * 4);
            };
            // chunk i in (both roles): its record and, for a new unit, the query
            // terms; both roles take the row's scales, the K warps convert its K
            // codes to TMEM, and the K stage is free.  False at the record past
            // the worker's last chunk (the K warps release the set's MMA issuer).
            // After a failed wait the record may be stale: only shared memory and
            // TMEM are touched until the set agrees to stop.
            auto stage_in = [&](int64_t i, TcChunk &m) -> bool {
                const int s = int(i % kTcStages), vb = 2 * set + int((i >> 1) & 1);
                const bool in_ok = tc_wait_warp(&full[s], uint32_t(i / kTcStages) & 1u, abort_flag);
                fail = fail || !in_ok;
                m = meta[i % kTcMeta];
                if (m.nsub < 0) {
                    if (role == 0) mbar_arrive(&kfull[set]);
                    return false;
                }
                const bool new_unit = m.b != pb || m.gl != pgl;
                if (new_unit) {
                    // the set's last score MMA has completed: the query buffer is free
                    if (role == 0 && !fail) prep_query(m);
                    pb = m.b;
                    pgl = m.gl;
                    q_new = true;
                    set_sync(set);  // every 2^-E_h is in
                }
                const bool v_ok = tc_wait_warp(&vrfull[vb], uint32_t(i >> 2) & 1u, abort_flag);
                fail = fail || !v_ok;
                load_scales(s, vb);
                if (role == 0) {
                    convert_k(s);
                    tc_fence_before();
                    if (new_unit) fence_proxy_async();
                    mbar_arrive(&kfull[set]);
                    mbar_arrive(&vrempty[vb]);  // (the V warps arrive after converting)
                }
                mbar_arrive(&empty[s]);
                return true;
            };
            // chunk i's V codes to V^T (V warps); their buffer is free after
            auto stage_v = [&](int64_t i) {
                if (role == 0) return;
                const int vb = 2 * set + int((i >> 1) & 1);
                convert_v(vb);
                mbar_arrive(&vrempty[vb]);
                fence_proxy_async();
                mbar_arrive(&vfull[set]);
            };

            TcChunk mi;
            bool have = stage_in(set, mi);
            if (have) stage_v(set);
            for (int64_t i = set; have; i += 2) {
                // ---- scores of this warp's heads: s[h] = 2^-E_h sum_g ks[g] (S[g][t1, h] + S[g][t2, h])
                const bool s_ok = tc_wait_warp(&sfull[set], uint32_t(i >> 1) & 1u, abort_flag);
                fail = fail || !s_ok;
                const int u = mi.row0 + rt;  // unit row of this thread's row
                bool valid = st_sub < mi.nsub && u < mi.Lb;
                if (OPT) valid = valid && u >= mi.lo;
                float sc[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) sc[h] = 0.0f;
                if (s_ok) {
                    tc_fence_after();
                    uint32_t d[4][2][8];  // [group][term][head]
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int t = 0; t < 2; ++t) tmem_ld8(so + uint32_t(32 * g + 16 * t + hb), d[g][t]);
                    tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int t = 0; t < 2; ++t) tmem_pin8(d[g][t]);
                    tc_fence_before();
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            sc[h] = fmaf(ksr[g], __uint_as_float(d[g][0][h]) + __uint_as_float(d[g][1][h]), sc[h]);
                }
                if (q_new) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) qx[h] = qexp[hb + h];
                    q_new = false;
                }
#pragma unroll
                for (int h = 0; h < 8; ++h) sc[h] *= qx[h];
                if (OPT && a.softcap2 > 0.0f) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) sc[h] = softcap_log2(sc[h], a.softcap2);
                }
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    bool vh = valid && s_ok;
                    if (OPT && a.K > 1) {
                        const int upto = mi.Lb - (a.K - 1 - (hb + h) / a.hg);
                        vh = vh && u < upto && u >= int(first_visible(upto, a.window));
                    }
                    if (!vh) sc[h] = -INFINITY;
                }
                if (IMP && valid && s_ok && !fail) {
                    float *sp = a.scores + mi.rbase * a.hpk + u;
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        if (hb + h < a.hpk) sp[int64_t(hb + h) * mi.cap] = sc[h];
                }

                // ---- the set's first chunk of a run: fresh state
                if (mi.flags & kTcSetStart) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        m_run[h] = -INFINITY;
                        l_part[h] = 0.0f;
                        acc[h] = 0.0f;
                    }
                    E = 0;
                }
                // ---- does this chunk move a maximum or the weight exponent?
                const float vsv = valid ? vsr : 0.0f;
                bool need = (mi.flags & kTcSetStart) != 0;
#pragma unroll
                for (int h = 0; h < 8; ++h) need = need || (sc[h] > m_run[h] + kTcHeadroom);
                need = need || (vsv * pow2i(E) >= pow2i(15 - int(kTcHeadroom)));
                // one barrier: whether any row needs the maxima, and whether any
                // thread of the set failed (the flag is written before it, read after)
                const bool fl = fail || *abort_flag;
                if (fl) set_fail[set] = 1;
                const bool any = set_any(set, need || fl);
                if (set_fail[set]) {
                    fail = true;
                    break;
                }
                if (any) {
                    // block maxima of the chunk's scores (this warp's heads) and V scales
                    float mt[8];
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        float v = sc[h];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                        mt[h] = v;
                    }
                    float vm = vsv;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                    if (lane == 0) {
#pragma unroll
                        for (int h = 0; h < 8; ++h) red[q * 12 + h] = mt[h];
                        red[q * 12 + 8] = vm;
                    }
                    set_sync(set);
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        mt[h] = fmaxf(fmaxf(red[h], red[12 + h]), fmaxf(red[24 + h], red[36 + h]));
                    vm = fmaxf(fmaxf(red[8], red[20]), fmaxf(red[32], red[44]));
                    set_sync(set);
                    // the warp's sums so far move to the new maxima
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float mn = fmaxf(m_run[h], mt[h]);
                        const float alpha = mn == m_run[h] ? 1.0f : fast_exp2(m_run[h] - mn);
                        m_run[h] = mn;
                        l_part[h] *= alpha;
                        acc[h] *= alpha;
                    }
                    const int e_new = vm > 0.0f ? min(14 - int(kTcHeadroom) - exponent_of(vm), 100) : E;
                    E = (mi.flags & kTcSetStart) ? e_new : min(E, e_new);
                }
                // ---- weights w = 2^(s - m) vs 2^E as two f16 terms -> P (B of the
                // values, M/N-major: (row, n = 16 t + h) at (n/8)*2048 + row*16 + (n%8)*2)
                {
                    const float vse = vsv * pow2i(E);
                    uint32_t w1[4], w2[4];
#pragma unroll
                    for (int h = 0; h < 8; h += 2) {
                        const float ma = m_run[h] == -INFINITY ? 0.0f : m_run[h];
                        const float mb = m_run[h + 1] == -INFINITY ? 0.0f : m_run[h + 1];
                        const float pa = fast_exp2(sc[h] - ma), pbv = fast_exp2(sc[h + 1] - mb);
                        l_part[h] += pa;
                        l_part[h + 1] += pbv;
                        const float wa_ = pa * vse, wb_ = pbv * vse;
                        w1[h >> 1] = pack_half2(wa_, wb_);
                        const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w1[h >> 1]));
                        w2[h >> 1] = pack_half2(wa_ - t.x, wb_ - t.y);
                    }
                    char *pd = pbuf + role * 2048 + rt * 16;
                    *reinterpret_cast<uint4 *>(pd) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<uint4 *>(pd + 4096) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                }
                fence_proxy_async();
                mbar_arrive(&pfull[set]);

                // ---- the set's next chunk comes in while the values of chunk i run
                TcChunk mn;
                const bool next = (mi.flags & kTcLast) == 0 && stage_in(i + 2, mn);

                // ---- the chunk's two value accumulators -> acc (row order)
                const bool o_ok = tc_wait_warp(&ofull[set], uint32_t(i >> 1) & 1u, abort_flag);
                fail = fail || !o_ok;
                if (o_ok) {
                    tc_fence_after();
                    uint32_t o[2][2][8];  // [64-row half][term][head]
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int t = 0; t < 2; ++t) tmem_ld8(oo + uint32_t(32 * hh + 16 * t + hb), o[hh][t]);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int t = 0; t < 2; ++t) tmem_pin8(o[hh][t]);
                    tc_fence_before();
                    const float un = pow2i(-E);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            acc[h] = fmaf(__uint_as_float(o[hh][0][h]) + __uint_as_float(o[hh][1][h]), un, acc[h]);
                }

                // ---- run ends: hand the set's state over, or write the run's partial
                if (mi.flags & kTcExport) {
                    float ls[8];
                    rows_sum(l_part, ls);
                    const bool x_ok =
                        mi.xseq == 0 || tc_wait_warp(xempty, uint32_t(mi.xseq - 1) & 1u, abort_flag);
                    fail = fail || !x_ok;
#pragma unroll
                    for (int h = 0; h < 8; ++h) xacc[(hb + h) * 128 + rt] = acc[h];
                    if (rt < 8) {
                        float mm = 0.0f, ll = 0.0f;
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            if (h == rt) {
                                mm = m_run[h];
                                ll = ls[h];
                            }
                        xm[hb + rt] = mm;
                        xl[hb + rt] = ll;
                    }
                    mbar_arrive(xfull);
                }
                if (mi.flags & kTcEmit) {
                    float ls[8];
                    rows_sum(l_part, ls);
                    if (mi.flags & kTcImport) {
                        const bool x_ok = tc_wait_warp(xfull, uint32_t(mi.xseq) & 1u, abort_flag);
                        fail = fail || !x_ok;
                        // combine the other set's (max, sum, accumulator) by log-sum-exp
#pragma unroll
                        for (int h = 0; h < 8; ++h) {
                            const float mo = xm[hb + h], lo = xl[hb + h], ao = xacc[(hb + h) * 128 + rt];
                            const float M = fmaxf(m_run[h], mo);
                            const float fs = M == m_run[h] ? 1.0f : fast_exp2(m_run[h] - M);
                            const float fo = M == mo ? 1.0f : fast_exp2(mo - M);
                            acc[h] = acc[h] * fs + ao * fo;
                            ls[h] = ls[h] * fs + lo * fo;
                            m_run[h] = M;
                        }
                        mbar_arrive(xempty);
                    }
                    if (!fail) {
                        const int64_t p0 = mi.slot * a.hpk;
                        if (rt < 8 && hb + rt < a.hpk) {
                            float mm = 0.0f, ll = 0.0f;
#pragma unroll
                            for (int h = 0; h < 8; ++h)
                                if (h == rt) {
                                    mm = m_run[h];
                                    ll = ls[h];
                                }
                            a.pm[p0 + hb + rt] = mm;
                            a.pl[p0 + hb + rt] = ll;
                        }
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            if (hb + h < a.hpk) a.pacc[(p0 + hb + h) * 128 + rt] = acc[h];
                    }
                }
                if (!next) break;
                // ---- the next chunk's V and scales (V^T and P are free: the values are in)
                stage_v(i + 2);
                mi = mn;
            }
            if (fail && rt == 0) {
                set_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols) : "memory");
    }
}

inline cudaError_t launch_split_h16_tc(const WarpArgs &wa, const LayerSrc &s, const MmaMaps &maps,
                                       cudaStream_t st) {
    const bool opt = wa.a.window > 0 || wa.a.softcap2 > 0.0f || wa.a.K > 1, imp = wa.a.scores != nullptr;
    auto kern = opt ? (imp ? split_h16_tc_kernel<true, true> : split_h16_tc_kernel<true, false>)
                    : (imp ? split_h16_tc_kernel<false, true> : split_h16_tc_kernel<false, false>);
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), TcCfg::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(unsigned(wa.G)), dim3(kTcWarps * 32), TcCfg::SMEM_ALLOC, st, wa, s, maps);
}

// One worker per SM (the CTA holds the SM's whole TMEM); 0 if the kernel
// cannot be resident.
inline int64_t split_h16_tc_workers() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    auto kern = split_h16_tc_kernel<false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM_ALLOC) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kTcWarps * 32, TcCfg::SMEM_ALLOC) != cudaSuccess)
        return 0;
    return occ >= 1 ? int64_t(sms) : 0;
}

}  // namespace kvd
