// kvd_evict.cu -- mass-based (Born) eviction on the device (cortiq
// LayerKvCache::evict_born, applied by KvCache::evict under
// EvictionPolicy::Born), batched over the sequences of a layer.
//
// Per sequence holding more than keep_last rows:
//   select  the middle rows [sinks, stored - recents) compete for the
//           budget keep_last - sinks - recents by accumulated mass.  An
//           exact radix select over order-preserving 32-bit keys of the
//           masses finds the budget-th largest key T; every row above T is
//           kept and, of the rows equal to T, the lowest positions (the
//           order of the page's stable sort).  Ordered sums of per-chunk
//           counts turn the keep flags into the ascending list of kept rows,
//           and imp follows it (the dropped rows' entries cleared).  A chain
//           of short kernels, each spreading every sequence over CTAs of
//           4096 rows (see the select section below).
//   gather  the kept rows move down to positions 0 .. keep_last - 1 of every
//           storage independently (f32 K / V, int8 codes, their scales).
//           Kept positions ascend and kept[j] >= j, so a pass over j in
//           order that reads a stretch of rows before writing it never reads
//           a row an earlier write overwrote.  With many regions (sequence x
//           live head x storage) one CTA walks each region's tiles in order,
//           in place; with few, the rows go in batches of j through a
//           workspace copy (one kernel reads a batch, the next writes it), so
//           every batch spreads over the whole GPU; only rows whose source
//           lies inside the batch's own rows take the copy, the others are
//           copied straight across by the second kernel.
// The device length becomes keep_last in the select's last kernel; the host
// mirror is updated by the entry point.
//
// Also here: cortiq LayerKvCache::truncate_last (the speculative-decode
// reject), which only shortens the lengths and clears the dropped rows' imp.

#include <algorithm>
#include <vector>

#include "kvd_internal.cuh"

namespace kvd {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnits = 8;  // 16-byte (or smaller) units per thread per tile

struct BornTable {
    int32_t n;
    int32_t seq[kSlice];       // sequence of entry i
    int32_t stored[kSlice];    // its rows before the eviction
    int64_t imp_base[kSlice];  // its first imp entry
};

struct BornArgs {
    float *imp;
    int32_t *idx;  // [kSlice][keep_last] kept rows of each table entry
    int32_t *seq_len;
    uint32_t *err;
    int32_t keep_last, sink_n, recent;
};

// Order-preserving key of a float: larger float -> larger unsigned key,
// -0 and +0 equal (as the page's comparison treats them).
__device__ __forceinline__ uint32_t mass_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// The select over many CTAs: a chain of short kernels that each spread every
// sequence's rows over CTAs of kChunkRows rows:
//   sel_init   per entry: the radix state (prefix 0, need = budget), zeroed
//              histogram;
//   sel_hist   (x4, digits from the top byte down) each CTA histograms the
//              digit of its chunk's middle keys that match the prefix so far
//              and adds its bins into the entry's histogram;
//   sel_pick   (x4) one warp per entry finds the digit holding the need-th
//              largest key, extends the prefix and zeroes the histogram;
//   sel_count  each CTA counts its chunk's rows kept for sure (sinks, recents,
//              middle keys above the threshold) and its threshold-equal ones;
//   sel_scan   per entry, exclusive sums of those counts over the chunks in
//              order, and the check that exactly keep_last rows are kept;
//   sel_write  each CTA keeps the threshold-equal rows whose rank over the
//              whole sequence is below `need` (lowest positions first), and
//              writes its kept rows' positions to the ascending list;
//   sel_imp    the kept rows' imp entries into a copy, then (sel_imp_put) back
//              to positions 0 .. keep_last - 1, the dropped rows' entries
//              cleared, and the device length set.
// Each kernel is launched as a dependent of the one before (it waits first).
constexpr int kChunkRows = 4096;          // rows per CTA
constexpr int kChunkThreads = 256;
constexpr int kRowsPerThread = kChunkRows / kChunkThreads;  // consecutive rows per thread

struct SelState {
    uint32_t prefix, mask;
    int32_t need;         // threshold-equal rows still to keep (after the passes: of the threshold key)
    int32_t identity;     // 1: the kept count came out wrong; the list is the identity
};

struct SelArgs {
    float *imp;
    int32_t *idx;         // [kSlice][keep_last]
    float *imp_copy;      // [kSlice][keep_last]
    SelState *state;      // [kSlice]
    uint32_t *hist;       // [kSlice][256]
    int32_t *counts;      // [kSlice][chunks][2]: sure kept, threshold-equal
    int32_t *offsets;     // [kSlice][chunks][2]: exclusive sums of them
    int32_t *seq_len;
    uint32_t *err;
    int32_t keep_last, sink_n, recent, chunks;
};

struct SelRange {
    int stored, hi, budget, recent_n;
};

__device__ __forceinline__ SelRange sel_range(const SelArgs &a, const BornTable &t, int i) {
    SelRange r;
    r.stored = t.stored[i];
    r.recent_n = min(a.recent, a.keep_last - a.sink_n);
    r.hi = r.stored - r.recent_n;  // middle rows: [sink_n, hi)
    r.budget = a.keep_last - a.sink_n - r.recent_n;
    return r;
}

__global__ void sel_init_kernel(SelArgs a, BornTable t) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    if (i >= t.n) return;
    a.hist[i * 256 + threadIdx.x] = 0u;
    if (threadIdx.x == 0) {
        const SelRange r = sel_range(a, t, i);
        a.state[i] = SelState{0u, 0u, r.budget > 0 ? r.budget : 0, 0};
    }
}

__global__ void __launch_bounds__(kChunkThreads) sel_hist_kernel(SelArgs a, BornTable t, int shift) {
    __shared__ uint32_t h[256];
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.y, tid = threadIdx.x;
    if (i >= t.n) return;
    const SelRange r = sel_range(a, t, i);
    const SelState s = a.state[i];
    const int p0 = a.sink_n + blockIdx.x * kChunkRows, p1 = min(r.hi, p0 + kChunkRows);
    if (s.need <= 0 || p0 >= p1) return;
    h[tid] = 0u;
    __syncthreads();
    const float *imp = a.imp + t.imp_base[i];
    float m[kRowsPerThread];
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        const int p = p0 + u * kChunkThreads + tid;
        m[u] = p < p1 ? imp[p] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        const uint32_t k = mass_key(m[u]);
        if (p0 + u * kChunkThreads + tid < p1 && (k & s.mask) == s.prefix) atomicAdd(&h[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (h[tid] != 0u) atomicAdd(&a.hist[i * 256 + tid], h[tid]);
}

// One warp per entry: lane l holds bins 8l .. 8l + 7; the digit holding the
// need-th largest key is the highest d with (keys of digits >= d) >= need.
__global__ void sel_pick_kernel(SelArgs a, BornTable t, int shift) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x, lane = threadIdx.x;
    if (i >= t.n) return;
    SelState s = a.state[i];
    uint32_t *hist = a.hist + i * 256;
    uint32_t c[8];
    uint32_t tot = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        c[k] = hist[8 * lane + k];
        tot += c[k];
    }
    // keys in the bins above this lane's: the totals of the higher lanes
    uint32_t above = 0;
#pragma unroll
    for (int L = 31; L > 0; --L) {
        const uint32_t v = __shfl_sync(0xffffffffu, tot, L);
        if (L > lane) above += v;
    }
    const uint32_t need = uint32_t(s.need);
    // the lane whose bins hold the need-th key: above < need <= above + tot
    const bool mine = s.need > 0 && above < need && need <= above + tot;
    const unsigned who = __ballot_sync(0xffffffffu, mine);
    if (s.need > 0 && who != 0u && lane == __ffs(who) - 1) {
        uint32_t cum = above;
        int d = 8 * lane + 7;
        for (; d > 8 * lane; --d) {
            if (cum + c[d - 8 * lane] >= need) break;
            cum += c[d - 8 * lane];
        }
        s.prefix |= uint32_t(d) << shift;
        s.mask |= 255u << shift;
        s.need = int32_t(need - cum);
        a.state[i] = s;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) hist[8 * lane + k] = 0u;
}

// Exclusive prefix sum of `v` over a kChunkThreads block in thread order, and
// the total.  `ws` holds kChunkThreads / 32 + 1 ints.
__device__ __forceinline__ int chunk_excl_sum(int v, int *ws, int &total) {
    constexpr int W = kChunkThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    __syncthreads();  // ws free (a previous call has read it)
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < W ? ws[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += t;
        }
        if (lane < W) ws[lane] = wi - w;
        if (lane == 31) ws[W] = wi;
    }
    __syncthreads();
    total = ws[W];
    return ws[warp] + incl - v;
}

// Keep flags of a thread's kRowsPerThread consecutive rows from pb: sure =
// sinks, recents, middle keys above the threshold; eq = middle keys equal to it.
__device__ __forceinline__ void sel_flags(const float *imp, const SelRange &r, int sink_n, uint32_t thr, int pb,
                                          bool (&sure)[kRowsPerThread], bool (&eq)[kRowsPerThread]) {
    float m[kRowsPerThread];
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        const int p = pb + u;
        m[u] = (r.budget > 0 && p >= sink_n && p < r.hi) ? imp[p] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        const int p = pb + u;
        const bool mid = r.budget > 0 && p >= sink_n && p < r.hi;
        const uint32_t k = mass_key(m[u]);
        sure[u] = p < r.stored && (p < sink_n || p >= r.hi || (mid && k > thr));
        eq[u] = mid && k == thr;
    }
}

__global__ void __launch_bounds__(kChunkThreads) sel_count_kernel(SelArgs a, BornTable t) {
    __shared__ int ws[kChunkThreads / 32 + 1];
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.y, c = blockIdx.x;
    if (i >= t.n) return;
    const SelRange r = sel_range(a, t, i);
    if (c * kChunkRows >= r.stored) return;
    const uint32_t thr = a.state[i].prefix;
    bool sure[kRowsPerThread], eq[kRowsPerThread];
    sel_flags(a.imp + t.imp_base[i], r, a.sink_n, thr, c * kChunkRows + threadIdx.x * kRowsPerThread, sure, eq);
    int ns = 0, ne = 0;
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        ns += sure[u];
        ne += eq[u];
    }
    int tot_s, tot_e;
    chunk_excl_sum(ns, ws, tot_s);
    chunk_excl_sum(ne, ws, tot_e);
    if (threadIdx.x == 0) {
        a.counts[(int64_t(i) * a.chunks + c) * 2] = tot_s;
        a.counts[(int64_t(i) * a.chunks + c) * 2 + 1] = tot_e;
    }
}

// One warp per entry: exclusive sums of the chunk counts in chunk order.
__global__ void sel_scan_kernel(SelArgs a, BornTable t) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x, lane = threadIdx.x;
    if (i >= t.n) return;
    const SelRange r = sel_range(a, t, i);
    const int nc = (r.stored + kChunkRows - 1) / kChunkRows;
    int carry_s = 0, carry_e = 0;
    for (int c0 = 0; c0 < nc; c0 += 32) {
        const int c = c0 + lane;
        const int64_t o = (int64_t(i) * a.chunks + c) * 2;
        const int vs = c < nc ? a.counts[o] : 0, ve = c < nc ? a.counts[o + 1] : 0;
        int is = vs, ie = ve;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int ts = __shfl_up_sync(0xffffffffu, is, off), te = __shfl_up_sync(0xffffffffu, ie, off);
            if (lane >= off) is += ts, ie += te;
        }
        if (c < nc) {
            a.offsets[o] = carry_s + is - vs;
            a.offsets[o + 1] = carry_e + ie - ve;
        }
        carry_s += __shfl_sync(0xffffffffu, is, 31);
        carry_e += __shfl_sync(0xffffffffu, ie, 31);
    }
    if (lane == 0) {
        const int need = a.state[i].need;
        if (carry_s + min(carry_e, need) != a.keep_last) {
            // cannot happen for finite masses: report it, and make the list
            // the identity so that the gather leaves every row where it is
            set_error(a.err, kErrBounds);
            a.state[i].identity = 1;
        }
    }
}

__global__ void __launch_bounds__(kChunkThreads) sel_write_kernel(SelArgs a, BornTable t) {
    __shared__ int ws[kChunkThreads / 32 + 1];
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.y, c = blockIdx.x;
    if (i >= t.n) return;
    const SelRange r = sel_range(a, t, i);
    if (c * kChunkRows >= r.stored) return;
    int32_t *idx = a.idx + int64_t(i) * a.keep_last;
    const SelState s = a.state[i];
    if (s.identity) {
        for (int j = c * kChunkRows + threadIdx.x; j < min(a.keep_last, (c + 1) * kChunkRows); j += kChunkThreads)
            idx[j] = j;
        return;
    }
    const int pb = c * kChunkRows + threadIdx.x * kRowsPerThread;
    bool sure[kRowsPerThread], eq[kRowsPerThread];
    sel_flags(a.imp + t.imp_base[i], r, a.sink_n, s.prefix, pb, sure, eq);
    const int64_t o = (int64_t(i) * a.chunks + c) * 2;
    const int sure_before = a.offsets[o], eq_before = a.offsets[o + 1];
    int ne = 0;
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) ne += eq[u];
    int tot;
    int eq_rank = eq_before + chunk_excl_sum(ne, ws, tot);
    bool keep[kRowsPerThread];
    int nk = 0;
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        keep[u] = sure[u] || (eq[u] && eq_rank < s.need);  // equal keys: the lowest positions first
        eq_rank += eq[u];
        nk += keep[u];
    }
    int pos = sure_before + min(eq_before, s.need) + chunk_excl_sum(nk, ws, tot);
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        if (keep[u] && pos < a.keep_last) idx[pos] = pb + u;
        pos += keep[u];
    }
}

// The kept rows' masses into the copy (rows below sink_n stay where they are).
__global__ void sel_imp_get_kernel(SelArgs a, BornTable t) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.y;
    if (i >= t.n || a.state[i].identity) return;
    const float *imp = a.imp + t.imp_base[i];
    const int32_t *idx = a.idx + int64_t(i) * a.keep_last;
    float *cp = a.imp_copy + int64_t(i) * a.keep_last;
    const int j0 = a.sink_n + blockIdx.x * kChunkRows;
    for (int j = j0 + threadIdx.x; j < min(a.keep_last, j0 + kChunkRows); j += blockDim.x) cp[j] = imp[idx[j]];
}

// The copy back to rows sink_n .. keep_last - 1, the dropped rows' entries
// cleared (a row appended there later starts from zero mass, as each appended
// row does on the page), and the device length.
__global__ void sel_imp_put_kernel(SelArgs a, BornTable t) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.y;
    if (i >= t.n || a.state[i].identity) return;
    const int stored = t.stored[i];
    float *imp = a.imp + t.imp_base[i];
    const float *cp = a.imp_copy + int64_t(i) * a.keep_last;
    const int j0 = a.sink_n + blockIdx.x * kChunkRows;
    for (int j = j0 + threadIdx.x; j < min(stored, j0 + kChunkRows); j += blockDim.x)
        imp[j] = j < a.keep_last ? cp[j] : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) a.seq_len[t.seq[i]] = a.keep_last;
}

// log2 of a power of two.
__host__ __device__ __forceinline__ int log2_exact(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

struct GatherStorage {
    char *base;         // the storage buffer
    int32_t row_bytes;  // bytes per row (a multiple of 4)
};

struct GatherArgs {
    GatherStorage st[4];
    int32_t n_st;
    const int32_t *idx;
    const int64_t *row_base, *cap;
    uint32_t *err;
    int32_t keep_last, sink_n;
};

// Move the kept rows of one region (rows of `upr` units of type U) down to
// positions sink_n .. keep_last - 1, tile by tile in order.  A kept row
// outside [0, cap) (corrupt metadata) is reported and skipped.
template <typename U>
__device__ void gather_region(U *region, int upr, const int32_t *kept, int sink_n, int keep_last,
                              int64_t cap, uint32_t *err) {
    const int lu = log2_exact(upr);  // upr is a power of two
    const int tile_rows = max(1, kGatherThreads * kGatherUnits / upr);
    for (int j0 = sink_n; j0 < keep_last; j0 += tile_rows) {
        const int rows = min(tile_rows, keep_last - j0);
        // a tile whose last row stays in place stays entirely (kept ascends, kept[j] >= j)
        if (kept[j0 + rows - 1] == j0 + rows - 1) continue;
        U r[kGatherUnits];
        const int units = rows * upr;
#pragma unroll
        for (int k = 0; k < kGatherUnits; ++k) {
            const int e = threadIdx.x + k * kGatherThreads;
            if (e < units) {
                const int32_t src = kept[j0 + (e >> lu)];
                if (src >= 0 && src < cap) r[k] = region[(int64_t(src) << lu) + (e & (upr - 1))];
                else set_error(err, kErrBounds);
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kGatherUnits; ++k) {
            const int e = threadIdx.x + k * kGatherThreads;
            if (e < units) region[(int64_t(j0 + (e >> lu)) << lu) + (e & (upr - 1))] = r[k];
        }
        __syncthreads();
    }
}

// Batched gather: rows j in [j0, j1) of every region (blockIdx.y = live head
// x storage, blockIdx.z = table entry), the rows whose sources lie inside the
// batch through the workspace copy `stage` laid out [entry][live head][storage
// block of (j1 - j0) rows, padded to 16 bytes].
struct BatchArgs {
    GatherArgs g;
    char *stage;
    int64_t stage_group;   // bytes of one (entry, live head) block, a multiple of 16
    int64_t st_off[4];     // byte offset of each storage's block in it, multiples of 16
    int32_t n_live, j0, j1;
};

// Rows are a power-of-two number of units U (16-byte units where the row
// holds whole ones, else 4-byte words), so row and unit come from shifts.
// Rows j0 .. j0 + rows - 1 of one region.  A row whose source lies at or past
// the batch's end (kept[j] >= j1) is copied straight across by the second
// kernel: neither kernel writes there, and later batches write there only
// after this one.  A row whose source lies inside the batch's own rows goes
// through the stage: the first kernel reads all of those before the second
// writes any row.  Rows are a power-of-two number of units U (16-byte units
// where the row holds whole ones, else 4-byte words), so row and unit come
// from shifts.
template <bool TO_STAGE, typename U>
__device__ __forceinline__ void batch_copy(U *region, U *stage, int lu, const int32_t *kept, int j0, int rows,
                                           int64_t cap, uint32_t *err) {
    constexpr int kIn = 4;  // units per thread in flight
    const int n = rows << lu, j1 = j0 + rows;
    const int stride = gridDim.x * blockDim.x;
    for (int e0 = blockIdx.x * blockDim.x + threadIdx.x; e0 < n; e0 += kIn * stride) {
        int32_t src[kIn];
        U v[kIn];
#pragma unroll
        for (int k = 0; k < kIn; ++k) {
            const int e = e0 + k * stride;
            src[k] = -1;
            if (e < n) {
                const int j = j0 + (e >> lu), w = e & ((1 << lu) - 1);
                src[k] = kept[j];
                if (src[k] < 0 || src[k] >= cap) {
                    if (TO_STAGE) set_error(err, kErrBounds);
                    src[k] = -1;
                } else if (TO_STAGE ? src[k] < j1 : src[k] >= j1) {
                    v[k] = region[(int64_t(src[k]) << lu) + w];
                } else if (!TO_STAGE) {
                    v[k] = stage[e];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kIn; ++k) {
            const int e = e0 + k * stride;
            if (src[k] < 0) continue;
            if (TO_STAGE) {
                if (src[k] < j1) stage[e] = v[k];
            } else {
                region[(int64_t(j0 + (e >> lu)) << lu) + (e & ((1 << lu) - 1))] = v[k];
            }
        }
    }
}

// to_stage: read the batch's rows whose sources lie inside it into the stage;
// else write every row of the batch (from the stage, or from its source).
template <bool TO_STAGE>
__global__ void __launch_bounds__(kGatherThreads) born_batch_kernel(BatchArgs a, BornTable t) {
    const int i = blockIdx.z;
    if (i >= t.n) return;
    const int s = blockIdx.y % a.g.n_st, gl = blockIdx.y / a.g.n_st;
    const int b = t.seq[i];
    const GatherStorage g = a.g.st[s];
    const int64_t cap = a.g.cap[b];
    char *region = g.base + (a.g.row_base[b] + int64_t(gl) * cap) * g.row_bytes;
    char *stage = a.stage + (int64_t(i) * a.n_live + gl) * a.stage_group + a.st_off[s];
    const int32_t *kept = a.g.idx + int64_t(i) * a.g.keep_last;
    const int rows = a.j1 - a.j0;
    if (TO_STAGE && kept[a.j0] >= a.j1) return;  // every source lies past the batch
    if (g.row_bytes % 16 == 0)
        batch_copy<TO_STAGE>(reinterpret_cast<uint4 *>(region), reinterpret_cast<uint4 *>(stage),
                             log2_exact(g.row_bytes / 16), kept, a.j0, rows, cap, a.g.err);
    else
        batch_copy<TO_STAGE>(reinterpret_cast<uint32_t *>(region), reinterpret_cast<uint32_t *>(stage),
                             log2_exact(g.row_bytes / 4), kept, a.j0, rows, cap, a.g.err);
}

__global__ void __launch_bounds__(kGatherThreads) born_gather_kernel(GatherArgs a, BornTable t) {
    const int i = blockIdx.y;
    if (i >= t.n) return;
    const int s = blockIdx.x % a.n_st, gl = blockIdx.x / a.n_st;
    const int b = t.seq[i];
    const GatherStorage g = a.st[s];
    const int64_t row0 = a.row_base[b] + int64_t(gl) * a.cap[b];
    char *region = g.base + row0 * g.row_bytes;
    const int32_t *kept = a.idx + int64_t(i) * a.keep_last;
    const int64_t cap = a.cap[b];
    if (g.row_bytes % 16 == 0)
        gather_region(reinterpret_cast<uint4 *>(region), g.row_bytes / 16, kept, a.sink_n, a.keep_last, cap, a.err);
    else if (g.row_bytes % 8 == 0)
        gather_region(reinterpret_cast<uint2 *>(region), g.row_bytes / 8, kept, a.sink_n, a.keep_last, cap, a.err);
    else
        gather_region(reinterpret_cast<uint32_t *>(region), g.row_bytes / 4, kept, a.sink_n, a.keep_last, cap,
                      a.err);
}

struct TruncTable {
    int32_t n;
    int32_t seq[kSlice];
    int32_t new_len[kSlice];
    int32_t old_len[kSlice];
    int64_t imp_base[kSlice];
};

__global__ void truncate_kernel(int32_t *seq_len, float *imp, TruncTable t) {
    const int i = blockIdx.x;
    if (i >= t.n) return;
    if (imp != nullptr) {
        float *m = imp + t.imp_base[i];
        for (int p = t.new_len[i] + int(threadIdx.x); p < t.old_len[i]; p += blockDim.x) m[p] = 0.0f;
    }
    if (threadIdx.x == 0) seq_len[t.seq[i]] = t.new_len[i];
}

constexpr int64_t kEvictStage = int64_t(64) << 20;  // most bytes of the batched gather's copy
constexpr int kSerialRegions = 2 * 152;               // enough regions to walk each in one CTA

// Bytes per row summed over the layer's storages.
int64_t row_bytes_all(const Layer *l) {
    const bool qk = l->mode == KVD_Q8 || l->mode == KVD_Q8K;
    const bool qv = l->mode == KVD_Q8 || l->mode == KVD_Q8V;
    return (qk ? l->hd + (l->hd / 32) * 4 : l->hd * 4) + (qv ? l->hd + 4 : l->hd * 4);
}

int64_t ceil_div_ev(int64_t x, int64_t y) { return (x + y - 1) / y; }

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

int64_t evict_idx_bytes(const Layer *l, int64_t keep_last) {
    return round256(int64_t(std::min(kSlice, l->n_seq)) * keep_last * 4);
}

// Chunks of kChunkRows rows of the longest sequence the layer can hold.
int32_t sel_chunks(const Layer *l) { return int32_t(std::max<int64_t>(1, ceil_div_ev(l->max_cap, kChunkRows))); }

// The workspace before the batched gather's copy: the kept lists, the masses'
// copy, then the select's state, histograms, chunk counts and their sums.
struct SelLayout {
    int64_t idx, imp_copy, state, hist, counts, offsets, end;
};

SelLayout sel_layout(const Layer *l, int64_t keep_last) {
    const int64_t n = std::min(kSlice, l->n_seq);
    SelLayout w;
    w.idx = 0;
    w.imp_copy = evict_idx_bytes(l, keep_last);
    w.state = w.imp_copy + evict_idx_bytes(l, keep_last);
    w.hist = w.state + round256(n * int64_t(sizeof(SelState)));
    w.counts = w.hist + round256(n * 256 * 4);
    w.offsets = w.counts + round256(n * sel_chunks(l) * 8);
    w.end = w.offsets + round256(n * sel_chunks(l) * 8);
    return w;
}

int64_t evict_ws_bytes(const Layer *l, int64_t keep_last) {
    const int64_t stage = std::min(kEvictStage, int64_t(std::min(kSlice, l->n_seq)) * std::max(1, l->n_live) *
                                                    keep_last * row_bytes_all(l));
    return sel_layout(l, keep_last).end + round256(stage);
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kv_evict_workspace_bytes(const kvd_layer *L, int64_t keep_last, int64_t *bytes_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || bytes_out == nullptr || keep_last < 0 || keep_last > (int64_t(1) << 31) - 1)
        return KVD_EINVAL;
    *bytes_out = evict_ws_bytes(l, keep_last);
    return KVD_OK;
}

extern "C" kvd_status kv_evict_born(kvd_layer *L, float *imp, int64_t keep_last, int32_t sink,
                                    int32_t recent, void *workspace, int64_t workspace_bytes,
                                    void *stream) {
    KVD_NVTX_RANGE("kv_evict_born");
    Layer *l = checked_layer(L);
    if (l == nullptr || imp == nullptr || (reinterpret_cast<uintptr_t>(imp) & 3)) return KVD_EINVAL;
    if (keep_last < 0 || keep_last > (int64_t(1) << 31) - 1 || sink < 0 || recent < 0) return KVD_EINVAL;
    const int64_t need = evict_ws_bytes(l, keep_last);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return KVD_EINVAL;
    std::vector<int32_t> todo;
    for (int b = 0; b < l->n_seq; ++b)
        if (l->h_seq_len[b] > keep_last) todo.push_back(b);
    if (todo.empty()) return KVD_OK;
    cudaStream_t st = as_stream(stream);
    const SelLayout wl = sel_layout(l, keep_last);
    char *wsb = static_cast<char *>(workspace);
    BornArgs a;
    a.imp = imp;
    a.idx = reinterpret_cast<int32_t *>(wsb + wl.idx);  // the stage of the batched gather follows the select's data
    a.seq_len = l->d_seq_len;
    a.err = l->d_err;
    a.keep_last = int32_t(keep_last);
    a.sink_n = int32_t(std::min<int64_t>(sink, keep_last));
    a.recent = recent;
    GatherArgs g;
    g.n_st = 0;
    auto add = [&](int slot, int32_t row_bytes) {
        if (l->buf[slot] != nullptr) g.st[g.n_st++] = GatherStorage{static_cast<char *>(l->buf[slot]), row_bytes};
    };
    const bool qk = l->mode == KVD_Q8 || l->mode == KVD_Q8K;
    const bool qv = l->mode == KVD_Q8 || l->mode == KVD_Q8V;
    if (qk) {
        add(KVD_BUF_KQ, l->hd);
        add(KVD_BUF_KS, (l->hd / 32) * 4);
    } else {
        add(KVD_BUF_K, l->hd * 4);
    }
    if (qv) {
        add(KVD_BUF_VQ, l->hd);
        add(KVD_BUF_VS, 4);
    } else {
        add(KVD_BUF_V, l->hd * 4);
    }
    g.idx = a.idx;
    g.err = l->d_err;
    g.row_base = l->d_row_base;
    g.cap = l->d_cap;
    g.keep_last = a.keep_last;
    g.sink_n = a.sink_n;
    SelArgs sa;
    sa.imp = imp;
    sa.idx = a.idx;
    sa.imp_copy = reinterpret_cast<float *>(wsb + wl.imp_copy);
    sa.state = reinterpret_cast<SelState *>(wsb + wl.state);
    sa.hist = reinterpret_cast<uint32_t *>(wsb + wl.hist);
    sa.counts = reinterpret_cast<int32_t *>(wsb + wl.counts);
    sa.offsets = reinterpret_cast<int32_t *>(wsb + wl.offsets);
    sa.seq_len = l->d_seq_len;
    sa.err = l->d_err;
    sa.keep_last = a.keep_last;
    sa.sink_n = a.sink_n;
    sa.recent = a.recent;
    sa.chunks = sel_chunks(l);
    for (size_t s0 = 0; s0 < todo.size(); s0 += kSlice) {
        BornTable t;
        t.n = int32_t(std::min<size_t>(kSlice, todo.size() - s0));
        for (int i = 0; i < t.n; ++i) {
            const int b = todo[s0 + i];
            t.seq[i] = b;
            t.stored[i] = int32_t(l->h_seq_len[b]);
            t.imp_base[i] = l->h_imp_base[b];
        }
        int64_t most = 0;
        for (int i = 0; i < t.n; ++i) most = std::max<int64_t>(most, t.stored[i]);
        const unsigned chunks = unsigned(ceil_div_ev(most, kChunkRows));
        const dim3 cgrid(chunks, unsigned(t.n)), eg(unsigned(t.n));
        cudaError_t e = launch_pdl(sel_init_kernel, eg, dim3(256), 0, st, sa, t);
        for (int shift = 24; shift >= 0 && e == cudaSuccess; shift -= 8) {
            e = launch_pdl(sel_hist_kernel, cgrid, dim3(kChunkThreads), 0, st, sa, t, shift);
            if (e == cudaSuccess) e = launch_pdl(sel_pick_kernel, eg, dim3(32), 0, st, sa, t, shift);
        }
        if (e == cudaSuccess) e = launch_pdl(sel_count_kernel, cgrid, dim3(kChunkThreads), 0, st, sa, t);
        if (e == cudaSuccess) e = launch_pdl(sel_scan_kernel, eg, dim3(32), 0, st, sa, t);
        if (e == cudaSuccess) e = launch_pdl(sel_write_kernel, cgrid, dim3(kChunkThreads), 0, st, sa, t);
        if (e == cudaSuccess) e = launch_pdl(sel_imp_get_kernel, cgrid, dim3(kChunkThreads), 0, st, sa, t);
        if (e == cudaSuccess) e = launch_pdl(sel_imp_put_kernel, cgrid, dim3(kChunkThreads), 0, st, sa, t);
        if (e != cudaSuccess) return KVD_ECUDA;
        if (l->n_live <= 0 || g.n_st <= 0 || keep_last <= a.sink_n) continue;
        const int64_t regions = int64_t(t.n) * l->n_live * g.n_st;
        const int64_t stage_bytes = workspace_bytes - wl.end;
        const int64_t per_row = int64_t(t.n) * l->n_live * row_bytes_all(l);  // one j across the batch
        const int64_t pad = int64_t(t.n) * l->n_live * g.n_st * 16;            // blocks padded to 16 bytes
        const int64_t batch = (stage_bytes - pad) / per_row;
        if (regions >= kSerialRegions || batch < 1) {
            dim3 grid(unsigned(l->n_live * g.n_st), unsigned(t.n));
            born_gather_kernel<<<grid, kGatherThreads, 0, st>>>(g, t);
            if (launch_status() != cudaSuccess) return KVD_ECUDA;
            continue;
        }
        BatchArgs ba;
        ba.g = g;
        ba.stage = wsb + wl.end;
        ba.n_live = l->n_live;
        for (int64_t j0 = a.sink_n; j0 < keep_last; j0 += batch) {
            ba.j0 = int32_t(j0);
            ba.j1 = int32_t(std::min<int64_t>(keep_last, j0 + batch));
            int64_t off = 0;
            for (int k = 0; k < g.n_st; ++k) {
                ba.st_off[k] = off;
                off += (int64_t(ba.j1 - ba.j0) * g.st[k].row_bytes + 15) / 16 * 16;
            }
            ba.stage_group = off;
            // a code region's 16-byte units, four per thread in flight
            const int64_t units = int64_t(ba.j1 - ba.j0) * 8;
            dim3 grid(unsigned(std::max<int64_t>(1, std::min<int64_t>(ceil_div_ev(units, 4 * kGatherThreads), 256))),
                      unsigned(l->n_live * g.n_st), unsigned(t.n));
            born_batch_kernel<true><<<grid, kGatherThreads, 0, st>>>(ba, t);
            born_batch_kernel<false><<<grid, kGatherThreads, 0, st>>>(ba, t);
            if (launch_status() != cudaSuccess) return KVD_ECUDA;
        }
    }
    for (int b : todo) l->h_seq_len[b] = keep_last;
    return KVD_OK;
}

extern "C" kvd_status kv_truncate_last(kvd_layer *L, const int32_t *n_drop, float *imp, void *stream) {
    KVD_NVTX_RANGE("kv_truncate_last");
    Layer *l = checked_layer(L);
    if (l == nullptr || (reinterpret_cast<uintptr_t>(imp) & 3)) return KVD_EINVAL;
    for (int b = 0; b < l->n_seq; ++b)
        if (n_drop != nullptr && n_drop[b] < 0) return KVD_EINVAL;
    std::vector<int32_t> todo;
    for (int b = 0; b < l->n_seq; ++b)
        if ((n_drop ? n_drop[b] : 1) > 0 && l->h_seq_len[b] > 0) todo.push_back(b);
    cudaStream_t st = as_stream(stream);
    for (size_t s0 = 0; s0 < todo.size(); s0 += kSlice) {
        TruncTable t;
        t.n = int32_t(std::min<size_t>(kSlice, todo.size() - s0));
        for (int i = 0; i < t.n; ++i) {
            const int b = todo[s0 + i];
            const int64_t d = std::min<int64_t>(n_drop ? n_drop[b] : 1, l->h_seq_len[b]);
            t.seq[i] = b;
            t.old_len[i] = int32_t(l->h_seq_len[b]);
            t.new_len[i] = int32_t(l->h_seq_len[b] - d);
            t.imp_base[i] = l->h_imp_base[b];
        }
        truncate_kernel<<<unsigned(t.n), 256, 0, st>>>(l->d_seq_len, imp, t);
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    // the host mirror changes once every launch has gone in
    for (int b : todo) l->h_seq_len[b] -= std::min<int64_t>(n_drop ? n_drop[b] : 1, l->h_seq_len[b]);
    return KVD_OK;
}
