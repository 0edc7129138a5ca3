// kvd_evict.cu -- mass-based (Born) eviction on the device (cortiq
// LayerKvCache::evict_born, applied by KvCache::evict under
// EvictionPolicy::Born), batched over the sequences of a layer.
//
// Per sequence holding more than keep_last rows:
//   select  one CTA: the middle rows [sinks, stored - recents) compete for
//           the budget keep_last - sinks - recents by accumulated mass.  An
//           exact radix select over order-preserving 32-bit keys of the
//           masses finds the budget-th largest key T; every row above T is
//           kept and, of the rows equal to T, the lowest positions (the
//           order of the page's stable sort).  Two ordered block scans turn
//           the keep flags into the ascending list of kept rows, and the
//           CTA gathers imp along it (clearing the dropped rows' entries).
//   gather  the kept rows move down to positions 0 .. keep_last - 1 of every
//           storage independently (f32 K / V, int8 codes, their scales).
//           Kept positions ascend and kept[j] >= j, so a pass over j in
//           order that reads a stretch of rows before writing it never reads
//           a row an earlier write overwrote.  With many regions (sequence x
//           live head x storage) one CTA walks each region's tiles in order,
//           in place; with few, the rows go in batches of j through a
//           workspace copy (one kernel reads a batch, the next writes it), so
//           every batch spreads over the whole GPU -- or straight from their
//           sources when the batch's first source lies past its last row.
// The device length becomes keep_last in the select kernel; the host mirror
// is updated by the entry point.
//
// Also here: cortiq LayerKvCache::truncate_last (the speculative-decode
// reject), which only shortens the lengths and clears the dropped rows' imp.

#include <algorithm>
#include <vector>

#include "kvd_internal.cuh"

namespace kvd {
namespace {

constexpr int kSelectThreads = 1024;
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

// Exclusive prefix sum of `v` over the block in thread order, and the total.
__device__ __forceinline__ int block_excl_sum(int v, int *warp_sums, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    __syncthreads();  // warp_sums free (a previous call has read it)
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kSelectThreads / 32 ? warp_sums[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += t;
        }
        if (lane < kSelectThreads / 32) warp_sums[lane] = wi - w;  // exclusive
        if (lane == 31) warp_sums[kSelectThreads / 32] = wi;
    }
    __syncthreads();
    total = warp_sums[kSelectThreads / 32];
    return warp_sums[warp] + incl - v;
}

constexpr int kSelectRows = 8;   // consecutive rows per thread in the ordered scans
constexpr int kSelectLoads = 8;  // strided loads in flight per thread in the histogram passes

__global__ void __launch_bounds__(kSelectThreads) born_select_kernel(BornArgs a, BornTable t) {
    __shared__ uint32_t hist[256];
    __shared__ int warp_sums[kSelectThreads / 32 + 1];
    __shared__ uint32_t sel_digit;
    __shared__ int sel_need;
    const int i = blockIdx.x, tid = threadIdx.x;
    if (i >= t.n) return;
    const int b = t.seq[i], stored = t.stored[i];
    const int keep_last = a.keep_last, sink_n = a.sink_n;
    const int recent_n = min(a.recent, keep_last - sink_n);
    const int hi = stored - recent_n;  // middle rows: [sink_n, hi)
    const int budget = keep_last - sink_n - recent_n;
    float *imp = a.imp + t.imp_base[i];
    int32_t *idx = a.idx + int64_t(i) * keep_last;

    // ---- radix select of the budget-th largest key among the middle rows
    uint32_t prefix = 0, mask = 0;
    int need = budget;
    if (budget > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int d = tid; d < 256; d += kSelectThreads) hist[d] = 0;
            __syncthreads();
            // kSelectLoads loads in flight per thread before any is used
            for (int p0 = sink_n; p0 < hi; p0 += kSelectThreads * kSelectLoads) {
                float m[kSelectLoads];
#pragma unroll
                for (int u = 0; u < kSelectLoads; ++u) {
                    const int p = p0 + u * kSelectThreads + tid;
                    m[u] = p < hi ? imp[p] : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < kSelectLoads; ++u) {
                    const uint32_t k = mass_key(m[u]);
                    if (p0 + u * kSelectThreads + tid < hi && (k & mask) == prefix)
                        atomicAdd(&hist[(k >> shift) & 255u], 1u);
                }
            }
            __syncthreads();
            if (tid == 0) {
                int cum = 0, d = 255;
                for (; d > 0; --d) {
                    if (cum + int(hist[d]) >= need) break;
                    cum += int(hist[d]);
                }
                sel_digit = uint32_t(d);
                sel_need = need - cum;
            }
            __syncthreads();
            prefix |= sel_digit << shift;
            mask |= 255u << shift;
            need = sel_need;
        }
    }
    // prefix = the threshold key; `need` rows equal to it are kept, lowest first

    // ---- keep flags -> ascending list of kept rows (kSelectRows consecutive
    // rows per thread, in thread order)
    int eq_carry = 0, out_carry = 0;
    for (int p0 = 0; p0 < stored; p0 += kSelectThreads * kSelectRows) {
        const int pb = p0 + tid * kSelectRows;
        bool mid_gt[kSelectRows], mid_eq[kSelectRows];
        float mv[kSelectRows];
#pragma unroll
        for (int u = 0; u < kSelectRows; ++u) {
            const int p = pb + u;
            mv[u] = (budget > 0 && p >= sink_n && p < hi) ? imp[p] : 0.0f;
        }
        int n_eq = 0;
#pragma unroll
        for (int u = 0; u < kSelectRows; ++u) {
            const int p = pb + u;
            mid_gt[u] = mid_eq[u] = false;
            if (budget > 0 && p >= sink_n && p < hi) {
                const uint32_t k = mass_key(mv[u]);
                mid_gt[u] = k > prefix;
                mid_eq[u] = k == prefix;
            }
            n_eq += mid_eq[u];
        }
        int eq_total;
        int eq_rank = eq_carry + block_excl_sum(n_eq, warp_sums, eq_total);
        eq_carry += eq_total;
        bool keep[kSelectRows];
        int n_keep = 0;
#pragma unroll
        for (int u = 0; u < kSelectRows; ++u) {
            const int p = pb + u;
            keep[u] = p < stored && (p < sink_n || p >= hi || mid_gt[u] || (mid_eq[u] && eq_rank < need));
            eq_rank += mid_eq[u];
            n_keep += keep[u];
        }
        int out_total;
        int pos = out_carry + block_excl_sum(n_keep, warp_sums, out_total);
        out_carry += out_total;
#pragma unroll
        for (int u = 0; u < kSelectRows; ++u) {
            if (keep[u] && pos < keep_last) idx[pos] = pb + u;
            pos += keep[u];
        }
    }
    __syncthreads();
    if (out_carry != keep_last) {
        // cannot happen for finite masses: report it, and make the list the
        // identity so that the gather leaves every row where it is
        if (tid == 0) set_error(a.err, kErrBounds);
        for (int j = tid; j < keep_last; j += kSelectThreads) idx[j] = j;
        return;
    }

    // ---- imp follows its rows (in place, tiles in order); the entries of the
    // dropped rows are cleared: a row appended there later starts from zero
    // mass, as each appended row does on the page
    for (int j0 = sink_n; j0 < keep_last; j0 += kSelectThreads * kSelectLoads) {
        float v[kSelectLoads];
#pragma unroll
        for (int u = 0; u < kSelectLoads; ++u) {
            const int j = j0 + u * kSelectThreads + tid;
            v[u] = j < keep_last ? imp[idx[j]] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kSelectLoads; ++u) {
            const int j = j0 + u * kSelectThreads + tid;
            if (j < keep_last) imp[j] = v[u];
        }
        __syncthreads();
    }
    for (int j = keep_last + tid; j < stored; j += kSelectThreads) imp[j] = 0.0f;
    if (tid == 0) a.seq_len[b] = keep_last;
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
// x storage, blockIdx.z = table entry), through the workspace copy `stage`
// laid out [entry][live head][storage block of (j1 - j0) rows, padded to 16
// bytes].  to_stage: read the kept sources into it; else write it to rows j.
struct BatchArgs {
    GatherArgs g;
    char *stage;
    int64_t stage_group;   // bytes of one (entry, live head) block, a multiple of 16
    int64_t st_off[4];     // byte offset of each storage's block in it, multiples of 16
    int32_t n_live, j0, j1;
};

// Rows are a power-of-two number of units U (16-byte units where the row
// holds whole ones, else 4-byte words), so row and unit come from shifts.
template <bool TO_STAGE, typename U>
__device__ __forceinline__ void batch_copy(U *region, U *stage, int lu, const int32_t *kept, int j0, int rows,
                                           int64_t cap, uint32_t *err) {
    const int n = rows << lu;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
        const int j = j0 + (e >> lu), w = e & ((1 << lu) - 1);
        if (TO_STAGE) {
            const int32_t src = kept[j];
            if (src >= 0 && src < cap) stage[e] = region[(int64_t(src) << lu) + w];
            else set_error(err, kErrBounds);
        } else {
            region[(int64_t(j) << lu) + w] = stage[e];
        }
    }
}

// The batch's rows straight from their sources, for a batch whose every source
// lies at or past its end (kept[j0] >= j1, kept ascending): no row the batch
// writes is a source of it or of a later batch.
template <typename U>
__device__ __forceinline__ void direct_copy(U *region, int lu, const int32_t *kept, int j0, int rows, int64_t cap,
                                            uint32_t *err) {
    const int n = rows << lu;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
        const int j = j0 + (e >> lu), w = e & ((1 << lu) - 1);
        const int32_t src = kept[j];
        if (src >= 0 && src < cap) region[(int64_t(j) << lu) + w] = region[(int64_t(src) << lu) + w];
        else set_error(err, kErrBounds);
    }
}

// to_stage: read the batch's sources into the stage (or, for a batch whose
// sources all lie past it, copy it directly); else write the stage to its rows
// (nothing for a direct batch).
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
    if (kept[a.j0] >= a.j1) {
        if (!TO_STAGE) return;
        if (g.row_bytes % 16 == 0)
            direct_copy(reinterpret_cast<uint4 *>(region), log2_exact(g.row_bytes / 16), kept, a.j0, rows, cap, a.g.err);
        else
            direct_copy(reinterpret_cast<uint32_t *>(region), log2_exact(g.row_bytes / 4), kept, a.j0, rows, cap,
                        a.g.err);
        return;
    }
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

int64_t evict_idx_bytes(const Layer *l, int64_t keep_last) {
    return (int64_t(std::min(kSlice, l->n_seq)) * keep_last * 4 + 255) / 256 * 256;
}

int64_t evict_ws_bytes(const Layer *l, int64_t keep_last) {
    const int64_t stage = std::min(kEvictStage, int64_t(std::min(kSlice, l->n_seq)) * std::max(1, l->n_live) *
                                                    keep_last * row_bytes_all(l));
    return evict_idx_bytes(l, keep_last) + (stage + 255) / 256 * 256;
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
    BornArgs a;
    a.imp = imp;
    a.idx = static_cast<int32_t *>(workspace);  // the stage of the batched gather follows the lists
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
    for (size_t s0 = 0; s0 < todo.size(); s0 += kSlice) {
        BornTable t;
        t.n = int32_t(std::min<size_t>(kSlice, todo.size() - s0));
        for (int i = 0; i < t.n; ++i) {
            const int b = todo[s0 + i];
            t.seq[i] = b;
            t.stored[i] = int32_t(l->h_seq_len[b]);
            t.imp_base[i] = l->h_imp_base[b];
        }
        born_select_kernel<<<unsigned(t.n), kSelectThreads, 0, st>>>(a, t);
        if (cudaGetLastError() != cudaSuccess) return KVD_ECUDA;
        if (l->n_live <= 0 || g.n_st <= 0 || keep_last <= a.sink_n) continue;
        const int64_t regions = int64_t(t.n) * l->n_live * g.n_st;
        const int64_t stage_bytes = workspace_bytes - evict_idx_bytes(l, keep_last);
        const int64_t per_row = int64_t(t.n) * l->n_live * row_bytes_all(l);  // one j across the batch
        const int64_t pad = int64_t(t.n) * l->n_live * g.n_st * 16;            // blocks padded to 16 bytes
        const int64_t batch = (stage_bytes - pad) / per_row;
        if (regions >= kSerialRegions || batch < 1) {
            dim3 grid(unsigned(l->n_live * g.n_st), unsigned(t.n));
            born_gather_kernel<<<grid, kGatherThreads, 0, st>>>(g, t);
            if (cudaGetLastError() != cudaSuccess) return KVD_ECUDA;
            continue;
        }
        BatchArgs ba;
        ba.g = g;
        ba.stage = static_cast<char *>(workspace) + evict_idx_bytes(l, keep_last);
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
            const int64_t units = int64_t(ba.j1 - ba.j0) * 8;  // a code region's 16-byte units, for the grid
            dim3 grid(unsigned(std::max<int64_t>(1, std::min<int64_t>(ceil_div_ev(units, kGatherThreads), 1024))),
                      unsigned(l->n_live * g.n_st), unsigned(t.n));
            born_batch_kernel<true><<<grid, kGatherThreads, 0, st>>>(ba, t);
            born_batch_kernel<false><<<grid, kGatherThreads, 0, st>>>(ba, t);
            if (cudaGetLastError() != cudaSuccess) return KVD_ECUDA;
        }
    }
    for (int b : todo) l->h_seq_len[b] = keep_last;
    return KVD_OK;
}

extern "C" kvd_status kv_truncate_last(kvd_layer *L, const int32_t *n_drop, float *imp, void *stream) {
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
        if (cudaGetLastError() != cudaSuccess) return KVD_ECUDA;
        for (int i = 0; i < t.n; ++i) l->h_seq_len[t.seq[i]] = t.new_len[i];
    }
    return KVD_OK;
}
