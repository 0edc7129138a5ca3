// kvd_decode.cu -- host entry points of the decode path: GQA decode attention
// over a layer (cortiq attend_group for every group, batched over sequences)
// and the R-SWA ring write / decode (rswa RingCache::write_decode_step,
// decode_attention), plus their merge and imp kernels' launches.

#include <algorithm>
#include <cmath>
#include <vector>

#include <cstring>

#include "kvd_split_mma.cuh"

namespace kvd {

cudaError_t split_layer_f32(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
cudaError_t split_layer_q8(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
cudaError_t split_layer_q8k(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
cudaError_t split_layer_q8v(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
int q8_tc_variant(int);
cudaError_t split_layer_q8_tc(int, const WarpArgs &, const LayerSrc &, const MmaMaps &, cudaStream_t);
int64_t split_q8_tc_workers(int);

namespace {


struct DecodeWs {
    int64_t pm, pl, pacc, ml, scores, units, total;  // byte offsets; total < 0 if unknown
    int64_t slots;                            // tensor-core path partial slots
    int32_t nc_max;
};

// The q8_2f cache with head_dim 128 runs on the tensor-core kernel when its
// TMA descriptors exist.
bool warp_path(const Layer *l) {
    return l->mode == KVD_Q8 && l->hd == 128 && l->have_tmap_kq && l->have_tmap_vq;
}

// Partial slots the tensor-core kernel may write: every unit's blocks at full
// capacity plus one per worker (each worker start splits at most one block).
int64_t warp_slots(const Layer *l, int hpk) {
    int64_t nb = 0;
    for (int b = 0; b < l->n_seq; ++b)
        nb += int64_t(l->n_live) * ceil_div(ceil_div(l->h_cap[b], kWR), kBlockTiles);
    const int64_t g = split_q8_tc_workers(q8_tc_variant(hpk));
    return g > 0 ? nb + g : -1;
}

DecodeWs decode_ws(const Layer *l, int32_t n_q, bool imp) {
    DecodeWs w;
    const int hpk = n_q / l->n_kv;
    w.nc_max = int32_t(std::max<int64_t>(1, ceil_div(l->max_cap, kMinChunk)));
    int64_t P = int64_t(l->n_seq) * std::max(1, l->n_live) * w.nc_max * hpk;
    w.slots = 0;
    if (warp_path(l)) {
        w.slots = warp_slots(l, hpk);
        if (w.slots < 0) {
            w.total = -1;
            return w;
        }
        P = std::max(P, w.slots * hpk);
    }
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.pm = take(P * 4);
    w.pl = take(P * 4);
    w.pacc = take(P * l->hd * 4);
    w.ml = take(int64_t(l->n_seq) * n_q * 2 * 4);
    w.scores = imp ? take((l->total_rows + kRowAlign) * hpk * 4) : -1;
    w.units = take(int64_t(l->n_seq) * std::max(1, l->n_live) * 2 * 8);
    w.total = o;
    return w;
}

// Most workers the tensor-core verify of the R-SWA int8 mirror launches (a
// bound on resident one-warp CTAs, so its workspace size needs no device).
constexpr int64_t kRswaTcWorkers = 2048;

struct RswaWs {
    int64_t err, pm, pl, pacc, total;
    int32_t nc_max;
    // tensor-core verify of the int8 mirror (tc): run partials [slot][K],
    // per-launch unit slot ranges and the stream tables the kernel reads
    // (lengths, capacities, row bases, head map)
    bool tc = false;
    int64_t slots = 0, tc_pm = -1, tc_pl = -1, tc_pacc = -1;
    int64_t units = -1, t_len = -1, t_cap = -1, t_base = -1, t_live = -1;
};

// The int8 mirror's verify runs on the tensor-core kernel at head_dim 128 with
// up to 8 drafts, when every head's block is a whole number of 32-row tiles
// (the tiles' scale copies stay inside it) and its rows fit the TMA's int32
// coordinates.
bool rswa_tc_shape(int32_t B, int32_t H, int32_t hd, int64_t ref_cap, int32_t K) {
    return hd == 128 && K <= 8 && ref_cap > 0 && ref_cap % kWR == 0 && int64_t(B) * H * ref_cap < (int64_t(1) << 31);
}

// K > 1: a verify of K drafts (K partial rows per chunk; the ring's chunk
// slots hold the one tail partial).  tc: also lay out the tensor-core verify's
// regions (they alias the chunk partials: a call uses one or the other).
RswaWs rswa_ws(int32_t B, int32_t H, int32_t hd, int64_t ref_cap, int32_t W, int32_t K = 1, bool tc = false) {
    RswaWs w;
    w.nc_max = int32_t(ceil_div(ref_cap, kMinChunk) + ceil_div(W, kMinChunk));
    const int64_t P = int64_t(B) * H * w.nc_max * K;
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.err = take(16);
    const int64_t base = o;
    w.pm = take(P * 4);
    w.pl = take(P * 4);
    w.pacc = take(P * hd * 4);
    const int64_t end_chunks = o;
    if (tc && rswa_tc_shape(B, H, hd, ref_cap, K)) {
        w.tc = true;
        o = base;
        const int64_t n = std::min<int32_t>(B, kSlice);
        w.slots = n * H * ceil_div(ceil_div(ref_cap, kWR), kBlockTiles) + kRswaTcWorkers;
        w.tc_pm = take(w.slots * K * 4);
        w.tc_pl = take(w.slots * K * 4);
        w.tc_pacc = take(w.slots * K * hd * 4);
        w.units = take(n * H * 2 * 8);
        w.t_len = take(n * 4);
        w.t_cap = take(n * 8);
        w.t_base = take(n * 8);
        w.t_live = take(int64_t(H) * 4);
    }
    w.total = std::max(o, end_chunks);
    return w;
}

// ------------------------------------------------------------- run merge

struct RunMergeArgs {
    const float *pm, *pl, *pacc;  // run partials [slot][hpk] (+ [128])
    const int64_t *unit_slots;    // [n_seq * n_live][2]: first and last run slot of each unit
    float *out;                   // [n_seq][n_q][128]
    float *ml;                    // (max, sum) per (sequence, query head) for imp, or null
    const float *sinks;           // learned sink logit per query head [n_q], or null
    int32_t n_q, hpk;
    int32_t K = 1, hg = 0;        // verify: K drafts, hg heads per group (hpk = K * hg)
};

// Log-sum-exp merge of the run partials of one (sequence, query head) written
// by the tensor-core kernel: out[d] = field[d] * sum_r acc_r[d] 2^(m_r - M) /
// sum_r l_r 2^(m_r - M).  A unit's runs fill the slot range between the
// first and last run slots the split kernel recorded for it, with empty
// markers (max -inf) in skipped slots.  Eight warps take every eighth slot,
// loading four slots' (max, sum, accumulator) before using any (long units
// have a hundred or more runs, so the loads must overlap); each keeps a
// running maximum, lanes own four channels, and the warps' sums are rescaled
// to the common maximum and added in a fixed order.
constexpr int kMergeWarps = 8;
constexpr int kMergeBatch = 4;

__global__ void __launch_bounds__(32 * kMergeWarps) merge_runs_kernel(RunMergeArgs a, MergeLayerSrc src) {
    __shared__ float wmax[kMergeWarps], wsum[kMergeWarps];
    __shared__ __align__(16) float wacc[kMergeWarps][128];
    const int h = blockIdx.x, b = blockIdx.y, k = blockIdx.z, t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    const int L = src.seq_len[b];
    const int hg = a.K > 1 ? a.hg : a.hpk;
    const int grp = src.slot[h / hg];
    float *o = a.out + ((int64_t(b) * a.K + k) * a.n_q + h) * 128;
    float *mlp = a.ml ? a.ml + (int64_t(b) * a.n_q + h) * 2 : nullptr;
    if (grp < 0 || L <= 0) {
        if (t < 128) o[t] = 0.0f;
        if (mlp && t == 0) {
            mlp[0] = -INFINITY;
            mlp[1] = 0.0f;
        }
        return;
    }
    const int64_t unit = int64_t(b) * src.n_live + grp;
    pdl_wait();     // the split kernel's partials are complete
    pdl_trigger();  // the imp pass may start (it reads the split's scores first)
    const int64_t first = a.unit_slots[2 * unit], last = a.unit_slots[2 * unit + 1];
    const int hh = a.K > 1 ? k * hg + h % hg : h % a.hpk;  // the query's row in the partials
    const float *pmh = a.pm + hh, *plh = a.pl + hh, *pah = a.pacc + int64_t(hh) * 128 + 4 * lane;
    float M = -INFINITY, Ls = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int64_t s0 = first + warp; s0 <= last; s0 += kMergeWarps * kMergeBatch) {
        float m[kMergeBatch], pl[kMergeBatch];
        float4 v[kMergeBatch];
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            const int64_t sl = s0 + int64_t(k) * kMergeWarps;
            m[k] = -INFINITY;
            if (sl <= last) {
                m[k] = pmh[sl * a.hpk];
                pl[k] = plh[sl * a.hpk];
                v[k] = *reinterpret_cast<const float4 *>(pah + sl * a.hpk * 128);
            }
        }
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            if (m[k] == -INFINITY) continue;  // past the range, or an empty marker
            if (m[k] > M) {
                const float r = exp2f(M - m[k]);  // 0 while M is -inf
                Ls *= r;
                acc.x *= r;
                acc.y *= r;
                acc.z *= r;
                acc.w *= r;
                M = m[k];
            }
            const float f = exp2f(m[k] - M);
            Ls = fmaf(pl[k], f, Ls);
            acc.x = fmaf(v[k].x, f, acc.x);
            acc.y = fmaf(v[k].y, f, acc.y);
            acc.z = fmaf(v[k].z, f, acc.z);
            acc.w = fmaf(v[k].w, f, acc.w);
        }
    }
    if (lane == 0) wmax[warp] = M;
    __syncthreads();
    float Mall = wmax[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) Mall = fmaxf(Mall, wmax[w]);
    if (Mall == -INFINITY) {  // no visible row (a verify query before every row)
        if (t < 128) o[t] = 0.0f;
        if (mlp && t == 0) {
            mlp[0] = -INFINITY;
            mlp[1] = 0.0f;
        }
        return;
    }
    const float fw = exp2f(M - Mall);  // 0 for a warp that saw no run
    acc.x *= fw;
    acc.y *= fw;
    acc.z *= fw;
    acc.w *= fw;
    *reinterpret_cast<float4 *>(&wacc[warp][4 * lane]) = acc;
    if (lane == 0) wsum[warp] = Ls * fw;
    __syncthreads();
    if (t < 128) {
        float sum = 0.0f, r = 0.0f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            sum += wsum[w];
            r += wacc[w][t];
        }
        if (a.sinks) {
            // a learned sink joins the maximum and the sum; it has no value row
            const float z = a.sinks[h] * kLog2e;
            const float Mf = fmaxf(Mall, z), f = exp2f(Mall - Mf);
            sum = fmaf(sum, f, exp2f(z - Mf));
            r *= f;
            Mall = Mf;
        }
        const float vc = src.vcol ? src.vcol[(int64_t(b) * src.n_live + grp) * 128 + t] : 1.0f;
        o[t] = r / sum * vc;
        if (mlp && t == 0) {
            mlp[0] = Mall;
            mlp[1] = sum;
        }
    }
}

// The same merge with one warp per (sequence, draft, query head), for units
// with few runs: the warp loads the (max, sum, accumulator) of kHeadBatch
// slots at once -- every lane the same maxima and sums, its own four channels
// -- so a unit of up to kHeadBatch slots merges in one round of loads; longer
// ranges go batch by batch under a running maximum.  Slots are taken in
// order, so the result does not depend on timing.
constexpr int kHeadWarps = 4;
constexpr int kHeadBatch = 16;

__global__ void __launch_bounds__(32 * kHeadWarps) merge_heads_kernel(RunMergeArgs a, MergeLayerSrc src) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * kHeadWarps + warp, b = blockIdx.y, k = blockIdx.z;
    if (h >= a.n_q) return;
    const int L = src.seq_len[b];
    const int hg = a.K > 1 ? a.hg : a.hpk;
    const int grp = src.slot[h / hg];
    float4 res = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float Mall = -INFINITY, sum = 0.0f;
    if (grp >= 0 && L > 0) {
        const int64_t unit = int64_t(b) * src.n_live + grp;
        pdl_wait();     // the split kernel's partials are complete
        pdl_trigger();  // the imp pass may start (it reads the split's scores first)
        const int64_t first = a.unit_slots[2 * unit], last = a.unit_slots[2 * unit + 1];
        const int hh = a.K > 1 ? k * hg + h % hg : h % a.hpk;  // the query's row in the partials
        const float *pmh = a.pm + hh, *plh = a.pl + hh, *pah = a.pacc + int64_t(hh) * 128 + 4 * lane;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int64_t s0 = first; s0 <= last; s0 += kHeadBatch) {
            float m[kHeadBatch], pl[kHeadBatch];
            float4 v[kHeadBatch];
#pragma unroll
            for (int j = 0; j < kHeadBatch; ++j) {
                const int64_t sl = s0 + j;
                m[j] = -INFINITY;
                if (sl <= last) {
                    m[j] = pmh[sl * a.hpk];
                    pl[j] = plh[sl * a.hpk];
                    v[j] = *reinterpret_cast<const float4 *>(pah + sl * a.hpk * 128);
                }
            }
            float bm = Mall;
#pragma unroll
            for (int j = 0; j < kHeadBatch; ++j) bm = fmaxf(bm, m[j]);
            if (bm == -INFINITY) continue;  // only empty markers so far
            const float r = exp2f(Mall - bm);  // 0 while Mall is -inf
            sum *= r;
            acc.x *= r;
            acc.y *= r;
            acc.z *= r;
            acc.w *= r;
            Mall = bm;
#pragma unroll
            for (int j = 0; j < kHeadBatch; ++j) {
                if (m[j] == -INFINITY) continue;  // past the range, or an empty marker
                const float f = exp2f(m[j] - Mall);
                sum = fmaf(pl[j], f, sum);
                acc.x = fmaf(v[j].x, f, acc.x);
                acc.y = fmaf(v[j].y, f, acc.y);
                acc.z = fmaf(v[j].z, f, acc.z);
                acc.w = fmaf(v[j].w, f, acc.w);
            }
        }
        if (Mall != -INFINITY) {  // else no visible row (a verify query before every row)
            if (a.sinks) {
                // a learned sink joins the maximum and the sum; it has no value row
                const float z = a.sinks[h] * kLog2e;
                const float Mf = fmaxf(Mall, z), f = exp2f(Mall - Mf);
                sum = fmaf(sum, f, exp2f(z - Mf));
                acc.x *= f;
                acc.y *= f;
                acc.z *= f;
                acc.w *= f;
                Mall = Mf;
            }
            const float4 vc = src.vcol ? reinterpret_cast<const float4 *>(src.vcol + unit * 128)[lane]
                                       : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
            res = make_float4(acc.x / sum * vc.x, acc.y / sum * vc.y, acc.z / sum * vc.z, acc.w / sum * vc.w);
        }
    }
    reinterpret_cast<float4 *>(a.out + ((int64_t(b) * a.K + k) * a.n_q + h) * 128)[lane] = res;
    if (a.ml && lane == 0) {
        float *mlp = a.ml + (int64_t(b) * a.n_q + h) * 2;
        mlp[0] = Mall;
        mlp[1] = sum;
    }
}

// Whether every unit's slot range under the tensor-core work split --
// blocks(u) + c(last tile of u) - c(first tile of u), with c(x) the worker
// holding global tile x (units in sequence-major, live-group order) -- has
// at most `limit` slots.
bool unit_slots_within(const Layer *l, int64_t window, int32_t K, int64_t T, int64_t G, int64_t limit) {
    if (T <= 0 || G <= 0) return true;
    auto worker = [&](int64_t x) { return std::min(((x + 1) * G + T - 1) / T, G) - 1; };
    int64_t t = 0;
    for (int b = 0; b < l->n_seq; ++b) {
        const int64_t Tb = tiles_of(l->h_seq_len[b], window, K);
        if (Tb <= 0) continue;
        for (int gl = 0; gl < l->n_live; ++gl) {
            if (ceil_div(Tb, kBlockTiles) + worker(t + Tb - 1) - worker(t) > limit) return false;
            t += Tb;
        }
    }
    return true;
}

// Merge of the run partials: a warp per query head while every unit has at
// most two batches of slots, else a CTA per query head.
cudaError_t launch_run_merge(const RunMergeArgs &rm, const MergeLayerSrc &ms, int n_seq, int K,
                             bool few_slots, cudaStream_t st) {
    // launched as dependents of the split kernel: their set-up overlaps its tail
    if (few_slots)
        return launch_pdl(merge_heads_kernel, dim3(unsigned(ceil_div(rm.n_q, kHeadWarps)), unsigned(n_seq), unsigned(K)),
                          dim3(32 * kHeadWarps), 0, st, rm, ms);
    return launch_pdl(merge_runs_kernel, dim3(unsigned(rm.n_q), unsigned(n_seq), unsigned(K)), dim3(32 * kMergeWarps),
                      0, st, rm, ms);
}

// ------------------------------------------------------------------ imp

struct ImpArgs {
    const float *scores;  // per (sequence, live group): [hpk][cap] log2 scores
    const float *ml;      // [n_seq][n_q][2]
    float *imp;
    const int64_t *row_base, *cap, *imp_base;
    const int32_t *seq_len, *live;
    int64_t window;  // sliding window in rows (0 = none): rows before the first visible one are untouched
    int32_t n_q, hpk, n_live;
};

// imp[b][p] += sum over the live heads of sequence b of 2^(s - M) / L: the
// softmax weight of every live query head on row p.  A block owns 256 rows of
// one sequence: it stages the (max, 1/sum) of the sequence's live heads in
// shared memory (in live order, head i = gl * hpk + hh) while its threads, 64
// row quads x 4 head classes (i mod 4), already load their scores (one
// 16-byte load per head: a unit's scores start on a 16-row boundary and its
// capacity is a multiple of 16 rows) and the old imp values, so those loads
// overlap.  The four classes' sums are added in a fixed order.
constexpr int kImpThreads = 256;
constexpr int kImpRows = 256;   // rows per block
constexpr int kImpClasses = 4;  // head classes per row quad
constexpr int kImpBatch = 8;    // score loads in flight per thread

__global__ void __launch_bounds__(kImpThreads) imp_kernel(ImpArgs a) {
    extern __shared__ float mlinv[];  // [n_live * hpk][2]: max, 1/sum
    __shared__ __align__(16) float part[kImpClasses][kImpRows];
    const int b = blockIdx.y, t = threadIdx.x;
    const int L = a.seq_len[b];
    // blocks cover the visible rows, from the first one rounded down to 16
    const int first = int(first_visible(L, a.window));
    const int p0 = first / kRowAlign * kRowAlign + blockIdx.x * kImpRows;
    if (p0 >= L) return;
    const int nh = a.n_live * a.hpk;
    const int64_t cap = a.cap[b];
    const int quad = t % (kImpRows / 4), cls = t / (kImpRows / 4);
    const int p = p0 + 4 * quad;
    const int r = p0 + t;
    const bool mine = r < L && r >= first;
    float *dst = a.imp + a.imp_base[b] + r;
    const float old = mine ? *dst : 0.0f;
    // the scores of live head i start at row_base * hpk + i * cap
    const float *sb = a.scores + a.row_base[b] * a.hpk + p;
    float add[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float4 sv[kImpBatch];
    auto load = [&](int i0) {
#pragma unroll
        for (int k = 0; k < kImpBatch; ++k) {
            const int i = i0 + k * kImpClasses;
            if (p < L && i < nh) sv[k] = *reinterpret_cast<const float4 *>(sb + int64_t(i) * cap);
        }
    };
    load(cls);  // the first batch (scores of the finished split kernel) is in flight across the wait
    pdl_wait();     // the merge's maxima and sums are complete
    pdl_trigger();  // the next append may be scheduled (it waits for this grid)
    for (int i = t; i < nh; i += kImpThreads) {
        const int h = a.live[i / a.hpk] * a.hpk + i % a.hpk;
        const float M = a.ml[(int64_t(b) * a.n_q + h) * 2];
        const float Ls = a.ml[(int64_t(b) * a.n_q + h) * 2 + 1];
        mlinv[2 * i] = M;
        mlinv[2 * i + 1] = Ls > 0.0f ? 1.0f / Ls : 0.0f;
    }
    __syncthreads();  // the staged maxima and sums are visible
    for (int i0 = cls; i0 < nh; i0 += kImpClasses * kImpBatch) {
        if (i0 != cls) load(i0);
#pragma unroll
        for (int k = 0; k < kImpBatch; ++k) {
            const int i = i0 + k * kImpClasses;
            if (p < L && i < nh) {
                const float M = mlinv[2 * i], il = mlinv[2 * i + 1];
                add[0] += exp2f(sv[k].x - M) * il;
                add[1] += exp2f(sv[k].y - M) * il;
                add[2] += exp2f(sv[k].z - M) * il;
                add[3] += exp2f(sv[k].w - M) * il;
            }
        }
    }
    *reinterpret_cast<float4 *>(&part[cls][4 * quad]) = make_float4(add[0], add[1], add[2], add[3]);
    __syncthreads();
    if (mine) *dst = old + ((part[0][t] + part[1][t]) + (part[2][t] + part[3][t]));
}

// ---------------------------------------------------------------- R-SWA copies

struct RingWriteTable {
    int32_t s0, n;
    int32_t slot[kSlice];
};

// Stream s0 + i copies its token's H rows of K and V into ring slot slot[i].
__global__ void ring_write_kernel(float *ring_k, float *ring_v, const float *k, const float *v,
                                  int32_t H, int32_t hd, int32_t W, RingWriteTable t) {
    const int i = blockIdx.y;
    if (i >= t.n) return;
    const int s = t.s0 + i;
    const int64_t per = int64_t(H) * hd;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < per;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = e / hd, d = e % hd;
        const int64_t dst = ((int64_t(s) * H + h) * W + t.slot[i]) * hd + d;
        ring_k[dst] = k[int64_t(s) * per + e];
        ring_v[dst] = v[int64_t(s) * per + e];
    }
}

// Copy a [H][seq][hd] prefill into the reference block of stream s.
__global__ void prefill_copy_kernel(float *ref_k, float *ref_v, const float *k, const float *v,
                                    int32_t s, int32_t seq, int32_t H, int32_t hd,
                                    int64_t ref_cap) {
    const int64_t per_head = int64_t(seq) * hd;
    const int64_t total = per_head * H;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = e / per_head, r = e % per_head;
        const int64_t dst = (int64_t(s) * H + h) * ref_cap * hd + r;
        ref_k[dst] = k[e];
        ref_v[dst] = v[e];
    }
}

// rswa quantize_row_i8 of one HD-value row by one warp (lane = CPL
// consecutive values): codes and the row scale, with the f32 row copied to
// `copy` on the way.
template <int HD>
__device__ __forceinline__ void quant_row_i8_warp(const float *x, float *copy, int8_t *codes,
                                                  float *scale, int lane) {
    constexpr int CPL = HD / 32;
    float v[CPL];
    if (CPL == 4) {
        const float4 f = reinterpret_cast<const float4 *>(x)[lane];
        reinterpret_cast<float4 *>(copy)[lane] = f;
        v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
    } else {
        const float2 f = reinterpret_cast<const float2 *>(x)[lane];
        reinterpret_cast<float2 *>(copy)[lane] = f;
        v[0] = f.x, v[1] = f.y;
    }
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) mx = fmaxf(mx, fabsf(v[j]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float sc = mx > 0.0f ? __fdiv_rn(mx, 127.0f) : 1.0f;
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < CPL; ++j) w |= (uint32_t(quant_code_i8(v[j], sc)) & 0xffu) << (8 * j);
    if (CPL == 4) reinterpret_cast<uint32_t *>(codes)[lane] = w;
    else reinterpret_cast<uint16_t *>(codes)[lane] = uint16_t(w);
    if (lane == 0) *scale = sc;
}

// record_prefill with the int8 mirror: one warp per (head, row) of stream s
// copies the K and V rows and writes their codes and scales.
template <int HD>
__global__ void prefill_i8_kernel(float *ref_k, float *ref_v, rswa_i8_mirror m, const float *k,
                                  const float *v, int32_t s, int32_t seq, int32_t H, int64_t ref_cap) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = int64_t(H) * seq;
    for (int64_t w = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; w < rows;
         w += (int64_t(gridDim.x) * blockDim.x) >> 5) {
        const int64_t h = w / seq, r = w % seq;
        const int64_t dst = (int64_t(s) * H + h) * ref_cap + r;
        quant_row_i8_warp<HD>(k + w * HD, ref_k + dst * HD, m.ref_k + dst * HD, m.ref_ks + dst, lane);
        quant_row_i8_warp<HD>(v + w * HD, ref_v + dst * HD, m.ref_v + dst * HD, m.ref_vs + dst, lane);
    }
}

// write_decode_step with the int8 mirror: one warp per (stream, head).
template <int HD>
__global__ void ring_write_i8_kernel(float *ring_k, float *ring_v, rswa_i8_mirror m, const float *k,
                                     const float *v, int32_t H, int32_t W, RingWriteTable t) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = int64_t(t.n) * H;
    for (int64_t w = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; w < rows;
         w += (int64_t(gridDim.x) * blockDim.x) >> 5) {
        const int i = int(w / H), h = int(w % H);
        const int64_t src = (int64_t(t.s0 + i) * H + h) * HD;
        const int64_t dst = (int64_t(t.s0 + i) * H + h) * W + t.slot[i];
        quant_row_i8_warp<HD>(k + src, ring_k + dst * HD, m.ring_k + dst * HD, m.ring_ks + dst, lane);
        quant_row_i8_warp<HD>(v + src, ring_v + dst * HD, m.ring_v + dst * HD, m.ring_vs + dst, lane);
    }
}

template <int HD, bool I8, int HPK = 1>
cudaError_t launch_split_rswa(const SplitArgs &a, const RswaSrc &s, const RswaTable &t, dim3 grid,
                              cudaStream_t st) {
    using C = SplitCfg<HD, HPK, I8, I8, I8>;
    auto kern = split_rswa_kernel<HD, I8, HPK>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM, st>>>(a, s, t);
    return launch_status();
}

template <int HD, bool I8>
cudaError_t launch_split_rswa_k(int hb, const SplitArgs &a, const RswaSrc &s, const RswaTable &t, dim3 grid,
                                cudaStream_t st) {
    switch (hb) {
        case 1: return launch_split_rswa<HD, I8, 1>(a, s, t, grid, st);
        case 2: return launch_split_rswa<HD, I8, 2>(a, s, t, grid, st);
        case 4: return launch_split_rswa<HD, I8, 4>(a, s, t, grid, st);
        case 8: return launch_split_rswa<HD, I8, 8>(a, s, t, grid, st);
        case 16: return launch_split_rswa<HD, I8, 16>(a, s, t, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

// rswa verify_attention, the ring-and-drafts part: query i of a head sees the
// live ring rows and drafts 0..i that survive in the last W written rows --
// the ring in logical order (oldest at slot rp0) followed by the drafts; the
// reference rows are the split kernel's.  One CTA per (query, head, stream),
// four warps over the candidate rows, each warp an online softmax with the
// score of a row complete in every lane, then combined; the result is written
// as one more chunk partial (slot nc_ref) for the merge.
struct TailTable {
    int32_t s0, n;
    int32_t ring_len[kSlice];
    int32_t rp0[kSlice];     // slot of the oldest live ring row
    int32_t nc_ref[kSlice];  // chunk partials of the reference rows
};

struct TailArgs {
    const float *q, *dk, *dv;         // [B][K][H][HD]
    const float *ring_k, *ring_v;     // f32 ring (I8 false)
    const int8_t *ring_k8, *ring_v8;  // mirror codes (I8)
    const float *ring_ks, *ring_vs;   // mirror scales (I8)
    float *pm, *pl, *pacc;
    int32_t K, H, W, nc_max;
    float qscale;  // softmax scale * log2(e)
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// quantize_row_i8 of a row held CPL values per lane: codes packed per lane, scale returned
template <int CPL>
__device__ __forceinline__ uint32_t quant_lane_i8(const float (&x)[CPL], float &scale) {
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) mx = fmaxf(mx, fabsf(x[j]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    scale = mx > 0.0f ? __fdiv_rn(mx, 127.0f) : 1.0f;
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < CPL; ++j) w |= (uint32_t(quant_code_i8(x[j], scale)) & 0xffu) << (8 * j);
    return w;
}

template <int CPL>
__device__ __forceinline__ void load_f32_lane(const float *row, int lane, float (&x)[CPL]) {
    if (CPL == 4) {
        const float4 f = reinterpret_cast<const float4 *>(row)[lane];
        x[0] = f.x, x[1] = f.y, x[2] = f.z, x[3] = f.w;
    } else {
        const float2 f = reinterpret_cast<const float2 *>(row)[lane];
        x[0] = f.x, x[1] = f.y;
    }
}

struct RswaRunMerge {
    const float *pm, *pl, *pacc;     // run partials [slot][K] (+ [128])
    const int64_t *unit_slots;       // [stream of the launch][H][2]
    float *out;                      // [B][K][H][128]
    int32_t H, K;
};

// FUSED (the tensor-core path, head_dim 128): the kernel is the split kernel's
// programmatic dependent, computes the ring-and-drafts partial while the split
// drains, then waits for it and merges the partial with the head's run
// partials (t.nc_ref[si] = 1 if stream si has a reference block), writing out.
template <int HD, bool I8, bool FUSED = false>
__global__ void __launch_bounds__(128) rswa_verify_tail_kernel(TailArgs a, TailTable t, RswaRunMerge rm) {
    constexpr int CPL = HD / 32;
    __shared__ float sm_m[4], sm_l[4];
    __shared__ float sm_acc[4][HD];
    const int i = blockIdx.x, h = blockIdx.y, si = blockIdx.z;
    if (si >= t.n) return;
    const int s = t.s0 + si;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rl = t.ring_len[si], rp0 = t.rp0[si];
    const int drop = max(0, rl + i + 1 - a.W);  // oldest rows pushed out by drafts 0..i
    float qv[CPL];
    load_f32_lane<CPL>(a.q + ((int64_t(s) * a.K + i) * a.H + h) * HD, lane, qv);
    uint32_t qi = 0;
    float qfac = 0.0f;
    if (I8) {
        float sq;
        qi = quant_lane_i8<CPL>(qv, sq);
        qfac = sq * a.qscale;
    } else {
#pragma unroll
        for (int j = 0; j < CPL; ++j) qv[j] *= a.qscale;
    }
    float m = -INFINITY, l = 0.0f, acc[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) acc[j] = 0.0f;
    // one row into the warp's online softmax (score and weight scale uniform
    // over the warp, x this lane's CPL values)
    auto add_row = [&](float score, float w_scale, const float (&x)[CPL]) {
        const float mn = fmaxf(m, score);
        const float al = m == -INFINITY ? 0.0f : exp2f(m - mn);
        const float e = exp2f(score - mn);
        l = l * al + e;
        const float w = e * w_scale;
#pragma unroll
        for (int jj = 0; jj < CPL; ++jj) acc[jj] = fmaf(acc[jj], al, w * x[jj]);
        m = mn;
    };
    const int64_t ring0 = (int64_t(s) * a.H + h) * a.W;  // row of slot 0 of this head's ring
    // Ring rows, warp-strided, kTB rows per batch: every load of a batch is
    // issued before its first row is used, so the rows' latencies overlap.
    constexpr int kTB = 8;
    for (int r0 = warp; r0 < rl; r0 += 4 * kTB) {
        bool vis[kTB];
        uint32_t kw[kTB], vw[kTB];
        float ksr[kTB], vsr[kTB];
        float kx[I8 ? 1 : kTB][CPL], vx[I8 ? 1 : kTB][CPL];
#pragma unroll
        for (int u = 0; u < kTB; ++u) {
            const int r = r0 + 4 * u;
            vis[u] = r < rl && ((r - rp0 + a.W) % a.W) >= drop;  // the same for the whole warp
            if (!vis[u]) continue;
            if constexpr (I8) {
                const int8_t *kr = a.ring_k8 + (ring0 + r) * HD;
                const int8_t *vr = a.ring_v8 + (ring0 + r) * HD;
                kw[u] = CPL == 4 ? reinterpret_cast<const uint32_t *>(kr)[lane]
                                 : uint32_t(reinterpret_cast<const uint16_t *>(kr)[lane]);
                vw[u] = CPL == 4 ? reinterpret_cast<const uint32_t *>(vr)[lane]
                                 : uint32_t(reinterpret_cast<const uint16_t *>(vr)[lane]);
                ksr[u] = a.ring_ks[ring0 + r];
                vsr[u] = a.ring_vs[ring0 + r];
            } else {
                load_f32_lane<CPL>(a.ring_k + (ring0 + r) * HD, lane, kx[u]);
                load_f32_lane<CPL>(a.ring_v + (ring0 + r) * HD, lane, vx[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kTB; ++u) {
            if (!vis[u]) continue;
            float x[CPL];
            if constexpr (I8) {
                // exact integer dot (every partial sum an integer below 2^24)
                const float score = warp_sum(float(__dp4a(int(qi), int(kw[u]), 0))) * ksr[u] * qfac;
#pragma unroll
                for (int jj = 0; jj < CPL; ++jj) x[jj] = float(int8_t((vw[u] >> (8 * jj)) & 0xffu));
                add_row(score, vsr[u], x);
            } else {
                float p = 0.0f;
#pragma unroll
                for (int jj = 0; jj < CPL; ++jj) p = fmaf(qv[jj], kx[u][jj], p);
#pragma unroll
                for (int jj = 0; jj < CPL; ++jj) x[jj] = vx[u][jj];
                add_row(warp_sum(p), 1.0f, x);
            }
        }
    }
    // drafts 0..i (the int8 path quantises each like a cache row first)
    for (int j = warp; j <= i; j += 4) {
        if (rl + j < drop) continue;  // pushed out of the window (the same for the whole warp)
        const float *drow_k = a.dk + ((int64_t(s) * a.K + j) * a.H + h) * HD;
        const float *drow_v = a.dv + ((int64_t(s) * a.K + j) * a.H + h) * HD;
        float kx[CPL], x[CPL];
        load_f32_lane<CPL>(drow_k, lane, kx);
        load_f32_lane<CPL>(drow_v, lane, x);
        if constexpr (I8) {
            float ks, w_scale;
            const uint32_t kw = quant_lane_i8<CPL>(kx, ks);
            const float score = warp_sum(float(__dp4a(int(qi), int(kw), 0))) * ks * qfac;
            const uint32_t vw = quant_lane_i8<CPL>(x, w_scale);
#pragma unroll
            for (int jj = 0; jj < CPL; ++jj) x[jj] = float(int8_t((vw >> (8 * jj)) & 0xffu));
            add_row(score, w_scale, x);
        } else {
            float p = 0.0f;
#pragma unroll
            for (int jj = 0; jj < CPL; ++jj) p = fmaf(qv[jj], kx[jj], p);
            add_row(warp_sum(p), 1.0f, x);
        }
    }
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
#pragma unroll
    for (int jj = 0; jj < CPL; ++jj) sm_acc[warp][lane * CPL + jj] = acc[jj];
    __syncthreads();
    float M = fmaxf(fmaxf(sm_m[0], sm_m[1]), fmaxf(sm_m[2], sm_m[3]));
    if constexpr (FUSED) {
        static_assert(HD == 128, "one thread per channel");
        const int d = threadIdx.x;
        float Ls = 0.0f, A = 0.0f;
        for (int w2 = 0; w2 < 4; ++w2) {
            const float f = sm_m[w2] == -INFINITY ? 0.0f : exp2f(sm_m[w2] - M);
            Ls += sm_l[w2] * f;
            A += sm_acc[w2][d] * f;
        }
        pdl_wait();  // the split kernel's run partials are complete and visible
        if (t.nc_ref[si] > 0) {
            const int64_t unit = int64_t(si) * rm.H + h;
            const int64_t first = rm.unit_slots[2 * unit], last = rm.unit_slots[2 * unit + 1];
            constexpr int kBatch = 8;  // slots whose loads are in flight together
            for (int64_t s0 = first; s0 <= last; s0 += kBatch) {
                float mk[kBatch], lk[kBatch], vk[kBatch];
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int64_t p = (s0 + k) * rm.K + i;
                    mk[k] = -INFINITY;
                    if (s0 + k <= last) {
                        mk[k] = rm.pm[p];
                        lk[k] = rm.pl[p];
                        vk[k] = rm.pacc[p * 128 + d];
                    }
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    if (mk[k] == -INFINITY) continue;  // past the range, or an empty marker
                    if (mk[k] > M) {
                        const float r = exp2f(M - mk[k]);
                        Ls *= r;
                        A *= r;
                        M = mk[k];
                    }
                    const float f = exp2f(mk[k] - M);
                    Ls = fmaf(lk[k], f, Ls);
                    A = fmaf(vk[k], f, A);
                }
            }
        }
        rm.out[((int64_t(s) * rm.K + i) * rm.H + h) * 128 + d] = A / Ls;
        return;
    }
    const int64_t p = ((int64_t(s) * a.H + h) * a.nc_max + t.nc_ref[si]) * a.K + i;
    for (int d = threadIdx.x; d < HD; d += blockDim.x) {
        float L = 0.0f, A = 0.0f;
        for (int w2 = 0; w2 < 4; ++w2) {
            const float f = sm_m[w2] == -INFINITY ? 0.0f : exp2f(sm_m[w2] - M);
            L += sm_l[w2] * f;
            A += sm_acc[w2][d] * f;
        }
        a.pacc[p * HD + d] = A;
        if (d == 0) {
            a.pm[p] = M;
            a.pl[p] = L;
        }
    }
}

// The stream tables the tensor-core kernel walks, for the streams of one
// launch: stream si is "sequence" si with prefill_len rows per head, its
// H heads the live groups (identity map), head h's block at row
// ((s0 + si) H + h) ref_cap of the mirror.
struct RswaTcTables {
    int32_t *seq_len, *live;
    int64_t *cap, *row_base;
    int32_t H;
    int64_t ref_cap;
};

__global__ void rswa_tc_tables_kernel(RswaTable tb, RswaTcTables t) {
    for (int i = threadIdx.x; i < tb.n || i < t.H; i += blockDim.x) {
        if (i < tb.n) {
            t.seq_len[i] = tb.prefill_len[i];
            t.cap[i] = t.ref_cap;
            t.row_base[i] = (int64_t(tb.s0) + i) * t.H * t.ref_cap;
        }
        if (i < t.H) t.live[i] = i;
    }
}


bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_decode_workspace_bytes(const kvd_layer *L, int32_t n_q, int32_t with_imp,
                                                 int64_t *bytes_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || bytes_out == nullptr) return KVD_EINVAL;
    if (n_q < l->n_kv || n_q % l->n_kv != 0 || n_q / l->n_kv > kMaxHpk) return KVD_EINVAL;
    const int64_t total = decode_ws(l, n_q, with_imp != 0).total;
    if (total < 0) return KVD_ECUDA;
    *bytes_out = total;
    return KVD_OK;
}

extern "C" kvd_status decode_attention(const float *q, const kvd_layer *L, int32_t n_q, float scale,
                                       float *out, float *imp, void *workspace,
                                       int64_t workspace_bytes, void *stream) {
    KVD_NVTX_RANGE("decode_attention");
    return decode_attention_ex(q, L, n_q, scale, 0, 0.0f, nullptr, out, imp, workspace, workspace_bytes,
                               stream);
}

extern "C" kvd_status decode_attention_ex(const float *q, const kvd_layer *L, int32_t n_q, float scale,
                                          int64_t window, float softcap, const float *sinks, float *out,
                                          float *imp, void *workspace, int64_t workspace_bytes,
                                          void *stream) {
    KVD_NVTX_RANGE("decode_attention_ex");
    const Layer *l = checked_layer(L);
    if (l == nullptr || q == nullptr || out == nullptr) return KVD_EINVAL;
    if (n_q < l->n_kv || n_q % l->n_kv != 0 || n_q / l->n_kv > kMaxHpk) return KVD_EINVAL;
    if (!std::isfinite(scale)) return KVD_EINVAL;
    if (window < 0 || !std::isfinite(softcap) || softcap < 0.0f) return KVD_EINVAL;
    if (!aligned16(q) || !aligned16(out) || (imp && (reinterpret_cast<uintptr_t>(imp) & 3)) ||
        (sinks && (reinterpret_cast<uintptr_t>(sinks) & 3)))
        return KVD_EINVAL;
    const DecodeWs w = decode_ws(l, n_q, imp != nullptr);
    if (w.total < 0) return KVD_ECUDA;
    if (workspace == nullptr || workspace_bytes < w.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return KVD_EINVAL;
    const int hpk = n_q / l->n_kv;
    cudaStream_t st = as_stream(stream);
    char *ws = static_cast<char *>(workspace);

    // rows from each sequence's first visible row rounded down to kRowAlign
    int64_t work = 0, max_len = 0;
    for (int b = 0; b < l->n_seq; ++b) {
        const int64_t Lb = l->h_seq_len[b];
        const int64_t vis = Lb - first_visible(Lb, window) / kRowAlign * kRowAlign;
        work += vis * int64_t(l->n_live);
        max_len = std::max(max_len, vis);
    }
    const int32_t chunk = pick_chunk(work);

    SplitArgs a;
    a.q = q;
    a.n_q = n_q;
    a.hpk = hpk;
    a.qscale = scale * kLog2e;
    a.chunk = chunk;
    a.nc_max = w.nc_max;
    a.n_grp = std::max(1, l->n_live);
    a.pm = reinterpret_cast<float *>(ws + w.pm);
    a.pl = reinterpret_cast<float *>(ws + w.pl);
    a.pacc = reinterpret_cast<float *>(ws + w.pacc);
    a.scores = imp ? reinterpret_cast<float *>(ws + w.scores) : nullptr;
    a.err = l->d_err;
    a.window = window;
    a.softcap2 = softcap * kLog2e;

    LayerSrc s;
    s.kf = static_cast<const float *>(l->buf[KVD_BUF_K]);
    s.vf = static_cast<const float *>(l->buf[KVD_BUF_V]);
    s.kq = static_cast<const int8_t *>(l->buf[KVD_BUF_KQ]);
    s.vq = static_cast<const int8_t *>(l->buf[KVD_BUF_VQ]);
    s.ks = static_cast<const float *>(l->buf[KVD_BUF_KS]);
    s.vs = static_cast<const float *>(l->buf[KVD_BUF_VS]);
    s.kcol = static_cast<const float *>(l->buf[KVD_BUF_KCOL]);
    s.row_base = l->d_row_base;
    s.cap = l->d_cap;
    s.seq_len = l->d_seq_len;
    s.live = l->d_live;
    s.n_live = l->n_live;
    MergeLayerSrc ms;
    ms.seq_len = l->d_seq_len;
    ms.slot = l->d_slot;
    ms.vcol = static_cast<const float *>(l->buf[KVD_BUF_VCOL]);
    ms.n_live = l->n_live;
    float *ml = imp ? reinterpret_cast<float *>(ws + w.ml) : nullptr;

    if (warp_path(l)) {
        // tensor-core kernel over balanced tile ranges, then the run merge
        int64_t T = 0;
        for (int b = 0; b < l->n_seq; ++b) T += int64_t(l->n_live) * tiles_of(l->h_seq_len[b], window);
        const int variant = q8_tc_variant(hpk);
        const int64_t workers = split_q8_tc_workers(variant);
        if (workers <= 0) return KVD_ECUDA;
        WarpArgs wa;
        wa.a = a;
        wa.T = T;
        wa.G = int32_t(std::min(T, workers));
        wa.n_seq = l->n_seq;
        wa.unit_slots = reinterpret_cast<int64_t *>(ws + w.units);
        if (T > 0) {
            MmaMaps maps;
            std::memcpy(&maps.kq, l->tmap_kq, sizeof(maps.kq));
            std::memcpy(&maps.vq, l->tmap_vq, sizeof(maps.vq));
            if (split_layer_q8_tc(variant, wa, s, maps, st) != cudaSuccess) return KVD_ECUDA;
        }
        RunMergeArgs rm;
        rm.pm = a.pm;
        rm.pl = a.pl;
        rm.pacc = a.pacc;
        rm.out = out;
        rm.ml = ml;
        rm.n_q = n_q;
        rm.hpk = hpk;
        rm.unit_slots = wa.unit_slots;
        rm.sinks = sinks;
        const bool few = unit_slots_within(l, window, 1, T, wa.G, 2 * kHeadBatch);
        if (launch_run_merge(rm, ms, l->n_seq, 1, few, st) != cudaSuccess) return KVD_ECUDA;
    } else {
        if (max_len > 0 && l->n_live > 0) {
            dim3 grid(unsigned(ceil_div(max_len, chunk)), unsigned(l->n_live), unsigned(l->n_seq));
            const int hb = hpk_bucket(hpk);
            cudaError_t e;
            switch (l->mode) {
                case KVD_F32: e = split_layer_f32(l->hd, hb, a, s, grid, st); break;
                case KVD_Q8: e = split_layer_q8(l->hd, hb, a, s, grid, st); break;
                case KVD_Q8K: e = split_layer_q8k(l->hd, hb, a, s, grid, st); break;
                default: e = split_layer_q8v(l->hd, hb, a, s, grid, st); break;
            }
            if (e != cudaSuccess) return KVD_ECUDA;
        }
        MergeArgs m;
        m.pm = a.pm;
        m.pl = a.pl;
        m.pacc = a.pacc;
        m.out = out;
        m.ml = ml;
        m.n_q = n_q;
        m.hpk = hpk;
        m.n_grp = a.n_grp;
        m.nc_max = w.nc_max;
        m.chunk = chunk;
        m.sinks = sinks;
        m.window = window;
        dim3 mgrid(unsigned(n_q), unsigned(l->n_seq));
        if (l->hd == 128) merge_layer_kernel<128><<<mgrid, 128, 0, st>>>(m, ms);
        else merge_layer_kernel<64><<<mgrid, 64, 0, st>>>(m, ms);
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }

    if (imp && max_len > 0 && l->n_live > 0) {
        ImpArgs ia;
        ia.scores = a.scores;
        ia.ml = ml;
        ia.imp = imp;
        ia.row_base = l->d_row_base;
        ia.cap = l->d_cap;
        ia.imp_base = reinterpret_cast<const int64_t *>(
            static_cast<const char *>(l->buf[KVD_BUF_META]) + l->ml.imp_base);
        ia.seq_len = l->d_seq_len;
        ia.live = l->d_live;
        ia.n_q = n_q;
        ia.hpk = hpk;
        ia.n_live = l->n_live;
        ia.window = window;
        dim3 igrid(unsigned(ceil_div(max_len, kImpRows)), unsigned(l->n_seq));
        const size_t ml_bytes = size_t(std::max(1, l->n_live * hpk)) * 2 * sizeof(float);
        if (ml_bytes > 40 * 1024 &&
            set_smem_once(reinterpret_cast<const void *>(imp_kernel), int(ml_bytes)) != cudaSuccess)
            return KVD_ECUDA;
        // a dependent of the merge: its score loads overlap the merge
        if (launch_pdl(imp_kernel, igrid, dim3(kImpThreads), ml_bytes, st, ia) != cudaSuccess) return KVD_ECUDA;
    }
    return KVD_OK;
}

// ------------------------------------------------------------ bounds self-test

namespace kvd {
namespace {

// Scratch of kvd_bounds_selftest: two copies of fake lengths, fake frozen
// flags, zero input rows for the append, and room for the partials and slot
// records the split launches are given (they write none: their guards return
// first).
struct BoundsWs {
    int64_t len, frozen, zeros, part, total;
};

BoundsWs bounds_ws(const Layer *l) {
    BoundsWs w;
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.len = take(int64_t(l->n_seq) * 2 * 4);
    w.frozen = take(int64_t(l->n_seq) * 4);
    w.zeros = take(int64_t(l->n_kv) * l->hd * 4);
    w.part = take(int64_t(kMaxHpk) * (2 + l->hd) * 4 + 256);
    w.total = o;
    return w;
}

}  // namespace
}  // namespace kvd

extern "C" kvd_status kvd_bounds_selftest_bytes(const kvd_layer *L, int64_t *bytes_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || bytes_out == nullptr) return KVD_EINVAL;
    *bytes_out = bounds_ws(l).total;
    return KVD_OK;
}

extern "C" kvd_status kvd_bounds_selftest(const kvd_layer *L, void *scratch, int64_t scratch_bytes,
                                          void *stream) {
    KVD_NVTX_RANGE("kvd_bounds_selftest");
    const Layer *l = checked_layer(L);
    if (l == nullptr || scratch == nullptr || l->n_seq < 1 || l->n_live < 1) return KVD_EINVAL;
    if (l->h_cap[0] >= (int64_t(1) << 31) - 1) return KVD_EINVAL;
    if (reinterpret_cast<uintptr_t>(scratch) & 255) return KVD_EINVAL;
    const BoundsWs w = bounds_ws(l);
    if (scratch_bytes < w.total) return KVD_ECAPACITY;
    char *ws = static_cast<char *>(scratch);
    cudaStream_t st = as_stream(stream);
    // fake lengths: sequence 0 one row past its capacity, the others as stored
    std::vector<int32_t> len(size_t(l->n_seq) * 2);
    for (int b = 0; b < l->n_seq; ++b) len[b] = len[l->n_seq + b] = int32_t(l->h_seq_len[b]);
    len[0] = int32_t(l->h_cap[0] + 1);
    if (cudaMemcpyAsync(ws + w.len, len.data(), len.size() * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemsetAsync(ws + w.frozen, 0, size_t(l->n_seq) * 4, st) != cudaSuccess ||
        cudaMemsetAsync(ws + w.zeros, 0, size_t(l->n_kv) * l->hd * 4, st) != cudaSuccess || fault_fires())
        return KVD_ECUDA;
    int32_t *fake_len = reinterpret_cast<int32_t *>(ws + w.len);
    const float *zeros = reinterpret_cast<const float *>(ws + w.zeros);
    if (append_bounds_selftest(l, zeros, fake_len, reinterpret_cast<int32_t *>(ws + w.frozen), st) != cudaSuccess)
        return KVD_ECUDA;

    // the decode's split kernel over the fake lengths: one CTA (CUDA-core
    // path) or one worker over one tile (tensor-core path), both on
    // sequence 0, whose guard returns before any read of the cache
    SplitArgs a;
    a.q = zeros;
    a.n_q = l->n_kv;
    a.hpk = 1;
    a.qscale = kLog2e;
    a.chunk = kMinChunk;
    a.nc_max = 1;
    a.n_grp = l->n_live;
    a.pm = reinterpret_cast<float *>(ws + w.part);
    a.pl = a.pm + kMaxHpk;
    a.pacc = a.pl + kMaxHpk;
    a.scores = nullptr;
    a.err = l->d_err;
    LayerSrc s;
    s.kf = static_cast<const float *>(l->buf[KVD_BUF_K]);
    s.vf = static_cast<const float *>(l->buf[KVD_BUF_V]);
    s.kq = static_cast<const int8_t *>(l->buf[KVD_BUF_KQ]);
    s.vq = static_cast<const int8_t *>(l->buf[KVD_BUF_VQ]);
    s.ks = static_cast<const float *>(l->buf[KVD_BUF_KS]);
    s.vs = static_cast<const float *>(l->buf[KVD_BUF_VS]);
    s.kcol = static_cast<const float *>(l->buf[KVD_BUF_KCOL]);
    s.row_base = l->d_row_base;
    s.cap = l->d_cap;
    s.seq_len = fake_len;
    s.live = l->d_live;
    s.n_live = l->n_live;
    if (warp_path(l)) {
        WarpArgs wa;
        wa.a = a;
        wa.T = 1;
        wa.G = 1;
        wa.n_seq = l->n_seq;
        wa.unit_slots = reinterpret_cast<int64_t *>(a.pacc + kMaxHpk * l->hd);
        MmaMaps maps;
        std::memcpy(&maps.kq, l->tmap_kq, sizeof(maps.kq));
        std::memcpy(&maps.vq, l->tmap_vq, sizeof(maps.vq));
        if (split_layer_q8_tc(q8_tc_variant(1), wa, s, maps, st) != cudaSuccess) return KVD_ECUDA;
    } else {
        const dim3 grid(1, 1, 1);
        cudaError_t e;
        switch (l->mode) {
            case KVD_F32: e = split_layer_f32(l->hd, 1, a, s, grid, st); break;
            case KVD_Q8: e = split_layer_q8(l->hd, 1, a, s, grid, st); break;
            case KVD_Q8K: e = split_layer_q8k(l->hd, 1, a, s, grid, st); break;
            default: e = split_layer_q8v(l->hd, 1, a, s, grid, st); break;
        }
        if (e != cudaSuccess) return KVD_ECUDA;
    }
    return KVD_OK;
}

// ------------------------------------------------------------ verify

extern "C" kvd_status kvd_verify_workspace_bytes(const kvd_layer *L, int32_t n_q, int32_t K,
                                                 int64_t *bytes_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || bytes_out == nullptr || K < 1) return KVD_EINVAL;
    if (n_q < l->n_kv || n_q % l->n_kv != 0 || int64_t(n_q / l->n_kv) * K > kMaxHpk) return KVD_EINVAL;
    const DecodeWs w = decode_ws(l, n_q * K, false);
    if (w.total < 0) return KVD_ECUDA;
    *bytes_out = w.total;
    return KVD_OK;
}

extern "C" kvd_status decode_attention_verify(const float *q, const kvd_layer *L, int32_t n_q, int32_t K,
                                              float scale, int64_t window, float softcap, const float *sinks,
                                              float *out, void *workspace, int64_t workspace_bytes,
                                              void *stream) {
    KVD_NVTX_RANGE("decode_attention_verify");
    const Layer *l = checked_layer(L);
    if (l == nullptr || q == nullptr || out == nullptr || K < 1) return KVD_EINVAL;
    if (n_q < l->n_kv || n_q % l->n_kv != 0 || int64_t(n_q / l->n_kv) * K > kMaxHpk) return KVD_EINVAL;
    if (!std::isfinite(scale)) return KVD_EINVAL;
    if (window < 0 || !std::isfinite(softcap) || softcap < 0.0f) return KVD_EINVAL;
    if (!aligned16(q) || !aligned16(out) || (sinks && (reinterpret_cast<uintptr_t>(sinks) & 3)))
        return KVD_EINVAL;
    const int hg = n_q / l->n_kv, hpk = hg * K;
    const DecodeWs w = decode_ws(l, n_q * K, false);
    if (w.total < 0) return KVD_ECUDA;
    if (workspace == nullptr || workspace_bytes < w.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return KVD_EINVAL;
    cudaStream_t st = as_stream(stream);
    char *ws = static_cast<char *>(workspace);
    int64_t work = 0, max_len = 0;
    for (int b = 0; b < l->n_seq; ++b) {
        const int64_t Lb = l->h_seq_len[b];
        const int64_t vis = Lb - first_visible(verify_len(Lb, K), window) / kRowAlign * kRowAlign;
        work += vis * int64_t(l->n_live);
        max_len = std::max(max_len, vis);
    }
    const int32_t chunk = pick_chunk(work);
    SplitArgs a;
    a.q = q;
    a.n_q = n_q;
    a.hpk = hpk;
    a.qscale = scale * kLog2e;
    a.chunk = chunk;
    a.nc_max = w.nc_max;
    a.n_grp = std::max(1, l->n_live);
    a.pm = reinterpret_cast<float *>(ws + w.pm);
    a.pl = reinterpret_cast<float *>(ws + w.pl);
    a.pacc = reinterpret_cast<float *>(ws + w.pacc);
    a.scores = nullptr;
    a.err = l->d_err;
    a.window = window;
    a.softcap2 = softcap * kLog2e;
    a.K = K;
    a.hg = hg;
    LayerSrc s;
    s.kf = static_cast<const float *>(l->buf[KVD_BUF_K]);
    s.vf = static_cast<const float *>(l->buf[KVD_BUF_V]);
    s.kq = static_cast<const int8_t *>(l->buf[KVD_BUF_KQ]);
    s.vq = static_cast<const int8_t *>(l->buf[KVD_BUF_VQ]);
    s.ks = static_cast<const float *>(l->buf[KVD_BUF_KS]);
    s.vs = static_cast<const float *>(l->buf[KVD_BUF_VS]);
    s.kcol = static_cast<const float *>(l->buf[KVD_BUF_KCOL]);
    s.row_base = l->d_row_base;
    s.cap = l->d_cap;
    s.seq_len = l->d_seq_len;
    s.live = l->d_live;
    s.n_live = l->n_live;
    MergeLayerSrc ms;
    ms.seq_len = l->d_seq_len;
    ms.slot = l->d_slot;
    ms.vcol = static_cast<const float *>(l->buf[KVD_BUF_VCOL]);
    ms.n_live = l->n_live;
    if (warp_path(l)) {
        // q8_2f at head_dim 128: the K * hg query rows of a group are the M rows
        // of the tensor-core kernel (heads in M), one read of every tile
        int64_t T = 0;
        for (int b = 0; b < l->n_seq; ++b) T += int64_t(l->n_live) * tiles_of(l->h_seq_len[b], window, K);
        const int64_t workers = split_q8_tc_workers(2);
        if (workers <= 0) return KVD_ECUDA;
        WarpArgs wa;
        wa.a = a;
        wa.T = T;
        wa.G = int32_t(std::min(T, workers));
        wa.n_seq = l->n_seq;
        wa.unit_slots = reinterpret_cast<int64_t *>(ws + w.units);
        if (T > 0) {
            MmaMaps maps;
            std::memcpy(&maps.kq, l->tmap_kq, sizeof(maps.kq));
            std::memcpy(&maps.vq, l->tmap_vq, sizeof(maps.vq));
            if (split_layer_q8_tc(2, wa, s, maps, st) != cudaSuccess) return KVD_ECUDA;
        }
        RunMergeArgs rm;
        rm.pm = a.pm;
        rm.pl = a.pl;
        rm.pacc = a.pacc;
        rm.out = out;
        rm.ml = nullptr;
        rm.n_q = n_q;
        rm.hpk = hpk;
        rm.K = K;
        rm.hg = hg;
        rm.unit_slots = wa.unit_slots;
        rm.sinks = sinks;
        const bool few = unit_slots_within(l, window, K, T, wa.G, 2 * kHeadBatch);
        return launch_run_merge(rm, ms, l->n_seq, K, few, st) == cudaSuccess ? KVD_OK : KVD_ECUDA;
    }
    if (max_len > 0 && l->n_live > 0) {
        dim3 grid(unsigned(ceil_div(max_len, chunk)), unsigned(l->n_live), unsigned(l->n_seq));
        const int hb = hpk_bucket(hpk);
        cudaError_t e;
        switch (l->mode) {
            case KVD_F32: e = split_layer_f32(l->hd, hb, a, s, grid, st); break;
            case KVD_Q8: e = split_layer_q8(l->hd, hb, a, s, grid, st); break;
            case KVD_Q8K: e = split_layer_q8k(l->hd, hb, a, s, grid, st); break;
            default: e = split_layer_q8v(l->hd, hb, a, s, grid, st); break;
        }
        if (e != cudaSuccess) return KVD_ECUDA;
    }
    MergeArgs m;
    m.pm = a.pm;
    m.pl = a.pl;
    m.pacc = a.pacc;
    m.out = out;
    m.ml = nullptr;
    m.n_q = n_q;
    m.hpk = hpk;
    m.n_grp = a.n_grp;
    m.nc_max = w.nc_max;
    m.chunk = chunk;
    m.sinks = sinks;
    m.window = window;
    dim3 mgrid(unsigned(n_q), unsigned(l->n_seq), unsigned(K));
    if (l->hd == 128) merge_verify_kernel<128><<<mgrid, 128, 0, st>>>(m, ms, K, hg);
    else merge_verify_kernel<64><<<mgrid, 64, 0, st>>>(m, ms, K, hg);
    return launch_status() == cudaSuccess ? KVD_OK : KVD_ECUDA;
}

// ------------------------------------------------------------------ R-SWA

// The eight mirror pointers are present and 16-byte aligned.
static bool mirror_ok(const rswa_i8_mirror *m) {
    return m != nullptr && aligned16(m->ref_k) && aligned16(m->ref_v) && aligned16(m->ref_ks) &&
           aligned16(m->ref_vs) && aligned16(m->ring_k) && aligned16(m->ring_v) &&
           aligned16(m->ring_ks) && aligned16(m->ring_vs) && m->ref_k && m->ref_v && m->ref_ks &&
           m->ref_vs && m->ring_k && m->ring_v && m->ring_ks && m->ring_vs;
}

static kvd_status record_prefill(float *ref_k, float *ref_v, const rswa_i8_mirror *m, const float *k,
                          const float *v, int32_t s, int32_t seq, int32_t B, int32_t H,
                          int32_t head_dim, int64_t ref_cap, int32_t W, int32_t *prefill_len,
                          int32_t *ring_len, int32_t *ring_pos, rswa_history *hist, void *stream) {
    if (ref_k == nullptr || ref_v == nullptr || prefill_len == nullptr || ring_len == nullptr ||
        ring_pos == nullptr)
        return KVD_EINVAL;
    if (B < 1 || s < 0 || s >= B || H < 1 || head_dim < 1 || W < 1 || ref_cap < 0 || seq < 0)
        return KVD_EINVAL;
    if (seq > ref_cap) return KVD_ECAPACITY;
    if (seq > 0 && (k == nullptr || v == nullptr)) return KVD_EINVAL;
    // the new lineage is reserved before anything changes
    if (hist != nullptr && hist[s].lineage_epoch == UINT64_MAX) return KVD_ESTATE;
    if (m != nullptr) {
        if (!mirror_ok(m) || (head_dim != 64 && head_dim != 128) || !aligned16(ref_k) ||
            !aligned16(ref_v) || (seq > 0 && (!aligned16(k) || !aligned16(v))))
            return KVD_EINVAL;
    }
    if (seq > 0) {
        cudaStream_t st = as_stream(stream);
        if (m != nullptr) {
            const int64_t warps = int64_t(H) * seq;
            const unsigned blocks = unsigned(std::min<int64_t>(ceil_div(warps, 8), 152 * 16));
            if (head_dim == 128)
                prefill_i8_kernel<128><<<blocks, 256, 0, st>>>(ref_k, ref_v, *m, k, v, s, seq, H, ref_cap);
            else
                prefill_i8_kernel<64><<<blocks, 256, 0, st>>>(ref_k, ref_v, *m, k, v, s, seq, H, ref_cap);
        } else {
            const int64_t total = int64_t(H) * seq * head_dim;
            const unsigned blocks = unsigned(std::min<int64_t>(ceil_div(total, 256), 152 * 16));
            prefill_copy_kernel<<<blocks, 256, 0, st>>>(ref_k, ref_v, k, v, s, seq, H, head_dim,
                                                        ref_cap);
        }
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    prefill_len[s] = seq;
    ring_len[s] = 0;
    ring_pos[s] = 0;
    if (hist != nullptr) {
        hist[s].decode_writes = 0;
        hist[s].lineage_epoch += 1;
    }
    return KVD_OK;
}

extern "C" kvd_status rswa_record_prefill(float *ref_k, float *ref_v, const float *k,
                                          const float *v, int32_t s, int32_t seq, int32_t B,
                                          int32_t H, int32_t head_dim, int64_t ref_cap, int32_t W,
                                          int32_t *prefill_len, int32_t *ring_len,
                                          int32_t *ring_pos, rswa_history *hist, void *stream) {
    KVD_NVTX_RANGE("rswa_record_prefill");
    return record_prefill(ref_k, ref_v, nullptr, k, v, s, seq, B, H, head_dim, ref_cap, W,
                          prefill_len, ring_len, ring_pos, hist, stream);
}

extern "C" kvd_status rswa_record_prefill_i8(float *ref_k, float *ref_v, const rswa_i8_mirror *m,
                                             const float *k, const float *v, int32_t s, int32_t seq,
                                             int32_t B, int32_t H, int32_t head_dim, int64_t ref_cap,
                                             int32_t W, int32_t *prefill_len, int32_t *ring_len,
                                             int32_t *ring_pos, rswa_history *hist, void *stream) {
    KVD_NVTX_RANGE("rswa_record_prefill_i8");
    if (m == nullptr) return KVD_EINVAL;
    return record_prefill(ref_k, ref_v, m, k, v, s, seq, B, H, head_dim, ref_cap, W, prefill_len,
                          ring_len, ring_pos, hist, stream);
}

static kvd_status ring_write(float *ring_k, float *ring_v, const rswa_i8_mirror *m, const float *k,
                      const float *v, const int32_t *prefill_len, int32_t *ring_len,
                      int32_t *ring_pos, rswa_history *hist, int32_t B, int32_t H, int32_t head_dim,
                      int32_t W, int32_t *slot_out, void *stream) {
    if (ring_k == nullptr || ring_v == nullptr || k == nullptr || v == nullptr ||
        prefill_len == nullptr || ring_len == nullptr || ring_pos == nullptr)
        return KVD_EINVAL;
    if (B < 1 || H < 1 || head_dim < 1 || W < 1) return KVD_EINVAL;
    if (m != nullptr && (!mirror_ok(m) || (head_dim != 64 && head_dim != 128) || !aligned16(k) ||
                         !aligned16(v) || !aligned16(ring_k) || !aligned16(ring_v)))
        return KVD_EINVAL;
    for (int s = 0; s < B; ++s) {
        if (prefill_len[s] < 0) return KVD_ESTATE;
        if (ring_len[s] < 0 || ring_len[s] > W || ring_pos[s] < 0 || ring_pos[s] >= W)
            return KVD_EINVAL;
        if (hist != nullptr && (hist[s].decode_writes < 0 || hist[s].decode_writes == INT64_MAX))
            return KVD_ESTATE;
    }
    std::vector<int32_t> slot(B);
    for (int s = 0; s < B; ++s) slot[s] = ring_len[s] < W ? ring_len[s] : ring_pos[s];
    for (int32_t s0 = 0; s0 < B; s0 += kSlice) {
        RingWriteTable t;
        t.s0 = s0;
        t.n = std::min(kSlice, B - s0);
        for (int i = 0; i < t.n; ++i) t.slot[i] = slot[s0 + i];
        if (m != nullptr) {
            const unsigned blocks = unsigned(ceil_div(int64_t(t.n) * H, 8));
            if (head_dim == 128)
                ring_write_i8_kernel<128><<<blocks, 256, 0, as_stream(stream)>>>(ring_k, ring_v, *m, k, v,
                                                                                H, W, t);
            else
                ring_write_i8_kernel<64><<<blocks, 256, 0, as_stream(stream)>>>(ring_k, ring_v, *m, k, v,
                                                                               H, W, t);
        } else {
            const int64_t per = int64_t(H) * head_dim;
            dim3 grid(unsigned(std::min<int64_t>(ceil_div(per, 256), 64)), unsigned(t.n));
            ring_write_kernel<<<grid, 256, 0, as_stream(stream)>>>(ring_k, ring_v, k, v, H, head_dim,
                                                                  W, t);
        }
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    for (int s = 0; s < B; ++s) {
        if (ring_len[s] < W) {
            ring_len[s] += 1;
            ring_pos[s] = ring_len[s] % W;
        } else {
            ring_pos[s] = (ring_pos[s] + 1) % W;
        }
        if (slot_out) slot_out[s] = slot[s];
        if (hist) hist[s].decode_writes += 1;
    }
    return KVD_OK;
}

extern "C" kvd_status rswa_ring_write(float *ring_k, float *ring_v, const float *k, const float *v,
                                      const int32_t *prefill_len, int32_t *ring_len,
                                      int32_t *ring_pos, rswa_history *hist, int32_t B, int32_t H,
                                      int32_t head_dim, int32_t W, int32_t *slot_out, void *stream) {
    KVD_NVTX_RANGE("rswa_ring_write");
    return ring_write(ring_k, ring_v, nullptr, k, v, prefill_len, ring_len, ring_pos, hist, B, H,
                      head_dim, W, slot_out, stream);
}

extern "C" kvd_status rswa_ring_write_i8(float *ring_k, float *ring_v, const rswa_i8_mirror *m,
                                         const float *k, const float *v, const int32_t *prefill_len,
                                         int32_t *ring_len, int32_t *ring_pos, rswa_history *hist,
                                         int32_t B, int32_t H, int32_t head_dim, int32_t W,
                                         int32_t *slot_out, void *stream) {
    KVD_NVTX_RANGE("rswa_ring_write_i8");
    if (m == nullptr) return KVD_EINVAL;
    return ring_write(ring_k, ring_v, m, k, v, prefill_len, ring_len, ring_pos, hist, B, H, head_dim,
                      W, slot_out, stream);
}

extern "C" kvd_status rswa_checkpoint_take(uint64_t cache_id, const int32_t *prefill_len,
                                           const int32_t *ring_len, const int32_t *ring_pos,
                                           const rswa_history *hist, int32_t s, rswa_checkpoint *out) {
    if (prefill_len == nullptr || ring_len == nullptr || ring_pos == nullptr || hist == nullptr ||
        out == nullptr || s < 0)
        return KVD_EINVAL;
    rswa_checkpoint cp{};
    cp.cache_id = cache_id;
    cp.lineage_epoch = hist[s].lineage_epoch;
    cp.decode_writes = hist[s].decode_writes;
    cp.prefill_len = prefill_len[s];
    cp.ring_len = ring_len[s];
    cp.ring_pos = ring_pos[s];
    *out = cp;
    return KVD_OK;
}

extern "C" kvd_status rswa_rollback_to(uint64_t cache_id, const int32_t *prefill_len, int32_t *ring_len,
                                       int32_t *ring_pos, rswa_history *hist, int32_t s, int32_t W,
                                       const rswa_checkpoint *cp) {
    if (prefill_len == nullptr || ring_len == nullptr || ring_pos == nullptr || hist == nullptr ||
        cp == nullptr || s < 0 || W < 1)
        return KVD_EINVAL;
    // the page's order of refusals; nothing changes on any of them
    if (cp->cache_id != cache_id) return KVD_ESTATE;
    if (cp->prefill_len != prefill_len[s]) return KVD_ESTATE;
    if (cp->lineage_epoch != hist[s].lineage_epoch) return KVD_ESTATE;
    if (cp->decode_writes > hist[s].decode_writes) return KVD_ESTATE;
    const int64_t discarded = hist[s].decode_writes - cp->decode_writes;
    if (cp->ring_len < 0 || cp->ring_len > W || discarded > int64_t(W) - cp->ring_len) return KVD_ESTATE;
    if (cp->ring_pos < 0 || cp->ring_pos >= W) return KVD_EINVAL;
    if (discarded > 0 && hist[s].lineage_epoch == UINT64_MAX) return KVD_ESTATE;
    ring_len[s] = cp->ring_len;
    ring_pos[s] = cp->ring_pos;
    hist[s].decode_writes = cp->decode_writes;
    if (discarded > 0) hist[s].lineage_epoch += 1;
    return KVD_OK;
}

extern "C" kvd_status rswa_decode_workspace_bytes(int32_t B, int32_t H, int32_t head_dim,
                                                  int64_t ref_cap, int32_t W, int64_t *bytes_out) {
    if (bytes_out == nullptr || B < 1 || H < 1 || (head_dim != 64 && head_dim != 128) ||
        ref_cap < 0 || W < 1)
        return KVD_EINVAL;
    *bytes_out = rswa_ws(B, H, head_dim, ref_cap, W).total;
    return KVD_OK;
}

// rswa decode over the f32 regions (I8 false) or the int8 mirror (I8 true);
// src holds the pointers of the one that is read, already checked.
template <bool I8>
static kvd_status rswa_decode_impl(const float *q, const RswaSrc &src_in, const int32_t *prefill_len,
                            const int32_t *ring_len, const int32_t *ring_pos, int32_t B, int32_t H,
                            int32_t head_dim, int64_t ref_cap, int32_t W, float scale, float *out,
                            void *workspace, int64_t workspace_bytes, void *stream) {
    if (q == nullptr || prefill_len == nullptr || ring_len == nullptr || out == nullptr)
        return KVD_EINVAL;
    if (B < 1 || H < 1 || (head_dim != 64 && head_dim != 128) || ref_cap < 0 || W < 1)
        return KVD_EINVAL;
    // Bulk copies move whole 16-row groups: both regions must hold them.
    if (ref_cap % kRowAlign != 0 || W % kRowAlign != 0) return KVD_EINVAL;
    if (!std::isfinite(scale)) return KVD_EINVAL;
    if (!aligned16(q) || !aligned16(out)) return KVD_EINVAL;
    const RswaWs w = rswa_ws(B, H, head_dim, ref_cap, W);
    if (workspace == nullptr || workspace_bytes < w.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return KVD_EINVAL;
    int64_t work = 0;
    for (int s = 0; s < B; ++s) {
        if (prefill_len[s] < 0) return KVD_ESTATE;
        if (prefill_len[s] > ref_cap || ring_len[s] < 0 || ring_len[s] > W) return KVD_EINVAL;
        if (ring_pos && (ring_pos[s] < 0 || ring_pos[s] >= W)) return KVD_EINVAL;
        if (prefill_len[s] + ring_len[s] == 0) return KVD_EEMPTY;
        work += int64_t(prefill_len[s] + ring_len[s]) * H;
    }
    const int32_t chunk = pick_chunk(work);
    char *ws = static_cast<char *>(workspace);
    cudaStream_t st = as_stream(stream);
    SplitArgs a;
    a.q = q;
    a.n_q = H;
    a.hpk = 1;
    a.qscale = scale * kLog2e;
    a.chunk = chunk;
    a.nc_max = w.nc_max;
    a.n_grp = H;
    a.pm = reinterpret_cast<float *>(ws + w.pm);
    a.pl = reinterpret_cast<float *>(ws + w.pl);
    a.pacc = reinterpret_cast<float *>(ws + w.pacc);
    a.scores = nullptr;
    a.err = reinterpret_cast<uint32_t *>(ws + w.err);
    RswaSrc src = src_in;
    src.ref_cap = ref_cap;
    src.W = W;
    src.H = H;
    MergeArgs m;
    m.pm = a.pm;
    m.pl = a.pl;
    m.pacc = a.pacc;
    m.out = out;
    m.ml = nullptr;
    m.n_q = H;
    m.hpk = 1;
    m.n_grp = H;
    m.nc_max = w.nc_max;
    m.chunk = chunk;
    for (int32_t s0 = 0; s0 < B; s0 += kSlice) {
        RswaTable t;
        t.s0 = s0;
        t.n = std::min(kSlice, B - s0);
        int32_t max_nc = 0;
        for (int i = 0; i < t.n; ++i) {
            t.prefill_len[i] = prefill_len[s0 + i];
            t.ring_len[i] = ring_len[s0 + i];
            const int32_t nc = int32_t(ceil_div(t.prefill_len[i], chunk) + ceil_div(t.ring_len[i], chunk));
            max_nc = std::max(max_nc, nc);
        }
        dim3 grid(unsigned(max_nc), unsigned(H), unsigned(t.n));
        cudaError_t e = head_dim == 128 ? launch_split_rswa<128, I8>(a, src, t, grid, st)
                                        : launch_split_rswa<64, I8>(a, src, t, grid, st);
        if (e != cudaSuccess) return KVD_ECUDA;
        dim3 mgrid(unsigned(H), unsigned(t.n));
        if (head_dim == 128) merge_rswa_kernel<128><<<mgrid, 128, 0, st>>>(m, t);
        else merge_rswa_kernel<64><<<mgrid, 64, 0, st>>>(m, t);
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    return KVD_OK;
}

extern "C" kvd_status rswa_decode(const float *q, const float *ref_k, const float *ref_v,
                                  const float *ring_k, const float *ring_v,
                                  const int32_t *prefill_len, const int32_t *ring_len,
                                  const int32_t *ring_pos, int32_t B, int32_t H, int32_t head_dim,
                                  int64_t ref_cap, int32_t W, float scale, float *out,
                                  void *workspace, int64_t workspace_bytes, void *stream) {
    KVD_NVTX_RANGE("rswa_decode");
    if (ref_k == nullptr || ref_v == nullptr || ring_k == nullptr || ring_v == nullptr ||
        !aligned16(ref_k) || !aligned16(ref_v) || !aligned16(ring_k) || !aligned16(ring_v))
        return KVD_EINVAL;
    RswaSrc src{};
    src.ref_k = ref_k;
    src.ref_v = ref_v;
    src.ring_k = ring_k;
    src.ring_v = ring_v;
    return rswa_decode_impl<false>(q, src, prefill_len, ring_len, ring_pos, B, H, head_dim, ref_cap, W,
                                   scale, out, workspace, workspace_bytes, stream);
}

extern "C" kvd_status rswa_decode_i8(const float *q, const rswa_i8_mirror *m,
                                     const int32_t *prefill_len, const int32_t *ring_len,
                                     const int32_t *ring_pos, int32_t B, int32_t H, int32_t head_dim,
                                     int64_t ref_cap, int32_t W, float scale, float *out,
                                     void *workspace, int64_t workspace_bytes, void *stream) {
    KVD_NVTX_RANGE("rswa_decode_i8");
    if (!mirror_ok(m)) return KVD_EINVAL;
    RswaSrc src{};
    src.ref_k8 = m->ref_k;
    src.ref_v8 = m->ref_v;
    src.ring_k8 = m->ring_k;
    src.ring_v8 = m->ring_v;
    src.ref_ks = m->ref_ks;
    src.ref_vs = m->ref_vs;
    src.ring_ks = m->ring_ks;
    src.ring_vs = m->ring_vs;
    return rswa_decode_impl<true>(q, src, prefill_len, ring_len, ring_pos, B, H, head_dim, ref_cap, W,
                                  scale, out, workspace, workspace_bytes, stream);
}

// rswa verify_attention over the f32 regions (I8 false) or the int8 mirror.
template <bool I8>
static kvd_status rswa_verify_impl(const float *q, const float *dk, const float *dv, int32_t K,
                                   const RswaSrc &src_in, const int32_t *prefill_len, const int32_t *ring_len,
                                   const int32_t *ring_pos, int32_t B, int32_t H, int32_t head_dim,
                                   int64_t ref_cap, int32_t W, float scale, float *out, void *workspace,
                                   int64_t workspace_bytes, void *stream) {
    if (q == nullptr || dk == nullptr || dv == nullptr || prefill_len == nullptr || ring_len == nullptr ||
        ring_pos == nullptr || out == nullptr)
        return KVD_EINVAL;
    if (K < 1 || K > kMaxHpk || B < 1 || H < 1 || (head_dim != 64 && head_dim != 128) || ref_cap < 0 || W < 1)
        return KVD_EINVAL;
    if (ref_cap % kRowAlign != 0 || W % kRowAlign != 0) return KVD_EINVAL;
    if (!std::isfinite(scale)) return KVD_EINVAL;
    if (!aligned16(q) || !aligned16(out) || !aligned16(dk) || !aligned16(dv)) return KVD_EINVAL;
    const RswaWs w = rswa_ws(B, H, head_dim, ref_cap, W, K, true);
    if (workspace == nullptr || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return KVD_EINVAL;
    int64_t work = 0;
    for (int s = 0; s < B; ++s) {
        if (prefill_len[s] < 0) return KVD_ESTATE;  // write_decode_step refuses a stream without prefill
        if (prefill_len[s] > ref_cap || ring_len[s] < 0 || ring_len[s] > W || ring_pos[s] < 0 ||
            ring_pos[s] >= W)
            return KVD_EINVAL;
        work += int64_t(prefill_len[s]) * H;
    }
    const int32_t chunk = pick_chunk(std::max<int64_t>(work, 1));
    char *ws = static_cast<char *>(workspace);
    cudaStream_t st = as_stream(stream);
    SplitArgs a;
    a.q = q;
    a.n_q = H;
    a.hpk = K;
    a.K = K;
    a.hg = 1;
    a.qscale = scale * kLog2e;
    a.chunk = chunk;
    a.nc_max = w.nc_max;
    a.n_grp = H;
    a.pm = reinterpret_cast<float *>(ws + w.pm);
    a.pl = reinterpret_cast<float *>(ws + w.pl);
    a.pacc = reinterpret_cast<float *>(ws + w.pacc);
    a.scores = nullptr;
    a.err = reinterpret_cast<uint32_t *>(ws + w.err);
    RswaSrc src = src_in;
    src.ref_cap = ref_cap;
    src.W = W;
    src.H = H;
    TailArgs ta;
    ta.q = q;
    ta.dk = dk;
    ta.dv = dv;
    ta.ring_k = src.ring_k;
    ta.ring_v = src.ring_v;
    ta.ring_k8 = src.ring_k8;
    ta.ring_v8 = src.ring_v8;
    ta.ring_ks = src.ring_ks;
    ta.ring_vs = src.ring_vs;
    ta.pm = a.pm;
    ta.pl = a.pl;
    ta.pacc = a.pacc;
    ta.K = K;
    ta.H = H;
    ta.W = W;
    ta.nc_max = w.nc_max;
    ta.qscale = a.qscale;
    MergeArgs m;
    m.pm = a.pm;
    m.pl = a.pl;
    m.pacc = a.pacc;
    m.out = out;
    m.ml = nullptr;
    m.n_q = H;
    m.hpk = K;
    m.n_grp = H;
    m.nc_max = w.nc_max;
    m.chunk = chunk;
    // The int8 mirror's reference block on the tensor-core kernel (the draft
    // rows of a head as the group's query rows), else the CUDA-core kernel.
    const int variant = K <= 4 ? 3 : 4;
    MmaMaps maps;
    int64_t workers = 0;
    bool tc = false;
    if (I8 && w.tc) {
        const int64_t rows = int64_t(B) * H * ref_cap;
        tc = encode_code_map(const_cast<int8_t *>(src_in.ref_k8), rows, head_dim,
                             reinterpret_cast<unsigned char *>(&maps.kq)) &&
             encode_code_map(const_cast<int8_t *>(src_in.ref_v8), rows, head_dim,
                             reinterpret_cast<unsigned char *>(&maps.vq));
        workers = tc ? std::min(split_q8_tc_workers(variant), kRswaTcWorkers) : 0;
        tc = workers > 0;
    }
    const int hb = hpk_bucket(K);
    for (int32_t s0 = 0; s0 < B; s0 += kSlice) {
        RswaTable t;  // the split kernel reads the reference rows only
        TailTable tt;
        t.s0 = tt.s0 = s0;
        t.n = tt.n = std::min(kSlice, B - s0);
        int32_t max_nc = 0;
        for (int i = 0; i < t.n; ++i) {
            const int s = s0 + i;
            t.prefill_len[i] = prefill_len[s];
            t.ring_len[i] = 0;
            tt.ring_len[i] = ring_len[s];
            tt.rp0[i] = ring_len[s] == W ? ring_pos[s] : 0;
            // tensor-core path: nc_ref only flags a reference block for the fused merge
            tt.nc_ref[i] = tc ? (prefill_len[s] > 0 ? 1 : 0) : int32_t(ceil_div(prefill_len[s], chunk));
            max_nc = std::max(max_nc, tt.nc_ref[i]);
        }
        if (tc) {
            RswaTcTables tabs;
            tabs.seq_len = reinterpret_cast<int32_t *>(ws + w.t_len);
            tabs.live = reinterpret_cast<int32_t *>(ws + w.t_live);
            tabs.cap = reinterpret_cast<int64_t *>(ws + w.t_cap);
            tabs.row_base = reinterpret_cast<int64_t *>(ws + w.t_base);
            tabs.H = H;
            tabs.ref_cap = ref_cap;
            rswa_tc_tables_kernel<<<1, 256, 0, st>>>(t, tabs);
            if (launch_status() != cudaSuccess) return KVD_ECUDA;
            int64_t T = 0;
            for (int i = 0; i < t.n; ++i) T += int64_t(H) * ceil_div(t.prefill_len[i], kWR);
            WarpArgs wa;
            wa.a = a;
            wa.a.q = q + int64_t(s0) * K * H * head_dim;
            wa.a.K = 1;  // every draft sees the whole block
            wa.a.hg = 0;
            wa.a.pm = reinterpret_cast<float *>(ws + w.tc_pm);
            wa.a.pl = reinterpret_cast<float *>(ws + w.tc_pl);
            wa.a.pacc = reinterpret_cast<float *>(ws + w.tc_pacc);
            wa.T = T;
            wa.G = int32_t(std::min(T, workers));
            wa.n_seq = t.n;
            wa.unit_slots = reinterpret_cast<int64_t *>(ws + w.units);
            LayerSrc ls{};
            ls.ks = src.ref_ks;
            ls.vs = src.ref_vs;
            ls.row_base = tabs.row_base;
            ls.cap = tabs.cap;
            ls.seq_len = tabs.seq_len;
            ls.live = tabs.live;
            ls.n_live = H;
            if (T > 0 && split_layer_q8_tc(variant, wa, ls, maps, st) != cudaSuccess) return KVD_ECUDA;
            RswaRunMerge rm;
            rm.pm = wa.a.pm;
            rm.pl = wa.a.pl;
            rm.pacc = wa.a.pacc;
            rm.unit_slots = wa.unit_slots;
            rm.out = out;
            rm.H = H;
            rm.K = K;
            // the ring-and-drafts partials and the merge, as the split's dependent
            if (launch_pdl(rswa_verify_tail_kernel<128, true, true>, dim3(unsigned(K), unsigned(H), unsigned(t.n)),
                           dim3(128), 0, st, ta, tt, rm) != cudaSuccess)
                return KVD_ECUDA;
            continue;
        }
        if (max_nc > 0) {
            dim3 grid(unsigned(max_nc), unsigned(H), unsigned(t.n));
            cudaError_t e = head_dim == 128 ? launch_split_rswa_k<128, I8>(hb, a, src, t, grid, st)
                                            : launch_split_rswa_k<64, I8>(hb, a, src, t, grid, st);
            if (e != cudaSuccess) return KVD_ECUDA;
        }
        dim3 tgrid(unsigned(K), unsigned(H), unsigned(t.n));
        if (head_dim == 128) rswa_verify_tail_kernel<128, I8><<<tgrid, 128, 0, st>>>(ta, tt, RswaRunMerge{});
        else rswa_verify_tail_kernel<64, I8><<<tgrid, 128, 0, st>>>(ta, tt, RswaRunMerge{});
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
        dim3 mgrid(unsigned(H), unsigned(t.n), unsigned(K));
        if (head_dim == 128) merge_rswa_verify_kernel<128><<<mgrid, 128, 0, st>>>(m, t, K);
        else merge_rswa_verify_kernel<64><<<mgrid, 64, 0, st>>>(m, t, K);
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    return KVD_OK;
}

extern "C" kvd_status rswa_verify_workspace_bytes(int32_t B, int32_t H, int32_t head_dim, int64_t ref_cap,
                                                  int32_t W, int32_t K, int64_t *bytes_out) {
    if (bytes_out == nullptr || B < 1 || H < 1 || (head_dim != 64 && head_dim != 128) || ref_cap < 0 || W < 1 ||
        K < 1 || K > kMaxHpk)
        return KVD_EINVAL;
    *bytes_out = rswa_ws(B, H, head_dim, ref_cap, W, K, true).total;
    return KVD_OK;
}

extern "C" kvd_status rswa_verify(const float *q, const float *draft_k, const float *draft_v, int32_t K,
                                  const float *ref_k, const float *ref_v, const float *ring_k,
                                  const float *ring_v, const int32_t *prefill_len, const int32_t *ring_len,
                                  const int32_t *ring_pos, int32_t B, int32_t H, int32_t head_dim,
                                  int64_t ref_cap, int32_t W, float scale, float *out, void *workspace,
                                  int64_t workspace_bytes, void *stream) {
    KVD_NVTX_RANGE("rswa_verify");
    if (ref_k == nullptr || ref_v == nullptr || ring_k == nullptr || ring_v == nullptr ||
        !aligned16(ref_k) || !aligned16(ref_v) || !aligned16(ring_k) || !aligned16(ring_v))
        return KVD_EINVAL;
    RswaSrc src{};
    src.ref_k = ref_k;
    src.ref_v = ref_v;
    src.ring_k = ring_k;
    src.ring_v = ring_v;
    return rswa_verify_impl<false>(q, draft_k, draft_v, K, src, prefill_len, ring_len, ring_pos, B, H, head_dim,
                                   ref_cap, W, scale, out, workspace, workspace_bytes, stream);
}

extern "C" kvd_status rswa_verify_i8(const float *q, const float *draft_k, const float *draft_v, int32_t K,
                                     const rswa_i8_mirror *m, const int32_t *prefill_len,
                                     const int32_t *ring_len, const int32_t *ring_pos, int32_t B, int32_t H,
                                     int32_t head_dim, int64_t ref_cap, int32_t W, float scale, float *out,
                                     void *workspace, int64_t workspace_bytes, void *stream) {
    KVD_NVTX_RANGE("rswa_verify_i8");
    if (!mirror_ok(m)) return KVD_EINVAL;
    RswaSrc src{};
    src.ref_k8 = m->ref_k;
    src.ref_v8 = m->ref_v;
    src.ring_k8 = m->ring_k;
    src.ring_v8 = m->ring_v;
    src.ref_ks = m->ref_ks;
    src.ref_vs = m->ref_vs;
    src.ring_ks = m->ring_ks;
    src.ring_vs = m->ring_vs;
    return rswa_verify_impl<true>(q, draft_k, draft_v, K, src, prefill_len, ring_len, ring_pos, B, H, head_dim,
                                  ref_cap, W, scale, out, workspace, workspace_bytes, stream);
}

extern "C" kvd_status rswa_device_error(const void *workspace, int32_t clear, uint32_t *word_out) {
    if (workspace == nullptr) return KVD_EINVAL;
    uint32_t w = 0;
    if (cudaMemcpy(&w, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVD_ECUDA;
    if (clear && cudaMemset(const_cast<void *>(workspace), 0, 4) != cudaSuccess) return KVD_ECUDA;
    if (word_out) *word_out = w;
    return w ? KVD_EDEVICE : KVD_OK;
}
