// kvd_append.cu -- append/quantise (cortiq LayerKvCache::append + quant_row)
// and the channel-field freeze (cortiq freeze_cols), batched over sequences.
//
// Bit-exactness: every f32 operation of the pages' quantiser and freeze is
// issued with an explicit IEEE rounding intrinsic (__fdiv_rn, __fmul_rn,
// __fadd_rn, __fsqrt_rn) so nothing is contracted or approximated; codes
// round half to even (__float2int_rn).

#include <algorithm>
#include <vector>

#include "kvd_internal.cuh"

namespace kvd {
namespace {

// Per-launch description of up to kSlice sequences: sequence seq0 + i
// appends count[i] rows read from input row in_row[i] onward (an input row is
// n_kv * hd floats) to storage rows start[i] .. start[i] + count[i].
struct AppendTable {
    int32_t seq0, n;
    int32_t in_row[kSlice];
    int32_t start[kSlice];
    int32_t count[kSlice];
};

struct AppendArgs {
    const float *k, *v;
    float *kf, *vf;         // f32 rows (unquantised components)
    int8_t *kq, *vq;        // codes
    float *ks, *vs;         // scales
    const float *kcol, *vcol;
    const int64_t *row_base, *cap;
    const int32_t *live;
    int32_t *seq_len;
    uint32_t *err;
    int32_t n_kv, n_live;
    int32_t qk, qv;
};

constexpr int kAppendWarps = 4;
constexpr int kItemsPerWarp = 1;

// Quantise one row held by a warp, CPL consecutive channels per lane, against
// the field `col` (1.0 before the freeze), with groups of `group` channels
// (group is 32 for K, the whole row for V).  Writes codes and scales.
template <int CPL>
__device__ __forceinline__ void quantise_row_warp(const float (&x)[CPL], const float (&col)[CPL],
                                                  int group, int8_t *q_row, float *s_row,
                                                  int lane) {
    float r[CPL];
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        r[j] = __fdiv_rn(x[j], col[j]);
        a = fmaxf(a, fabsf(r[j]));
    }
    const int lanes_per_group = group / CPL;  // power of two, <= 32
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
        if (off < lanes_per_group) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    float s = fmaxf(__fdiv_rn(a, 127.0f), 1e-12f);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        int c = __float2int_rn(__fdiv_rn(r[j], s));
        c = min(127, max(-127, c));
        packed |= (uint32_t(c) & 0xffu) << (8 * j);
    }
    if (CPL == 4) {
        reinterpret_cast<uint32_t *>(q_row)[lane] = packed;
    } else {
        reinterpret_cast<uint16_t *>(q_row)[lane] = uint16_t(packed);
    }
    if ((lane % lanes_per_group) == 0) s_row[(lane * CPL) / group] = s;
}

template <int HD>
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(AppendArgs a, AppendTable t) {
    // launched as a dependent of the kernel before (the previous step's imp
    // pass reads the lengths this kernel advances): wait for it, then let a
    // decode launched as a dependent be scheduled
    pdl_wait();
    pdl_trigger();
    constexpr int CPL = HD / 32;
    constexpr int NG = HD / kKGroup;
    const int i = blockIdx.y;
    if (i >= t.n) return;
    const int b = t.seq0 + i;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t count = t.count[i];
    const int64_t items = int64_t(count) * a.n_live;
    const int64_t cap = a.cap[b];
    const int64_t base = a.row_base[b];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (int64_t(t.start[i]) + count > cap) set_error(a.err, kErrBounds);
        else a.seq_len[b] = t.start[i] + count;
    }
    if (int64_t(t.start[i]) + count > cap) return;
    const int64_t first = (int64_t(blockIdx.x) * kAppendWarps + warp) * kItemsPerWarp;
    for (int it = 0; it < kItemsPerWarp; ++it) {
        const int64_t item = first + it;
        if (item >= items) return;
        const int r = int(item / a.n_live);
        const int gl = int(item % a.n_live);
        const int h = a.live[gl];
        const int64_t in_off = (int64_t(t.in_row[i] + r) * a.n_kv + h) * HD;
        const int64_t row = base + int64_t(gl) * cap + t.start[i] + r;
        float xk[CPL], xv[CPL], c[CPL];
        if (CPL == 4) {
            float4 k4 = reinterpret_cast<const float4 *>(a.k + in_off)[lane];
            float4 v4 = reinterpret_cast<const float4 *>(a.v + in_off)[lane];
            xk[0] = k4.x; xk[1] = k4.y; xk[2] = k4.z; xk[3] = k4.w;
            xv[0] = v4.x; xv[1] = v4.y; xv[2] = v4.z; xv[3] = v4.w;
        } else {
            float2 k2 = reinterpret_cast<const float2 *>(a.k + in_off)[lane];
            float2 v2 = reinterpret_cast<const float2 *>(a.v + in_off)[lane];
            xk[0] = k2.x; xk[1] = k2.y;
            xv[0] = v2.x; xv[1] = v2.y;
        }
        const int64_t col_off = (int64_t(b) * a.n_live + gl) * HD + lane * CPL;
        if (a.qk) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) c[j] = a.kcol[col_off + j];
            quantise_row_warp<CPL>(xk, c, kKGroup, a.kq + row * HD, a.ks + row * NG, lane);
        } else {
#pragma unroll
            for (int j = 0; j < CPL; ++j) a.kf[row * HD + lane * CPL + j] = xk[j];
        }
        if (a.qv) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) c[j] = a.vcol[col_off + j];
            quantise_row_warp<CPL>(xv, c, HD, a.vq + row * HD, a.vs + row, lane);
        } else {
#pragma unroll
            for (int j = 0; j < CPL; ++j) a.vf[row * HD + lane * CPL + j] = xv[j];
        }
    }
}

// ---------------------------------------------------------------- freeze

struct FreezeArgs {
    int8_t *kq, *vq;
    float *ks, *vs;
    float *kcol, *vcol;
    const int64_t *row_base, *cap;
    const int32_t *seq_len;
    int32_t *frozen;
    uint32_t *err;
    int32_t n_live, qk, qv;
    int32_t seq0, n;
    uint8_t todo[kSlice];  // 1 = this sequence freezes in this launch
};

// Freeze one component of one (sequence, live head): blockDim = HD threads,
// thread d owns channel d.  Rows are dequantised (code * scale, one rounded
// product), squared and summed in row order, col = max(sqrt(sum / n), 1e-6);
// then every row is requantised against col.  group = 32 (K) or HD (V).
template <int HD>
__device__ void freeze_component(int8_t *q, float *s, int spp, int group, float *col_out, int n,
                                 float *red) {
    const int d = threadIdx.x;
    const int lane = d & 31, warp = d >> 5;
    float acc = 0.0f;
    for (int p = 0; p < n; ++p) {
        const float r = __fmul_rn(float(q[int64_t(p) * HD + d]), s[int64_t(p) * spp + d / group]);
        acc = __fadd_rn(acc, __fmul_rn(r, r));
    }
    const float col = fmaxf(__fsqrt_rn(__fdiv_rn(acc, float(n))), 1e-6f);
    for (int p = 0; p < n; ++p) {
        const float row = __fmul_rn(float(q[int64_t(p) * HD + d]), s[int64_t(p) * spp + d / group]);
        const float r = __fdiv_rn(row, col);
        float a = fabsf(r);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if (group == HD) {  // one scale per row: reduce across the warps
            if (lane == 0) red[warp] = a;
            __syncthreads();
            a = red[0];
            for (int w = 1; w < HD / 32; ++w) a = fmaxf(a, red[w]);
        }
        const float sc = fmaxf(__fdiv_rn(a, 127.0f), 1e-12f);
        int c = __float2int_rn(__fdiv_rn(r, sc));
        c = min(127, max(-127, c));
        __syncthreads();  // every thread has read row p's old scale
        q[int64_t(p) * HD + d] = int8_t(c);
        if (group == HD) {
            if (d == 0) s[p] = sc;
        } else if (lane == 0) {
            s[int64_t(p) * spp + d / group] = sc;
        }
        __syncthreads();
    }
    col_out[d] = col;
}

template <int HD>
__global__ void __launch_bounds__(HD) freeze_kernel(FreezeArgs a) {
    __shared__ float red[HD / 32];
    const int i = blockIdx.y, gl = blockIdx.x;
    if (i >= a.n || !a.todo[i]) return;
    const int b = a.seq0 + i;
    // The host mirror decides which sequences freeze (todo); the device only
    // checks that its own length agrees with that decision.
    const int n = a.seq_len[b];
    const int64_t cap = a.cap[b];
    if (n < kColWarmup || n > cap) {
        if (threadIdx.x == 0) set_error(a.err, kErrBounds);
        return;
    }
    const int64_t row = a.row_base[b] + int64_t(gl) * cap;
    const int64_t col_off = (int64_t(b) * a.n_live + gl) * HD;
    constexpr int NG = HD / kKGroup;
    if (a.qk) freeze_component<HD>(a.kq + row * HD, a.ks + row * NG, NG, kKGroup, a.kcol + col_off, n, red);
    if (a.qv) freeze_component<HD>(a.vq + row * HD, a.vs + row, 1, HD, a.vcol + col_off, n, red);
    if (threadIdx.x == 0) a.frozen[b] = 1;  // same value from every head's block
}

AppendArgs append_args(const Layer *l, const float *k, const float *v) {
    AppendArgs a;
    a.k = k;
    a.v = v;
    a.kf = static_cast<float *>(l->buf[KVD_BUF_K]);
    a.vf = static_cast<float *>(l->buf[KVD_BUF_V]);
    a.kq = static_cast<int8_t *>(l->buf[KVD_BUF_KQ]);
    a.vq = static_cast<int8_t *>(l->buf[KVD_BUF_VQ]);
    a.ks = static_cast<float *>(l->buf[KVD_BUF_KS]);
    a.vs = static_cast<float *>(l->buf[KVD_BUF_VS]);
    a.kcol = static_cast<const float *>(l->buf[KVD_BUF_KCOL]);
    a.vcol = static_cast<const float *>(l->buf[KVD_BUF_VCOL]);
    a.row_base = l->d_row_base;
    a.cap = l->d_cap;
    a.live = l->d_live;
    a.seq_len = l->d_seq_len;
    a.err = l->d_err;
    a.n_kv = l->n_kv;
    a.n_live = l->n_live;
    a.qk = quant_k(l->mode);
    a.qv = quant_v(l->mode);
    return a;
}

kvd_status launch_append(const Layer *l, const float *k, const float *v, const AppendTable &t,
                         int64_t max_count, cudaStream_t s) {
    if (t.n == 0) return KVD_OK;
    const AppendArgs a = append_args(l, k, v);
    const int64_t items = std::max<int64_t>(1, max_count * l->n_live);
    const int64_t per_block = kAppendWarps * kItemsPerWarp;
    dim3 grid(unsigned((items + per_block - 1) / per_block), unsigned(t.n));
    const cudaError_t e = l->hd == 128 ? launch_pdl(append_kernel<128>, grid, dim3(kAppendWarps * 32), 0, s, a, t)
                                       : launch_pdl(append_kernel<64>, grid, dim3(kAppendWarps * 32), 0, s, a, t);
    return e == cudaSuccess ? KVD_OK : KVD_ECUDA;
}

FreezeArgs freeze_args(const Layer *l) {
    FreezeArgs a;
    a.kq = static_cast<int8_t *>(l->buf[KVD_BUF_KQ]);
    a.vq = static_cast<int8_t *>(l->buf[KVD_BUF_VQ]);
    a.ks = static_cast<float *>(l->buf[KVD_BUF_KS]);
    a.vs = static_cast<float *>(l->buf[KVD_BUF_VS]);
    a.kcol = static_cast<float *>(l->buf[KVD_BUF_KCOL]);
    a.vcol = static_cast<float *>(l->buf[KVD_BUF_VCOL]);
    a.row_base = l->d_row_base;
    a.cap = l->d_cap;
    a.seq_len = l->d_seq_len;
    a.frozen = l->d_frozen;
    a.err = l->d_err;
    a.n_live = l->n_live;
    a.qk = quant_k(l->mode);
    a.qv = quant_v(l->mode);
    return a;
}

// Freeze the sequences flagged in `todo` (host view); updates the host mirror.
kvd_status launch_freeze(Layer *l, const std::vector<uint8_t> &todo, cudaStream_t s) {
    if (l->mode == KVD_F32 || l->n_live == 0) return KVD_OK;
    for (int32_t s0 = 0; s0 < l->n_seq; s0 += kSlice) {
        FreezeArgs a = freeze_args(l);
        a.seq0 = s0;
        a.n = std::min(kSlice, l->n_seq - s0);
        bool any = false;
        for (int i = 0; i < a.n; ++i) {
            a.todo[i] = todo[s0 + i];
            any = any || a.todo[i];
        }
        if (!any) continue;
        dim3 grid(unsigned(l->n_live), unsigned(a.n));
        if (l->hd == 128) freeze_kernel<128><<<grid, 128, 0, s>>>(a);
        else freeze_kernel<64><<<grid, 64, 0, s>>>(a);
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    return KVD_OK;
}

bool freeze_due(const Layer *l, int b) {
    return l->mode != KVD_F32 && l->n_live > 0 && !l->h_frozen[b] && l->h_seq_len[b] >= kColWarmup;
}

}  // namespace

// Bounds self-test of the append and freeze kernels (kvd_bounds_selftest):
// launches whose metadata put sequence 0 one row past its capacity.  The
// append is asked for storage row cap[0]; the freeze reads lengths from
// `seq_len` (scratch holding cap[0] + 1 for sequence 0).  Each kernel's guard
// must set bit 1 of the error word and return before touching storage; the
// lengths and frozen flags they could write point at scratch too.
cudaError_t append_bounds_selftest(const Layer *l, const float *zeros, int32_t *seq_len, int32_t *frozen,
                                   cudaStream_t s) {
    AppendArgs a = append_args(l, zeros, zeros);
    a.seq_len = seq_len + l->n_seq;  // a second scratch copy: the append may only write past the first
    AppendTable t{};
    t.seq0 = 0;
    t.n = 1;
    t.in_row[0] = 0;
    t.start[0] = int32_t(l->h_cap[0]);
    t.count[0] = 1;
    if (l->hd == 128) append_kernel<128><<<dim3(1, 1), kAppendWarps * 32, 0, s>>>(a, t);
    else append_kernel<64><<<dim3(1, 1), kAppendWarps * 32, 0, s>>>(a, t);
    cudaError_t e = launch_status();
    if (e != cudaSuccess || l->mode == KVD_F32) return e;
    FreezeArgs f = freeze_args(l);
    f.seq_len = seq_len;
    f.frozen = frozen;
    f.seq0 = 0;
    f.n = 1;
    f.todo[0] = 1;
    if (l->hd == 128) freeze_kernel<128><<<dim3(unsigned(l->n_live), 1), 128, 0, s>>>(f);
    else freeze_kernel<64><<<dim3(unsigned(l->n_live), 1), 64, 0, s>>>(f);
    return launch_status();
}

}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kv_append(kvd_layer *L, const float *k, const float *v, const int32_t *n_new,
                                void *stream) {
    KVD_NVTX_RANGE("kv_append");
    Layer *l = checked_layer(L);
    if (l == nullptr || k == nullptr || v == nullptr) return KVD_EINVAL;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) return KVD_EINVAL;
    const int ns = l->n_seq;
    // Validate everything before touching anything.
    std::vector<int64_t> cnt(ns), in_row(ns);
    int64_t acc = 0;
    for (int b = 0; b < ns; ++b) {
        const int64_t c = n_new ? n_new[b] : 1;
        if (c < 0) return KVD_EINVAL;
        if (l->h_seq_len[b] + c > l->h_cap[b]) return KVD_ECAPACITY;
        cnt[b] = c;
        in_row[b] = acc;
        acc += c;
    }
    if (acc > (int64_t(1) << 31) - 1) return KVD_EINVAL;
    // Rows appended before the freeze point ("pre") and after it.
    std::vector<int64_t> pre(ns);
    std::vector<uint8_t> freeze(ns, 0);
    const bool quantises = l->mode != KVD_F32 && l->n_live > 0;
    for (int b = 0; b < ns; ++b) {
        pre[b] = cnt[b];
        if (quantises && !l->h_frozen[b] && cnt[b] > 0) {
            const int64_t j = std::max<int64_t>(0, kColWarmup - l->h_seq_len[b]);
            if (j < cnt[b]) {
                pre[b] = j;
                freeze[b] = 1;
            }
        }
    }
    cudaStream_t s = as_stream(stream);
    // Phase A: rows before the freeze point (all rows of most sequences).
    for (int32_t s0 = 0; s0 < ns; s0 += kSlice) {
        AppendTable t;
        t.seq0 = s0;
        t.n = std::min(kSlice, ns - s0);
        int64_t mx = 0;
        bool any = false;
        for (int i = 0; i < t.n; ++i) {
            const int b = s0 + i;
            t.in_row[i] = int32_t(in_row[b]);
            t.start[i] = int32_t(l->h_seq_len[b]);
            t.count[i] = int32_t(pre[b]);
            mx = std::max(mx, pre[b]);
            any = any || pre[b] > 0;
        }
        if (!any) continue;
        kvd_status st = launch_append(l, k, v, t, mx, s);
        if (st != KVD_OK) return st;
    }
    // The host mirror changes only once every launch of the call has gone in
    // (a failed launch leaves it as it was; the device state is then the
    // caller's to reset).
    bool any_freeze = false;
    for (int b = 0; b < ns; ++b) any_freeze = any_freeze || freeze[b];
    if (!any_freeze) {
        for (int b = 0; b < ns; ++b) l->h_seq_len[b] += cnt[b];
        return KVD_OK;
    }
    // Phase B: freeze; phase C: the remaining rows against the new fields.
    kvd_status st = launch_freeze(l, freeze, s);
    if (st != KVD_OK) return st;
    for (int32_t s0 = 0; s0 < ns; s0 += kSlice) {
        AppendTable t;
        t.seq0 = s0;
        t.n = std::min(kSlice, ns - s0);
        int64_t mx = 0;
        bool any = false;
        for (int i = 0; i < t.n; ++i) {
            const int b = s0 + i;
            const int64_t rest = cnt[b] - pre[b];
            t.in_row[i] = int32_t(in_row[b] + pre[b]);
            t.start[i] = int32_t(l->h_seq_len[b] + pre[b]);
            t.count[i] = int32_t(rest);
            mx = std::max(mx, rest);
            any = any || rest > 0;
        }
        if (!any) continue;
        st = launch_append(l, k, v, t, mx, s);
        if (st != KVD_OK) return st;
    }
    for (int b = 0; b < ns; ++b) {
        l->h_seq_len[b] += cnt[b];
        if (freeze[b]) l->h_frozen[b] = 1;
    }
    return KVD_OK;
}

extern "C" kvd_status kv_freeze_colfield(kvd_layer *L, void *stream) {
    KVD_NVTX_RANGE("kv_freeze_colfield");
    Layer *l = checked_layer(L);
    if (l == nullptr) return KVD_EINVAL;
    std::vector<uint8_t> todo(l->n_seq, 0);
    bool any = false;
    for (int b = 0; b < l->n_seq; ++b) {
        todo[b] = freeze_due(l, b) ? 1 : 0;
        any = any || todo[b];
    }
    if (!any) return KVD_OK;
    const kvd_status st = launch_freeze(l, todo, as_stream(stream));
    if (st != KVD_OK) return st;
    for (int b = 0; b < l->n_seq; ++b)
        if (todo[b]) l->h_frozen[b] = 1;
    return KVD_OK;
}
