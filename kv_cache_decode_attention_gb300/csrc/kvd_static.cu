// kvd_static.cu -- decode_attention_static: decode attention for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc on their decode path: an inference
// runtime whose device memory is planned up front and handed out from a fixed
// arena, a plug-in inside a host application that owns every allocation, or
// code that must not take cudaMalloc's implicit device-wide synchronisation
// in the middle of serving.  They can still supply the inputs and outputs of
// a call, but not the scratch space the split-KV decode needs for its
// per-chunk partial results.  This entry point takes that scratch from a
// fixed-size array compiled into the library instead.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds it until the process exits.  Host code may not use the
// array's name as a device address (on the host it is only a stand-in), so
// the first call on each device looks its device address up with
// cudaGetSymbolAddress, with that device current, and keeps it together with
// the id of the device's current context; a later call under another context
// (the device was reset, which unloads the module) looks the address up
// again.  Because the first call on a device (and the first after a reset)
// does this set-up, it should come before any stream capture.
// Every call shares the one array per device and leaves its contents behind;
// the partials are fully rewritten before they are read, so nothing in it
// must start at zero.  Two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on the array and give undefined
// results: callers must serialise them.

#include <algorithm>
#include <cmath>
#include <mutex>

#include <cuda.h>

#include "kvd_decode_kernels.cuh"

namespace kvd {

cudaError_t split_layer_f32(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
cudaError_t split_layer_q8(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
cudaError_t split_layer_q8k(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);
cudaError_t split_layer_q8v(int, int, const SplitArgs &, const LayerSrc &, dim3, cudaStream_t);

namespace {

// Maximum scratch of one call: 16 MiB of partial results.
constexpr int64_t kStaticScratchBytes = int64_t(16) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
unsigned long long g_static_ctx[kMaxDevices] = {};

// Id of the calling thread's current context (0 if the driver cannot tell).
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static std::once_flag once;
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(fn);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device (looked up once
// per device and context), or null if the lookup fails.
void *static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_mu);
    // (before the first lookup no context may be current yet: the lookup
    // makes the device's primary context current, then its id is taken)
    if (g_static_ptr[dev] == nullptr || g_static_ctx[dev] != current_context_id()) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = current_context_id();
    }
    return g_static_ptr[dev];
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status decode_attention_static(const float *q, const kvd_layer *L, int32_t n_q,
                                              float scale, float *out, void *stream) {
    KVD_NVTX_RANGE("decode_attention_static");
    const Layer *l = checked_layer(L);
    if (l == nullptr || q == nullptr || out == nullptr) return KVD_EINVAL;
    if (n_q < l->n_kv || n_q % l->n_kv != 0 || n_q / l->n_kv > kMaxHpk) return KVD_EINVAL;
    if (!std::isfinite(scale)) return KVD_EINVAL;
    if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) != 0)
        return KVD_EINVAL;
    const int hpk = n_q / l->n_kv;
    int64_t work = 0, max_len = 0;
    for (int b = 0; b < l->n_seq; ++b) {
        work += l->h_seq_len[b] * int64_t(l->n_live);
        max_len = std::max(max_len, l->h_seq_len[b]);
    }
    // the same chunking as decode_attention (one definition, kvd_internal.cuh)
    const int32_t chunk = pick_chunk(work);
    const int32_t nc = int32_t(std::max<int64_t>(1, ceil_div(max_len, chunk)));
    const int32_t n_grp = std::max(1, l->n_live);
    // Partials of this call: (max, sum, accumulator[hd]) per head per chunk.
    const int64_t P = int64_t(l->n_seq) * n_grp * nc * hpk;
    const int64_t off_pl = round_up(P * 4, 256), off_pacc = off_pl + round_up(P * 4, 256);
    const int64_t need = off_pacc + round_up(P * l->hd * 4, 256);
    if (need > kStaticScratchBytes) return KVD_ECAPACITY;
    char *ws = static_cast<char *>(static_scratch());
    if (ws == nullptr) return KVD_ECUDA;
    cudaStream_t st = as_stream(stream);

    SplitArgs a;
    a.q = q;
    a.n_q = n_q;
    a.hpk = hpk;
    a.qscale = scale * kLog2e;
    a.chunk = chunk;
    a.nc_max = nc;
    a.n_grp = n_grp;
    a.pm = reinterpret_cast<float *>(ws);
    a.pl = reinterpret_cast<float *>(ws + off_pl);
    a.pacc = reinterpret_cast<float *>(ws + off_pacc);
    a.scores = nullptr;
    a.err = l->d_err;
    if (max_len > 0 && l->n_live > 0) {
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
    m.n_grp = n_grp;
    m.nc_max = nc;
    m.chunk = chunk;
    MergeLayerSrc ms;
    ms.seq_len = l->d_seq_len;
    ms.slot = l->d_slot;
    ms.vcol = static_cast<const float *>(l->buf[KVD_BUF_VCOL]);
    ms.n_live = l->n_live;
    dim3 mgrid(unsigned(n_q), unsigned(l->n_seq));
    if (l->hd == 128) merge_layer_kernel<128><<<mgrid, 128, 0, st>>>(m, ms);
    else merge_layer_kernel<64><<<mgrid, 64, 0, st>>>(m, ms);
    return launch_status() == cudaSuccess ? KVD_OK : KVD_ECUDA;
}
