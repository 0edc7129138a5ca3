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
// cudaGetSymbolAddress, with that device current, and keeps it.  Because that
// first call does this set-up, it should come before any stream capture.
// Every call shares the one array per device and leaves its contents behind;
// the partials are fully rewritten before they are read, so nothing in it
// must start at zero.  Two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on the array and give undefined
// results: callers must serialise them.

#include <algorithm>
#include <cmath>
#include <mutex>

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

// Device address of the scratch array on the current device (looked up once
// per device), or null if the lookup fails.
void *static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        g_static_ptr[dev] = p;
    }
    return g_static_ptr[dev];
}

constexpr int kMinChunkRows = 256;
constexpr int kMaxChunkRows = 2048;
constexpr int64_t kCtaTarget = 152 * 8;

int64_t up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t x, int64_t a) { return (x + a - 1) / a; }

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status decode_attention_static(const float *q, const kvd_layer *L, int32_t n_q,
                                              float scale, float *out, void *stream) {
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
    // the same chunking as decode_attention
    const int32_t chunk = int32_t(std::min<int64_t>(
        kMaxChunkRows, up(std::max<int64_t>(kMinChunkRows, cdiv(work, kCtaTarget)), kMinChunkRows)));
    const int32_t nc = int32_t(std::max<int64_t>(1, cdiv(max_len, chunk)));
    const int32_t n_grp = std::max(1, l->n_live);
    // Partials of this call: (max, sum, accumulator[hd]) per head per chunk.
    const int64_t P = int64_t(l->n_seq) * n_grp * nc * hpk;
    const int64_t off_pl = up(P * 4, 256), off_pacc = off_pl + up(P * 4, 256);
    const int64_t need = off_pacc + up(P * l->hd * 4, 256);
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
        dim3 grid(unsigned(cdiv(max_len, chunk)), unsigned(l->n_live), unsigned(l->n_seq));
        int hb = 1;
        while (hb < hpk) hb <<= 1;
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
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ECUDA;
}
