// kvd_layer.cu -- layer layout, binding, reset and host-mirrored queries.
//
// The layer is cortiq's LayerKvCache batched over sequences: per sequence,
// one contiguous row region per live KV head ("head-major": a head's rows
// are a straight slice, dead heads store nothing).  The library computes
// where each region lives; the caller allocates the buffers.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvd_internal.cuh"

namespace kvd {

namespace {

struct Shape {
    int32_t n_seq, n_kv, hd, mode, n_live, ng;
    std::vector<int64_t> cap;  // rounded
    int64_t total_rows, imp_len, max_cap;
};

kvd_status make_shape(int32_t n_seq, int32_t n_kv, int32_t hd, int32_t mode,
                      const int64_t *capacity, const uint8_t *alive, Shape *s) {
    if (n_seq < 1 || n_kv < 1 || n_kv > 1024 || (hd != 64 && hd != 128) || mode < 0 || mode > 3 ||
        capacity == nullptr)
        return KVD_EINVAL;
    s->n_seq = n_seq;
    s->n_kv = n_kv;
    s->hd = hd;
    s->mode = mode;
    s->ng = hd / kKGroup;
    s->n_live = 0;
    for (int h = 0; h < n_kv; ++h) s->n_live += (alive == nullptr || alive[h]) ? 1 : 0;
    s->cap.resize(n_seq);
    s->total_rows = 0;
    s->imp_len = 0;
    s->max_cap = 0;
    const int64_t kMaxRows = int64_t(1) << 40;
    for (int b = 0; b < n_seq; ++b) {
        if (capacity[b] < 0 || capacity[b] > (int64_t(1) << 31) - 64) return KVD_EINVAL;
        int64_t c = round_up(capacity[b], kRowAlign);
        s->cap[b] = c;
        s->total_rows += c * s->n_live;
        s->imp_len += c;
        if (c > s->max_cap) s->max_cap = c;
        if (s->total_rows > kMaxRows) return KVD_EINVAL;
    }
    return KVD_OK;
}

MetaLayout meta_layout(int32_t n_seq, int32_t n_kv) {
    MetaLayout m;
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        int64_t at = o;
        o = round_up(o + bytes, 16);
        return at;
    };
    m.row_base = take(8 * int64_t(n_seq));
    m.cap = take(8 * int64_t(n_seq));
    m.imp_base = take(8 * int64_t(n_seq));
    m.seq_len = take(4 * int64_t(n_seq));
    m.frozen = take(4 * int64_t(n_seq));
    m.live = take(4 * int64_t(n_kv));
    m.slot = take(4 * int64_t(n_kv));
    m.err = take(16);
    m.total = round_up(o, 256);
    return m;
}

// Device bytes per slot; row buffers carry kRowAlign spare rows at the end so
// that a bulk copy rounded up to kRowAlign rows never leaves the buffer.
void slot_bytes(const Shape &s, int64_t *out) {
    const int64_t rows = s.total_rows + kRowAlign;
    for (int i = 0; i < KVD_BUF_COUNT; ++i) out[i] = 0;
    const bool qk = quant_k(s.mode), qv = quant_v(s.mode);
    if (qk) {
        out[KVD_BUF_KQ] = rows * s.hd;
        out[KVD_BUF_KS] = rows * s.ng * 4;
        out[KVD_BUF_KCOL] = int64_t(s.n_seq) * s.n_live * s.hd * 4;
    } else {
        out[KVD_BUF_K] = rows * s.hd * 4;
    }
    if (qv) {
        out[KVD_BUF_VQ] = rows * s.hd;
        out[KVD_BUF_VS] = rows * 4;
        out[KVD_BUF_VCOL] = int64_t(s.n_seq) * s.n_live * s.hd * 4;
    } else {
        out[KVD_BUF_V] = rows * s.hd * 4;
    }
    for (int i = 0; i < KVD_BUF_COUNT; ++i) out[i] = round_up(out[i], 256);
    out[KVD_BUF_META] = meta_layout(s.n_seq, s.n_kv).total;
}

int64_t host_block_bytes(int32_t n_seq, int32_t n_kv) {
    return 8 * 4 * int64_t(n_seq) + 4 * int64_t(n_seq) + 8 * int64_t(n_kv) + round_up(n_kv, 8);
}

}  // namespace

// TMA descriptor of an int8 code buffer: 2-D [rows][hd] bytes, row pitch hd,
// boxes of 32 rows x 128 bytes landing in shared memory with the 128-byte
// swizzle (16-byte chunk c of row r stored at chunk c ^ (r % 8)); rows past
// the end read as zeros.  Returns false if the driver entry point is missing
// or refuses the descriptor (the caller then uses the plain bulk-copy kernel).
bool encode_code_map(void *base, int64_t rows, int hd, unsigned char *out) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (encode == nullptr || hd != 128) return false;
    alignas(64) CUtensorMap m;
    const cuuint64_t dims[2] = {cuuint64_t(hd), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(hd)};
    const cuuint32_t box[2] = {128u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    if (encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
    std::memcpy(out, &m, sizeof(m));
    return true;
}

namespace {

__global__ void fill_f32_kernel(float *p, int64_t n, float v) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        p[i] = v;
}

// Reset sequences [seq0, seq0 + n): length 0, not frozen, fields 1.0.
__global__ void reset_kernel(int32_t *seq_len, int32_t *frozen, float *kcol, float *vcol,
                             int32_t seq0, int32_t n, int64_t field_elems_per_seq) {
    const int32_t b = seq0 + blockIdx.y;
    if (blockIdx.y >= n) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        seq_len[b] = 0;
        frozen[b] = 0;
    }
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < field_elems_per_seq;
         i += int64_t(gridDim.x) * blockDim.x) {
        if (kcol) kcol[b * field_elems_per_seq + i] = 1.0f;
        if (vcol) vcol[b * field_elems_per_seq + i] = 1.0f;
    }
}

}  // namespace

const Layer *checked_layer(const kvd_layer *L) {
    if (L == nullptr) return nullptr;
    const Layer *l = as_layer(L);
    return l->magic == kLayerMagic ? l : nullptr;
}

Layer *checked_layer(kvd_layer *L) {
    if (L == nullptr) return nullptr;
    Layer *l = as_layer(L);
    return l->magic == kLayerMagic ? l : nullptr;
}

}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_layer_bytes(int32_t n_seq, int32_t n_kv, int32_t head_dim, int32_t mode,
                                      const int64_t *capacity, const uint8_t *alive,
                                      int64_t *bytes_out, int64_t *host_bytes_out) {
    if (bytes_out == nullptr || host_bytes_out == nullptr) return KVD_EINVAL;
    Shape s;
    kvd_status st = make_shape(n_seq, n_kv, head_dim, mode, capacity, alive, &s);
    if (st != KVD_OK) return st;
    slot_bytes(s, bytes_out);
    *host_bytes_out = host_block_bytes(n_seq, n_kv);
    return KVD_OK;
}

extern "C" kvd_status kvd_layer_init(kvd_layer *L, int32_t n_seq, int32_t n_kv, int32_t head_dim,
                                     int32_t mode, const int64_t *capacity, const uint8_t *alive,
                                     void *const *dev_bufs, void *host_state, void *stream) {
    if (L == nullptr || dev_bufs == nullptr || host_state == nullptr) return KVD_EINVAL;
    Shape s;
    kvd_status st = make_shape(n_seq, n_kv, head_dim, mode, capacity, alive, &s);
    if (st != KVD_OK) return st;
    int64_t need[KVD_BUF_COUNT];
    slot_bytes(s, need);
    for (int i = 0; i < KVD_BUF_COUNT; ++i) {
        const bool used = need[i] > 0;
        if (used && dev_bufs[i] == nullptr) return KVD_EINVAL;
        if (used && (reinterpret_cast<uintptr_t>(dev_bufs[i]) & 255) != 0) return KVD_EINVAL;
    }
    Layer l;
    std::memset(&l, 0, sizeof(l));
    l.magic = kLayerMagic;
    l.mode = mode;
    l.n_seq = n_seq;
    l.n_kv = n_kv;
    l.hd = head_dim;
    l.n_live = s.n_live;
    l.ng = s.ng;
    l.total_rows = s.total_rows;
    l.imp_len = s.imp_len;
    l.max_cap = s.max_cap;
    for (int i = 0; i < KVD_BUF_COUNT; ++i) l.buf[i] = need[i] > 0 ? dev_bufs[i] : nullptr;
    l.ml = meta_layout(n_seq, n_kv);

    // host block
    char *h = static_cast<char *>(host_state);
    l.h_cap = reinterpret_cast<int64_t *>(h);
    l.h_row_base = l.h_cap + n_seq;
    l.h_imp_base = l.h_row_base + n_seq;
    l.h_seq_len = l.h_imp_base + n_seq;
    l.h_frozen = reinterpret_cast<int32_t *>(l.h_seq_len + n_seq);
    l.h_live = l.h_frozen + n_seq;
    l.h_slot = l.h_live + n_kv;
    l.h_alive = reinterpret_cast<uint8_t *>(l.h_slot + n_kv);
    int64_t rb = 0, ib = 0;
    for (int b = 0; b < n_seq; ++b) {
        l.h_cap[b] = s.cap[b];
        l.h_row_base[b] = rb;
        l.h_imp_base[b] = ib;
        l.h_seq_len[b] = 0;
        l.h_frozen[b] = 0;
        rb += s.cap[b] * s.n_live;
        ib += s.cap[b];
    }
    int gl = 0;
    for (int hh = 0; hh < n_kv; ++hh) {
        l.h_alive[hh] = (alive == nullptr || alive[hh]) ? 1 : 0;
        l.h_slot[hh] = l.h_alive[hh] ? gl : -1;
        if (l.h_alive[hh]) l.h_live[gl++] = hh;
    }
    for (int i = gl; i < n_kv; ++i) l.h_live[i] = -1;

    // device metadata: staged once, uploaded with one copy
    char *meta = static_cast<char *>(dev_bufs[KVD_BUF_META]);
    l.d_row_base = reinterpret_cast<int64_t *>(meta + l.ml.row_base);
    l.d_cap = reinterpret_cast<int64_t *>(meta + l.ml.cap);
    l.d_seq_len = reinterpret_cast<int32_t *>(meta + l.ml.seq_len);
    l.d_frozen = reinterpret_cast<int32_t *>(meta + l.ml.frozen);
    l.d_live = reinterpret_cast<int32_t *>(meta + l.ml.live);
    l.d_slot = reinterpret_cast<int32_t *>(meta + l.ml.slot);
    l.d_err = reinterpret_cast<uint32_t *>(meta + l.ml.err);
    std::vector<char> stage(l.ml.total, 0);
    std::memcpy(stage.data() + l.ml.row_base, l.h_row_base, 8 * size_t(n_seq));
    std::memcpy(stage.data() + l.ml.cap, l.h_cap, 8 * size_t(n_seq));
    std::memcpy(stage.data() + l.ml.imp_base, l.h_imp_base, 8 * size_t(n_seq));
    std::memcpy(stage.data() + l.ml.live, l.h_live, 4 * size_t(n_kv));
    std::memcpy(stage.data() + l.ml.slot, l.h_slot, 4 * size_t(n_kv));
    cudaStream_t cs = as_stream(stream);
    // Pageable source: the copy is staged before cudaMemcpyAsync returns.
    if (cudaMemcpyAsync(meta, stage.data(), stage.size(), cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        fault_fires())
        return KVD_ECUDA;
    const int64_t fe = int64_t(n_seq) * s.n_live * head_dim;
    if (fe > 0) {
        if (l.buf[KVD_BUF_KCOL]) {
            fill_f32_kernel<<<608, 256, 0, cs>>>(static_cast<float *>(l.buf[KVD_BUF_KCOL]), fe,
                                                     1.0f);
        }
        if (l.buf[KVD_BUF_VCOL]) {
            fill_f32_kernel<<<608, 256, 0, cs>>>(static_cast<float *>(l.buf[KVD_BUF_VCOL]), fe,
                                                     1.0f);
        }
        if (launch_status() != cudaSuccess) return KVD_ECUDA;
    }
    const int64_t code_rows = s.total_rows + kRowAlign;
    if (l.buf[KVD_BUF_KQ])
        l.have_tmap_kq = encode_code_map(l.buf[KVD_BUF_KQ], code_rows, head_dim, l.tmap_kq) ? 1 : 0;
    if (l.buf[KVD_BUF_VQ])
        l.have_tmap_vq = encode_code_map(l.buf[KVD_BUF_VQ], code_rows, head_dim, l.tmap_vq) ? 1 : 0;
    std::memcpy(L, &l, sizeof(l));
    return KVD_OK;
}

extern "C" kvd_status kvd_layer_reset(kvd_layer *L, int32_t seq, void *stream) {
    KVD_NVTX_RANGE("kvd_layer_reset");
    Layer *l = checked_layer(L);
    if (l == nullptr || seq < -1 || seq >= l->n_seq) return KVD_EINVAL;
    const int32_t seq0 = seq < 0 ? 0 : seq, n = seq < 0 ? l->n_seq : 1;
    const int64_t fe = int64_t(l->n_live) * l->hd;
    for (int32_t s0 = seq0; s0 < seq0 + n; s0 += 65535) {
        const int32_t cnt = (seq0 + n - s0) < 65535 ? (seq0 + n - s0) : 65535;
        dim3 grid(1, cnt);
        reset_kernel<<<grid, 128, 0, as_stream(stream)>>>(
            l->d_seq_len, l->d_frozen, static_cast<float *>(l->buf[KVD_BUF_KCOL]),
            static_cast<float *>(l->buf[KVD_BUF_VCOL]), s0, cnt, fe);
    }
    if (launch_status() != cudaSuccess) return KVD_ECUDA;
    for (int32_t b = seq0; b < seq0 + n; ++b) {
        l->h_seq_len[b] = 0;
        l->h_frozen[b] = 0;
    }
    return KVD_OK;
}

extern "C" kvd_status kvd_layer_seq_len(const kvd_layer *L, int32_t seq, int64_t *len_out,
                                        int32_t *frozen_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || seq < 0 || seq >= l->n_seq) return KVD_EINVAL;
    if (len_out) *len_out = l->h_seq_len[seq];
    if (frozen_out) *frozen_out = l->h_frozen[seq];
    return KVD_OK;
}

extern "C" kvd_status kvd_layer_memory_bytes(const kvd_layer *L, int64_t *bytes_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || bytes_out == nullptr) return KVD_EINVAL;
    const bool qk = quant_k(l->mode), qv = quant_v(l->mode);
    int64_t total = 0;
    for (int b = 0; b < l->n_seq; ++b) {
        const int64_t rows = l->h_seq_len[b] * int64_t(l->n_live);
        total += qk ? rows * l->hd + rows * l->ng * 4 : rows * l->hd * 4;
        total += qv ? rows * l->hd + rows * 4 : rows * l->hd * 4;
        if (l->h_frozen[b]) total += int64_t(l->n_live) * l->hd * 4 * ((qk ? 1 : 0) + (qv ? 1 : 0));
    }
    *bytes_out = total;
    return KVD_OK;
}

extern "C" kvd_status kvd_layer_device_error(const kvd_layer *L, int32_t clear,
                                             uint32_t *word_out) {
    const Layer *l = checked_layer(L);
    if (l == nullptr) return KVD_EINVAL;
    uint32_t w = 0;
    if (cudaMemcpy(&w, l->d_err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVD_ECUDA;
    if (clear && cudaMemset(l->d_err, 0, 4) != cudaSuccess) return KVD_ECUDA;
    if (word_out) *word_out = w;
    return w ? KVD_EDEVICE : KVD_OK;
}

namespace kvd {
namespace {

// One warp waits for a phase of an mbarrier that nothing completes, as a
// kernel whose copies never land would, gives up after limit_ns and records
// it the way every kernel here does: no trap, the error bit, a normal exit.
__global__ void wait_selftest_kernel(uint32_t *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, limit_ns)) set_error(err, kErrTimeout);
}

}  // namespace
}  // namespace kvd

extern "C" kvd_status kvd_wait_timeout_selftest(const kvd_layer *L, int64_t limit_ns, void *stream) {
    const Layer *l = checked_layer(L);
    if (l == nullptr || limit_ns < 1 || limit_ns > 1000000000) return KVD_EINVAL;
    wait_selftest_kernel<<<1, 32, 0, as_stream(stream)>>>(l->d_err, uint64_t(limit_ns));
    return launch_status() == cudaSuccess ? KVD_OK : KVD_ECUDA;
}

namespace kvd {
std::atomic<int64_t> g_fault_countdown{-1};
}  // namespace kvd

extern "C" kvd_status kvd_test_fail_after(int64_t n) {
    kvd::g_fault_countdown.store(n < 0 ? -1 : n);
    return KVD_OK;
}

extern "C" const char *kvd_status_string(int32_t status) {
    switch (status) {
        case KVD_OK: return "ok";
        case KVD_EINVAL: return "invalid argument";
        case KVD_ECAPACITY: return "capacity exceeded";
        case KVD_ESTATE: return "invalid state (no prefill recorded)";
        case KVD_EEMPTY: return "empty attention key set";
        case KVD_ECUDA: return "CUDA launch or copy failed";
        case KVD_EDEVICE: return "device error word set";
        default: return "unknown status";
    }
}
