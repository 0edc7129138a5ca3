// kvd_internal.cuh -- private declarations shared by the library's .cu files.
//
// Layer metadata, the device error word, and the sm_100-family PTX helpers
// used by the kernels: mbarrier waits with a time limit, and 1-D bulk
// asynchronous global->shared copies (the TMA bulk-copy engine).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/kvd.h"

namespace kvd {

constexpr int kColWarmup = 64;  // cortiq KV_COL_WARMUP: rows before the fields freeze
constexpr int kKGroup = 32;     // cortiq KV_K_GROUP: K channels per scale
constexpr int kRowAlign = 16;   // per-sequence capacity is rounded to this many rows
constexpr int kMaxHpk = 16;     // query heads per KV head handled by the kernels
constexpr int kSlice = 256;     // sequences/streams described per launch (kernel params)

// Device error-word bits.
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBounds = 2u;

inline bool quant_k(int mode) { return mode == KVD_Q8 || mode == KVD_Q8K; }

// ---- chunking of the CUDA-core split pass (shared by every entry point
// that launches it, so their grids and partial layouts agree)
constexpr int kMinChunk = 256;           // rows; multiple of every tile height
constexpr int kMaxChunk = 2048;          // rows; bounds one CTA's f32 accumulation chain
constexpr int64_t kTargetCtas = 152 * 8; // about four waves of two CTAs per SM

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t x, int64_t a) { return (x + a - 1) / a; }

// Query heads per group rounded up to the instantiated kernels' bucket (1, 2, 4, 8, 16).
inline int hpk_bucket(int hpk) {
    int b = 1;
    while (b < hpk) b <<= 1;
    return b;
}

// Rows per chunk: a multiple of kMinChunk, large enough that the grid holds
// about kTargetCtas chunks, but at most kMaxChunk.  The cap keeps each CTA's
// sequential f32 accumulation short (its rounding grows like the square root
// of the rows summed, and long diffuse softmaxes shrink the output), at the
// cost of more partials, which are ~0.2% of the bytes.
inline int32_t pick_chunk(int64_t work_rows) {
    const int64_t c = ceil_div(work_rows, kTargetCtas);
    const int64_t r = round_up(c > kMinChunk ? c : kMinChunk, kMinChunk);
    return int32_t(r < kMaxChunk ? r : kMaxChunk);
}
inline bool quant_v(int mode) { return mode == KVD_Q8 || mode == KVD_Q8V; }

// Device metadata block (KVD_BUF_META), laid out by layer_meta_layout().
struct MetaLayout {
    int64_t row_base;  // int64[n_seq]   first storage row of sequence b
    int64_t cap;       // int64[n_seq]   rows per live head of sequence b
    int64_t imp_base;  // int64[n_seq]   first imp entry of sequence b
    int64_t seq_len;   // int32[n_seq]   rows stored
    int64_t frozen;    // int32[n_seq]   1 once the fields are set
    int64_t live;      // int32[n_kv]    live slot -> KV head
    int64_t slot;      // int32[n_kv]    KV head -> live slot (-1 = dead)
    int64_t err;       // uint32          device error word
    int64_t total;     // bytes
};

// Private view of kvd_layer.
struct Layer {
    int32_t magic;
    int32_t mode, n_seq, n_kv, hd, n_live, ng;
    int32_t pad0;
    int64_t total_rows;  // sum_b n_live * cap_b
    int64_t imp_len;     // sum_b cap_b
    int64_t max_cap;     // max_b cap_b
    void *buf[KVD_BUF_COUNT];
    MetaLayout ml;
    // host state block
    int64_t *h_cap, *h_row_base, *h_imp_base, *h_seq_len;
    int32_t *h_frozen, *h_live, *h_slot;
    uint8_t *h_alive;
    // device pointers into the metadata block
    int64_t *d_row_base, *d_cap;
    int32_t *d_seq_len, *d_frozen, *d_live, *d_slot;
    uint32_t *d_err;
    // TMA tensor maps (CUtensorMap, 128 bytes each) of the int8 K and V code
    // buffers, 2-D [rows][head_dim] with 128-byte swizzled [32 x 128] boxes;
    // have_tmap = 0 when they are not built (head_dim 64 or no int8 buffer).
    int32_t have_tmap_kq, have_tmap_vq;
    unsigned char tmap_kq[128], tmap_vq[128];
};
static_assert(sizeof(Layer) <= sizeof(kvd_layer), "kvd_layer too small");
constexpr int32_t kLayerMagic = 0x4b564431;  // "KVD1"

inline Layer *as_layer(kvd_layer *L) { return reinterpret_cast<Layer *>(L); }
inline const Layer *as_layer(const kvd_layer *L) { return reinterpret_cast<const Layer *>(L); }
// An NVTX range named for the entry point around each call that launches work,
// so profilers can attribute kernels to calls (header-only NVTX: a pointer
// check when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define KVD_NVTX_RANGE(name) const ::kvd::NvtxRange kvd_nvtx_range_(name)

const Layer *checked_layer(const kvd_layer *L);
Layer *checked_layer(kvd_layer *L);

// The append and freeze halves of kvd_bounds_selftest (kvd_append.cu).
cudaError_t append_bounds_selftest(const Layer *l, const float *zeros, int32_t *seq_len, int32_t *frozen,
                                   cudaStream_t s);

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Failure injection for tests (kvd_test_fail_after): while armed with n >= 0,
// the (n+1)-th kernel launch or host/device copy that the library issues from
// then on reports failure (cudaErrorLaunchFailure) to its entry point, which
// returns KVD_ECUDA; the counter then disarms itself.  Host-only: the device
// never sees it.
extern std::atomic<int64_t> g_fault_countdown;
inline bool fault_fires() {
    int64_t c = g_fault_countdown.load(std::memory_order_relaxed);
    while (c >= 0 && !g_fault_countdown.compare_exchange_weak(c, c - 1, std::memory_order_relaxed)) {
    }
    return c == 0;
}

// Status of the launches since the last call (cudaGetLastError), or the
// injected failure.
inline cudaError_t launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess && fault_fires() ? cudaErrorLaunchFailure : e;
}

// Programmatic dependent launch.  A kernel that produces data calls
// pdl_trigger() to let the next kernel on the stream (launched with
// launch_pdl) start early; that kernel does the work that does not read the
// producer's output, then pdl_wait(), which returns once the producer grid has
// completed and its memory operations are visible.  Both are no-ops for a
// kernel launched the ordinary way.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    return e == cudaSuccess && fault_fires() ? cudaErrorLaunchFailure : e;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`
// nanoseconds of wall time.  Returns false on time-out (the caller records
// kErrTimeout and unwinds; no trap).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk asynchronous copy global -> shared (cp.async.bulk), completing
// `bytes` of transaction count on `bar`.  dst, src and bytes must be
// multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device):
// the attribute belongs to the function in a device's context, and setting
// it on every launch costs a driver call per launch.
inline cudaError_t set_smem_once(const void *kern, int bytes) {
    struct Done {
        const void *kern;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Done &d : done)
        if (d.kern == kern && d.dev == dev && d.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back(Done{kern, dev, bytes});
    return e;
}

// TMA descriptor (128 bytes, written to out) of an int8 code buffer
// [rows][hd]: boxes of 32 rows x 128 bytes, 128-byte swizzle, rows past the
// end read as zeros.  head_dim 128 only; false if the driver refuses it.
bool encode_code_map(void *base, int64_t rows, int hd, unsigned char *out);

__device__ __forceinline__ void set_error(uint32_t *err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

}  // namespace kvd
