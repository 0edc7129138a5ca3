// kvd_split_q8.cu -- split-KV decode kernels for the q8 storage mode
// (K quantised: true, V quantised: true), one instance per head dim and
// query-heads-per-group bucket.  Kept in its own unit so the four storage
// modes compile in parallel.
#include <mutex>

#include "kvd_split_h16.cuh"

namespace kvd {

cudaError_t split_layer_q8(int hd, int hpk_bucket, const SplitArgs &a, const LayerSrc &s,
                               dim3 grid, cudaStream_t st) {
#define KVD_CASE(HD, HPK)                                                               \
    if (hd == HD && hpk_bucket == HPK)                                                 \
        return launch_split_layer_impl<HD, HPK, true, true>(a, s, grid, st);
    KVD_CASE(128, 1) KVD_CASE(128, 2) KVD_CASE(128, 4) KVD_CASE(128, 8) KVD_CASE(128, 16)
    KVD_CASE(64, 1) KVD_CASE(64, 2) KVD_CASE(64, 4) KVD_CASE(64, 8) KVD_CASE(64, 16)
#undef KVD_CASE
    return cudaErrorInvalidValue;
}

// Tensor-core kernels for the q8_2f cache: heads in N for groups of up to 8
// query heads, heads in M for groups of 9..16 (nt = 1, 2).
cudaError_t split_layer_q8_warp(int nt, const WarpArgs &wa, const LayerSrc &s, const MmaMaps &maps,
                                cudaStream_t st) {
    if (nt == 1) return launch_split_warp<1>(wa, s, maps, st);
    if (nt == 2) return launch_split_h16(wa, s, maps, st);
    return cudaErrorInvalidValue;
}

// Workers (resident one-warp CTAs) of that kernel on the current device,
// cached per device; 0 if the query fails.
int64_t split_q8_warp_workers(int nt) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static int64_t cache[kMaxDev][2] = {};
    int dev = 0;
    if (nt < 1 || nt > 2 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int64_t &w = cache[dev][nt - 1];
    if (w == 0) w = nt == 1 ? split_warp_workers<1>() : split_h16_workers();
    return w;
}

}  // namespace kvd
