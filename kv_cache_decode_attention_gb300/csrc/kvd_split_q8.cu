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

// Tensor-core kernels for the q8_2f cache by query heads per group:
// variant 0 = up to 4 (terms packed in the columns), 1 = up to 8 (heads in
// the columns), 2 = up to 16 (heads in the MMA rows); 3 and 4 are 0 and 1
// over the R-SWA int8 mirror (one K scale per row, int8 query codes).
int q8_tc_variant(int hpk) { return hpk <= 4 ? 0 : hpk <= 8 ? 1 : 2; }

cudaError_t split_layer_q8_tc(int variant, const WarpArgs &wa, const LayerSrc &s, const MmaMaps &maps,
                              cudaStream_t st) {
    switch (variant) {
        case 0: return launch_split_warp<true>(wa, s, maps, st);
        case 1: return launch_split_warp<false>(wa, s, maps, st);
        case 2: return launch_split_h16(wa, s, maps, st);
        case 3: return launch_split_warp_rowk<true>(wa, s, maps, st);
        case 4: return launch_split_warp_rowk<false>(wa, s, maps, st);
        default: return cudaErrorInvalidValue;
    }
}

// Workers (resident one-warp CTAs) of a variant on the current device,
// cached per device; 0 if the query fails.
int64_t split_q8_tc_workers(int variant) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static int64_t cache[kMaxDev][5] = {};
    int dev = 0;
    if (variant < 0 || variant > 4 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int64_t &w = cache[dev][variant];
    if (w == 0) {
        switch (variant) {
            case 0: w = split_warp_workers<true>(); break;
            case 1: w = split_warp_workers<false>(); break;
            case 2: w = split_h16_workers(); break;
            case 3: w = split_warp_workers<true, true>(); break;
            default: w = split_warp_workers<false, true>(); break;
        }
    }
    return w;
}

}  // namespace kvd
