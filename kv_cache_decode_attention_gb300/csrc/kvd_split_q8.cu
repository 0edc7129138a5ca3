// kvd_split_q8.cu -- split-KV decode kernels for the q8 storage mode
// (K quantised: true, V quantised: true), one instance per head dim and
// query-heads-per-group bucket.  Kept in its own unit so the four storage
// modes compile in parallel.
#include "kvd_split_mma.cuh"

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

cudaError_t split_layer_q8_mma(int hpk_bucket, const SplitArgs &a, const LayerSrc &s,
                               const MmaMaps &maps, dim3 grid, cudaStream_t st) {
    switch (hpk_bucket) {
        case 1: return launch_split_mma<1>(a, s, maps, grid, st);
        case 2: return launch_split_mma<2>(a, s, maps, grid, st);
        case 4: return launch_split_mma<4>(a, s, maps, grid, st);
        case 8: return launch_split_mma<8>(a, s, maps, grid, st);
        case 16: return launch_split_mma<16>(a, s, maps, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvd
