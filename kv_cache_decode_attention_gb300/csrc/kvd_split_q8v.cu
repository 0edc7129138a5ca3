// kvd_split_q8v.cu -- split-KV decode kernels for the q8v storage mode
// (K quantised: false, V quantised: true), one instance per head dim and
// query-heads-per-group bucket.  Kept in its own unit so the four storage
// modes compile in parallel.
#include "kvd_decode_kernels.cuh"

namespace kvd {

cudaError_t split_layer_q8v(int hd, int hpk_bucket, const SplitArgs &a, const LayerSrc &s,
                               dim3 grid, cudaStream_t st) {
#define KVD_CASE(HD, HPK)                                                               \
    if (hd == HD && hpk_bucket == HPK)                                                 \
        return launch_split_layer_impl<HD, HPK, false, true>(a, s, grid, st);
    KVD_CASE(128, 1) KVD_CASE(128, 2) KVD_CASE(128, 4) KVD_CASE(128, 8) KVD_CASE(128, 16)
    KVD_CASE(64, 1) KVD_CASE(64, 2) KVD_CASE(64, 4) KVD_CASE(64, 8) KVD_CASE(64, 16)
#undef KVD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvd
