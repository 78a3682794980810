// Single-layer launches of the attention kernel (attn_kernel.cuh) for E4M3 caches.
#include "attn_kernel.cuh"

namespace hd {

int layer_cluster_limit_fp8(int group) {
    switch (group) {
    case 1: return cluster_limit_g<1, KV_FP8>();
    case 2: return cluster_limit_g<2, KV_FP8>();
    case 4: return cluster_limit_g<4, KV_FP8>();
    case 8: return cluster_limit_g<8, KV_FP8>();
    default: return 0;
    }
}

cudaError_t launch_layer_fp8(const LaunchTable<1> &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                             bool pdl, cudaStream_t s) {
    return launch_kv<KV_FP8, 1>(t, grid, rows, mt, consumer, stages, pdl, s);
}

}  // namespace hd
