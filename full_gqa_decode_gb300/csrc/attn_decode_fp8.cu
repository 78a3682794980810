// Single-layer launches of the attention kernel (attn_kernel.cuh) for E4M3 caches.
#include "attn_kernel.cuh"

namespace hd {

cudaError_t launch_layer_fp8(const LaunchTable<1> &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                             bool pdl, cudaStream_t s) {
    return launch_kv<KV_FP8, 1>(t, grid, rows, mt, consumer, stages, pdl, s);
}

}  // namespace hd
