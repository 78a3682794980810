// Step-table launches of the attention kernel (attn_kernel.cuh) for bf16
// caches: every layer of a decode step in one grid.
#include "attn_kernel.cuh"

namespace hd {

cudaError_t launch_step_bf16(const StepTable &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                             cudaStream_t s) {
    return launch_kv<KV_BF16, kStepLayers>(t, grid, rows, mt, consumer, stages, false, s);
}

}  // namespace hd
