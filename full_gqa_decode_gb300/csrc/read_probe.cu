// Read-bandwidth probe: what HBM delivers to a pure read stream on this part.
//
// Every CTA streams its own contiguous slice of a device buffer into a
// 3-stage shared-memory ring with 1-D bulk copies (two 16 KiB copies per
// stage, completion on an mbarrier), two CTAs per SM, no arithmetic.  It
// exists for measurement: the benchmark reports the attention kernel's
// achieved bandwidth against this read ceiling as well as against the
// measured copy figure (which counts a read and a write per byte).
#include "hd_internal.h"

namespace hd {
namespace {

constexpr int kProbeStages = 3;
constexpr int kProbeCopy = 16 * 1024;
constexpr int kProbeStage = 2 * kProbeCopy;
constexpr unsigned long long kProbeWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool probe_wait(uint64_t *bar, uint32_t parity) {
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(su32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > kProbeWaitNs) return false;
    }
}

// Warp 0 lane 0 waits for stages and releases them; warp 1 lane 0 issues copies.
__global__ void __launch_bounds__(64, 2) read_probe_kernel(const uint8_t *base, int64_t stages_per_cta,
                                                           int32_t *timed_out) {
    extern __shared__ uint8_t raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kProbeStages * kProbeStage);
    uint64_t *empty = full + kProbeStages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kProbeStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&empty[s])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint8_t *src = base + (size_t)blockIdx.x * stages_per_cta * kProbeStage;
    if (threadIdx.x == 32) {
        for (int64_t s = 0; s < stages_per_cta; ++s) {
            const int slot = (int)(s % kProbeStages);
            if (s >= kProbeStages && !probe_wait(&empty[slot], (uint32_t)((s / kProbeStages) - 1) & 1)) {
                atomicOr(timed_out, 1);
                break;
            }
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[slot])),
                         "r"(kProbeStage)
                         : "memory");
            for (int h = 0; h < 2; ++h)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        su32(sm + slot * kProbeStage + h * kProbeCopy)),
                    "l"(src + s * kProbeStage + h * kProbeCopy), "r"(kProbeCopy), "r"(su32(&full[slot]))
                    : "memory");
        }
    } else if (threadIdx.x == 0) {
        for (int64_t s = 0; s < stages_per_cta; ++s) {
            const int slot = (int)(s % kProbeStages);
            if (!probe_wait(&full[slot], (uint32_t)(s / kProbeStages) & 1)) {
                atomicOr(timed_out, 2);
                break;
            }
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(&empty[slot])) : "memory");
        }
    }
    __syncthreads();
}

__device__ int32_t g_probe_timeout;

}  // namespace
}  // namespace hd

extern "C" hd_status hybrid_decode_read_probe(const void *buffer, int64_t bytes, void *stream) {
    using namespace hd;
    if (!buffer || bytes <= 0 || (reinterpret_cast<uintptr_t>(buffer) & 15)) return HD_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return HD_ERR_STATE;
    const int ctas = 2 * sms;
    const int64_t stages = bytes / kProbeStage / ctas;
    if (stages < 1) return HD_ERR_INVALID_ARG;
    const size_t smem = 128 + kProbeStages * kProbeStage + 2 * kProbeStages * sizeof(uint64_t);
    static std::atomic<uint64_t> configured{0};   // devices whose attribute is set
    int device = -1;
    if (!hd::done_on_device(configured, &device)) {
        if (cudaFuncSetAttribute(read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return HD_ERR_CUDA;
        hd::mark_done_on_device(configured, device);
    }
    int32_t *flag = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&flag), g_probe_timeout) != cudaSuccess) return HD_ERR_CUDA;
    read_probe_kernel<<<ctas, 64, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(buffer), stages, flag);
    return cudaGetLastError() == cudaSuccess ? HD_OK : HD_ERR_CUDA;
}
