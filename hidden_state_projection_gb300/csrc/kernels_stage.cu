// kernels_stage.cu -- the token staging kernel of the host entry point.
//
// proj_fused_gemm_host takes the tokens X[M, K] in host memory.  When that buffer is
// page-locked and mapped into the device's address space, this kernel copies it into the
// device staging buffer instead of a DMA copy: it is launched on the stream like the
// projection kernel that follows it, so the two are chained by programmatic dependent
// launch rather than by a copy-engine completion (on GB300 a 80 KB copy-engine copy cost
// about 2.5 us per step, most of it start-up).
//
//   * it triggers its dependent launch at entry: the dependent is always the projection
//     kernel of the same call, which issues its weight loads at once and waits on its
//     grid dependency (this kernel's completion and memory flush) before it reads the
//     tokens, so the weight stream starts while the tokens are in transit;
//   * it waits on its own grid dependency before touching either buffer: the previous
//     kernel on the stream (typically the last step's projection) may still read the
//     staging buffer, and it may have written the host buffer;
//   * each thread moves four 16-byte chunks per pass (all four loads before the stores),
//     256 threads per CTA, enough CTAs for one pass when possible.
#include <stdint.h>

#include "launch.h"
#include "ptx.cuh"

namespace hsp {

constexpr int kStageThreads = 256;
constexpr int kStageChunks = 4;  // 16-byte chunks per thread and pass

__global__ void __launch_bounds__(kStageThreads) hsp_stage_kernel(const uint4 *__restrict__ src,
                                                                  uint4 *__restrict__ dst, int64_t n16) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t per_cta = static_cast<int64_t>(kStageThreads) * kStageChunks;
    const int64_t step = static_cast<int64_t>(gridDim.x) * per_cta;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * per_cta + threadIdx.x; i0 < n16; i0 += step) {
        uint4 v[kStageChunks];
#pragma unroll
        for (int j = 0; j < kStageChunks; ++j) {
            const int64_t i = i0 + static_cast<int64_t>(j) * kStageThreads;
            if (i < n16) v[j] = src[i];
        }
#pragma unroll
        for (int j = 0; j < kStageChunks; ++j) {
            const int64_t i = i0 + static_cast<int64_t>(j) * kStageThreads;
            if (i < n16) dst[i] = v[j];
        }
    }
}

cudaError_t launch_stage(const void *src, void *dst, int64_t n16, int max_ctas, int pdl, cudaStream_t stream) {
    const int64_t per_cta = static_cast<int64_t>(kStageThreads) * kStageChunks;
    int64_t ctas = (n16 + per_cta - 1) / per_cta;
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(kStageThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[1];
    unsigned n = 0;
    if (pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, hsp_stage_kernel, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                              n16);
}

}  // namespace hsp
