// kernels_umma.cu -- instances of the tensor-memory kernel and their launch.
#include <atomic>

#include "launch.h"
#include "umma_kernel.cuh"

namespace hsp {

namespace {

constexpr int kMaxDev = 64;

template <int COMPUTE, int NT>
cudaError_t launch_umma_variant(const UmmaLaunchReq &r) {
    auto kern = hsp_umma_kernel<COMPUTE, NT>;
    static std::atomic<uint64_t> configured[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (!set_up_in_current_context(configured[dev])) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e != cudaSuccess) return e;
        // clusters of 16 K slices (tf32 rows of 16 KB and more) exceed the portable 8
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[dev].store(current_context_id(), std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = r.grid;
    cfg.blockDim = dim3(kUmmaThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(r.smem_bytes);
    cfg.stream = r.stream;
    cudaLaunchAttribute attrs[2];
    unsigned n = 0;
    if (r.grid.y > 1) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = 1;
        attrs[n].val.clusterDim.y = r.grid.y;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    if (r.pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, r.tmap_w, r.tmap_x, r.args);
}

}  // namespace

cudaError_t launch_umma(const UmmaLaunchReq &r) {
    if (r.compute == kMmaBf16) {
        if (r.NT == 16) return launch_umma_variant<kMmaBf16, 16>(r);
        if (r.NT == 32) return launch_umma_variant<kMmaBf16, 32>(r);
        if (r.NT == 64) return launch_umma_variant<kMmaBf16, 64>(r);
    } else if (r.compute == kMmaTf32) {
        if (r.NT == 16) return launch_umma_variant<kMmaTf32, 16>(r);
        if (r.NT == 32) return launch_umma_variant<kMmaTf32, 32>(r);
        if (r.NT == 64) return launch_umma_variant<kMmaTf32, 64>(r);
    }
    return cudaErrorInvalidConfiguration;
}

}  // namespace hsp
