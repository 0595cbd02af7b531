// kernels_reg.cu -- the register-ring kernel instance and its launch.
#include <atomic>

#include "launch.h"
#include "reg_kernel.cuh"

namespace hsp {

namespace {

template <bool NORM>
cudaError_t launch_reg_variant(const RegLaunchReq &r) {
    auto kern = hsp_reg_kernel<kRegDepth, NORM>;
    constexpr int kMaxDev = 64;
    static std::atomic<uint64_t> configured[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (!set_up_in_current_context(configured[dev])) {
        // the opt-in limit covers static and dynamic shared memory together
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 232448 - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        configured[dev].store(current_context_id(), std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = r.grid;
    cfg.blockDim = dim3(kRegThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(r.smem_bytes);
    cfg.stream = r.stream;
    cudaLaunchAttribute attrs[1];
    unsigned n = 0;
    if (r.pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, r.tmap_x, r.args);
}

}  // namespace

cudaError_t launch_reg(const RegLaunchReq &r) {
    return r.args.norm.active ? launch_reg_variant<true>(r) : launch_reg_variant<false>(r);
}

}  // namespace hsp
