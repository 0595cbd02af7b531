// launch_impl.cuh -- template dispatch from a LaunchReq to one kernel instance.
#pragma once

#include <atomic>

#include "launch.h"
#include "stream_kernel.cuh"

namespace hsp {

constexpr int kMaxDevices = 64;
constexpr int kMaxDynamicSmem = 232448;  // 227 KiB, the per-block opt-in limit of sm_103

template <int COMPUTE, int MT, int RT, int WR, int WK, bool TENSOR, bool NORM>
cudaError_t launch_one(const LaunchReq &r) {
    auto kern = hsp_stream_kernel<COMPUTE, MT, RT, WR, WK, TENSOR, NORM>;
    // The shared-memory opt-in is per function and per context; set it once in each.
    static std::atomic<uint64_t> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!set_up_in_current_context(configured[dev])) {
        // the opt-in limit covers static and dynamic shared memory together
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxDynamicSmem - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        // clusters of 16 K slices (fp32 rows with many tokens) exceed the portable 8
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[dev].store(current_context_id(), std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = r.grid;
    cfg.blockDim = dim3(StreamCfg<COMPUTE, MT, RT, WR, WK>::kThreads, 1, 1);
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

template <int COMPUTE, int MT, int RT, int WR, int WK>
cudaError_t launch_variant(const LaunchReq &r) {
    if constexpr (COMPUTE == kMmaBf16 && MT == 1) {
        // the RMSNorm epilogue (bf16, M <= 8) has instances of its own
        if (r.args.norm.active)
            return r.tensor ? launch_one<COMPUTE, MT, RT, WR, WK, true, true>(r)
                            : launch_one<COMPUTE, MT, RT, WR, WK, false, true>(r);
    } else {
        if (r.args.norm.active) return cudaErrorInvalidConfiguration;
    }
    return r.tensor ? launch_one<COMPUTE, MT, RT, WR, WK, true, false>(r)
                    : launch_one<COMPUTE, MT, RT, WR, WK, false, false>(r);
}

// fp32 FMA above 8 tokens: eight K warps (one 16-byte chunk of every unit each) over
// 16 to 64 row slots; 33-64 tokens take at most 48 (12 x 8 register tiles per lane).
template <int MT>
cudaError_t launch_fp32_chunk(const LaunchReq &r) {
    switch (r.RT) {
        case 1: return launch_variant<kFmaFp32, MT, 1, 1, 8>(r);
        case 2: return launch_variant<kFmaFp32, MT, 2, 1, 8>(r);
        case 3: return launch_variant<kFmaFp32, MT, 3, 1, 8>(r);
        case 4:
            if constexpr (MT < 8) return launch_variant<kFmaFp32, MT, 4, 1, 8>(r);
            break;
        default:
            break;
    }
    return cudaErrorInvalidConfiguration;
}

template <int COMPUTE>
cudaError_t launch_compute(const LaunchReq &r) {
    const bool rt1 = (r.RT == 1);
    if constexpr (COMPUTE == kFmaFp32) {
        if (r.bucket > 0) {
            if (r.MT == 2) return launch_fp32_chunk<2>(r);
            if (r.MT == 4) return launch_fp32_chunk<4>(r);
            if (r.MT == 8) return launch_fp32_chunk<8>(r);
            return cudaErrorInvalidConfiguration;
        }
    }
    switch (r.bucket) {
        case 0:
            if (r.MT != 1) break;
            return rt1 ? launch_variant<COMPUTE, 1, 1, 1, 8>(r) : launch_variant<COMPUTE, 1, 2, 1, 8>(r);
        case 1:
            if constexpr (COMPUTE != kFmaFp32) {
                if (r.MT == 2)
                    return rt1 ? launch_variant<COMPUTE, 2, 1, 2, 4>(r) : launch_variant<COMPUTE, 2, 2, 2, 4>(r);
                if (r.MT == 4)
                    return rt1 ? launch_variant<COMPUTE, 4, 1, 2, 4>(r) : launch_variant<COMPUTE, 4, 2, 2, 4>(r);
            }
            break;
        case 2:
            if constexpr (COMPUTE != kFmaFp32) {
                if (r.MT == 8)
                    return rt1 ? launch_variant<COMPUTE, 8, 1, 2, 4>(r) : launch_variant<COMPUTE, 8, 2, 2, 4>(r);
            }
            break;
        default:
            break;
    }
    return cudaErrorInvalidConfiguration;
}

}  // namespace hsp
