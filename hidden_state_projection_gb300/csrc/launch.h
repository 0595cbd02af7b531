// launch.h -- host-side launch request for the streaming kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "stream_args.h"

namespace hsp {

// Id of the CUDA context current on the calling thread (0: none yet); proj_api.cu.
uint64_t current_context_id();

// Per-device set-up (a kernel's shared-memory opt-in) is recorded as the id of the
// context it was made in: true when that is the current context.  A reset device or
// another context on it gets the set-up again.
inline bool set_up_in_current_context(const std::atomic<uint64_t> &slot) {
    const uint64_t ctx = current_context_id();
    return ctx != 0 && slot.load(std::memory_order_acquire) == ctx;
}

struct LaunchReq {
    int compute;     // Compute
    int bucket;      // 0: (WR, WK) = (1, 8); 1 and 2: (2, 4), fp32 FMA (1, 8)
    int MT;          // token tiles of 8
    int RT;          // 16-row tiles per warp
    int tensor;      // 1: 3-D tensor copies (tmap_w / tmap_x used), 0: 1-D bulk copies
    dim3 grid;       // (row CTAs, slices, 1)
    int smem_bytes;  // dynamic shared memory
    int pdl;         // programmatic stream serialization
    cudaStream_t stream;
    CUtensorMap tmap_w;  // weights viewed as [units][rows][128 bytes], box [stage units][R][128 bytes]
    CUtensorMap tmap_x;  // tokens viewed as [units][M][128 bytes], box [stage units][M][128 bytes]
    StreamArgs args;
};

// Implemented once per element type (kernels_bf16.cu, kernels_tf32.cu, kernels_fp32.cu).
cudaError_t launch_bf16(const LaunchReq &r);
cudaError_t launch_tf32(const LaunchReq &r);
cudaError_t launch_fp32(const LaunchReq &r);

// Tensor-memory kernel launch (9 <= M <= 64).
struct UmmaLaunchReq {
    int compute;     // kMmaBf16 or kMmaTf32
    int NT;          // token tile: 16, 32 or 64
    dim3 grid;       // (128-row tiles, slices, 1)
    int smem_bytes;
    int pdl;
    cudaStream_t stream;
    CUtensorMap tmap_w;
    CUtensorMap tmap_x;
    UmmaArgs args;
};
cudaError_t launch_umma(const UmmaLaunchReq &r);

// Register-ring kernel launch (bf16, M <= 8, rows of at most kRegMaxUnits k-units).
struct RegLaunchReq {
    dim3 grid;       // (row CTAs, 1, 1)
    int smem_bytes;  // the token box + 1024 bytes of alignment slack
    int pdl;
    cudaStream_t stream;
    CUtensorMap tmap_x;  // tokens viewed as [units][M][128 bytes], one box for all of them
    StreamArgs args;     // w, x, row_bytes, n_rows, rows_per_cta, M, units_total, hooks, splits, prefetch, norm
};
cudaError_t launch_reg(const RegLaunchReq &r);
constexpr int kRegThreadsHost = 16 * 32;
constexpr int kRegDepthHost = 5;

// fp32 register GEMV launch (PROJ_FP32, K <= 8192; one token group per CTA along grid.y).
struct GemvLaunchReq {
    dim3 grid;       // (row CTAs, token groups, 1)
    int smem_bytes;  // the tokens of one group: ceil(M / groups) * K * 4
    int pdl;
    cudaStream_t stream;
    StreamArgs args;  // w, x, row_bytes, n_rows, rows_per_cta, M, hooks, splits, prefetch
};
cudaError_t launch_gemv(const GemvLaunchReq &r);
constexpr int kGemvThreadsHost = 16 * 32;
constexpr int kGemvMaxTokenBytes = 192 * 1024;

// Token staging for the host entry point: n16 16-byte chunks from `src` (the device
// address of page-locked host memory) to `dst`, at most max_ctas CTAs, PDL-chained.
cudaError_t launch_stage(const void *src, void *dst, int64_t n16, int max_ctas, int pdl, cudaStream_t stream);

// Weight packer: part p's n16 chunks run from src[p] to chunk dst16[p] of W_cat; the
// parts are laid end to end in the launch (first16[p] = chunks before part p,
// first16[count] = all chunks).  One launch, at most max_ctas CTAs, no PDL attribute.
struct PackArgs {
    int32_t count;
    const uint4 *src[kMaxSplits];
    int64_t dst16[kMaxSplits];
    int64_t first16[kMaxSplits + 1];
};
cudaError_t launch_pack(void *dst, const PackArgs &a, int max_ctas, cudaStream_t stream);

// Threads per CTA of a bucket (eight consumer warps + one producer warp).
constexpr int kThreadsPerCta = 9 * 32;
constexpr int kUmmaThreadsHost = 128;

}  // namespace hsp
