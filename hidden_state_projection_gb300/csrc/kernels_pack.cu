// kernels_pack.cu -- the weight packer's copy kernel (proj_pack_weights).
//
// TensorRT-LLM PR #20636, Description: after loading, the projection weights that
// read the same hidden state are copied one after another into a single
// row-concatenated tensor, and the per-projection weights become views of it, so a
// later reload through a view updates the fused weight.  This kernel is the copy:
// up to kMaxSplits source matrices (parts whose source already is its own rows of
// the destination are left out by the host) moved into their rows of W_cat in one
// launch.
//
//   * the parts are laid end to end in 16-byte chunks (every row is a multiple of 16
//     bytes, so every part is); chunk c belongs to the part whose prefix range holds
//     it, and goes to that part's destination offset plus its rank in the part;
//   * each thread moves four chunks per pass (all loads before the stores), grid-stride;
//   * the launch carries no programmatic-serialization attribute (it starts after
//     everything before it on the stream, including projections still reading the old
//     W_cat) and never triggers its dependents early.  Projection kernels request
//     weights before their grid-dependency wait, so every CTA makes its stores visible
//     at GPU scope before it exits: a CTA barrier, then one release fence (cumulative
//     over the barrier) by thread 0.  A projection launched after the pack therefore
//     reads the new weights.
#include <stdint.h>

#include "launch.h"
#include "ptx.cuh"

namespace hsp {

constexpr int kPackThreads = 256;
constexpr int kPackChunks = 4;  // 16-byte chunks per thread and pass

__global__ void __launch_bounds__(kPackThreads) hsp_pack_kernel(uint4 *__restrict__ dst, const PackArgs a) {
    const int64_t total = a.first16[a.count];
    const int64_t per_cta = static_cast<int64_t>(kPackThreads) * kPackChunks;
    const int64_t step = static_cast<int64_t>(gridDim.x) * per_cta;
    for (int64_t c0 = static_cast<int64_t>(blockIdx.x) * per_cta + threadIdx.x; c0 < total; c0 += step) {
        uint4 v[kPackChunks];
        int64_t to[kPackChunks];
#pragma unroll
        for (int j = 0; j < kPackChunks; ++j) {
            const int64_t c = c0 + static_cast<int64_t>(j) * kPackThreads;
            to[j] = -1;
            if (c < total) {
                int p = 0;
                while (p + 1 < a.count && c >= a.first16[p + 1]) ++p;
                const int64_t r = c - a.first16[p];
                v[j] = a.src[p][r];
                to[j] = a.dst16[p] + r;
            }
        }
#pragma unroll
        for (int j = 0; j < kPackChunks; ++j)
            if (to[j] >= 0) dst[to[j]] = v[j];
    }
    __syncthreads();
    if (threadIdx.x == 0) fence_release_gpu();
}

cudaError_t launch_pack(void *dst, const PackArgs &a, int max_ctas, cudaStream_t stream) {
    const int64_t total = a.first16[a.count];
    const int64_t per_cta = static_cast<int64_t>(kPackThreads) * kPackChunks;
    int64_t ctas = (total + per_cta - 1) / per_cta;
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(kPackThreads, 1, 1);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, hsp_pack_kernel, static_cast<uint4 *>(dst), a);
}

}  // namespace hsp
