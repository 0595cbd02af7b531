// norm_epilogue.cuh -- the RMSNorm epilogue shared by the projection kernels.
//
// The consumers of the q_a / kv_a projections normalise them (TensorRT-LLM PR
// #20636, Description: the q_norm / kv_norm RMSNorms read the wq_a / wkv outputs).
// The mean of squares of a token spans all CTAs holding the normalized columns of a
// split, so each such CTA parks its fp32 values and per-token sums of squares in a
// caller workspace and arrives on the split's counter; the last CTA to arrive adds
// the sums in CTA order, normalizes the split and stores it.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "stream_args.h"

namespace hsp {

// After the combine loop of a single-slice CTA: red[slot * kXRows + tok] holds the
// fp32 sums of this CTA's rows.  For every normalized split this CTA meets, the
// per-token sum of squares over its rows of that split (increasing row order) goes to
// the workspace; the CTA then arrives on the split's counter, and the last CTA to
// arrive finishes the split.  Every order is fixed, so the results do not depend on
// which CTA finishes.
//
// Returns true when this thread stored an output (the caller fences before its
// trigger).  A flag returned by value, not through a reference: a reference would
// put the caller's flag in local memory, and its local store would then sit in
// front of the caller's release fence.
template <bool BF16_OUT, int kSlots, int kXRows>
__device__ __noinline__ bool norm_epilogue(const StreamArgs &a, float *red, int *finish, int row0, int rows_here,
                                           bool aborted, int tid) {
    bool stored = false;
    __syncthreads();
    const NormArgs &nm = a.norm;
    const int bx = blockIdx.x;
    if (!aborted) {
        for (int e = tid; e < a.splits.count * a.M; e += blockDim.x) {
            const int i = e / a.M, tok = e - i * a.M;
            if (nm.cols[i] == 0 || bx < nm.cta_first[i] || bx >= nm.cta_first[i] + nm.cta_count[i]) continue;
            const int lo = max(a.splits.off[i] - row0, 0);
            const int hi = min(a.splits.off[i] + nm.cols[i] - row0, rows_here);
            float ss = 0.f;
            for (int slot = lo; slot < hi; ++slot) {
                const float v = red[slot * kXRows + tok];
                ss = fmaf(v, v, ss);
            }
            nm.partial[nm.part_off[i] + (bx - nm.cta_first[i]) * a.M + tok] = ss;
        }
    }
    __threadfence();  // this CTA's values and sums are visible before it arrives
    __syncthreads();
    if (tid < a.splits.count) {
        const int i = tid;
        int last = 0;
        if (!aborted && nm.cols[i] > 0 && bx >= nm.cta_first[i] && bx < nm.cta_first[i] + nm.cta_count[i])
            last = (atomicAdd(&nm.counter[i], 1u) == static_cast<unsigned>(nm.cta_count[i] - 1)) ? 1 : 0;
        finish[i] = last;
    }
    __syncthreads();
    for (int i = 0; i < a.splits.count; ++i) {
        if (!finish[i]) continue;
        __threadfence();  // every other CTA's values and sums are visible from here on
        const int c = nm.cols[i];
        float *scale = red;  // [M]: this CTA's own sums are in the workspace by now
        __syncthreads();
        if (tid < a.M) {
            float ss = 0.f;
            for (int k = 0; k < nm.cta_count[i]; ++k) ss += __ldcg(&nm.partial[nm.part_off[i] + k * a.M + tid]);
            scale[tid] = 1.0f / sqrtf(ss / static_cast<float>(c) + nm.eps);
        }
        __syncthreads();
        char *out = static_cast<char *>(a.splits.out[i]);
        const int64_t stride = a.splits.rows[i];
        for (int e = tid; e < c * a.M; e += blockDim.x) {
            const int tok = e / c, col = e - tok * c;
            float g;
            if constexpr (BF16_OUT) g = __bfloat162float(static_cast<const __nv_bfloat16 *>(nm.gamma[i])[col]);
            else g = static_cast<const float *>(nm.gamma[i])[col];
            const float v = __ldcg(&nm.vals[nm.vals_off[i] + e]) * scale[tok] * g;
            const int64_t idx = static_cast<int64_t>(tok) * stride + col;
            if constexpr (BF16_OUT) reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
            else reinterpret_cast<float *>(out)[idx] = v;
            stored = true;
        }
        __syncthreads();
        if (tid == 0) nm.counter[i] = 0u;  // ready for the next call
    }
    return stored;
}

}  // namespace hsp
