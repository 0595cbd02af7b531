// scatter.cuh -- the split-output epilogue shared by both kernels.
//
// TensorRT-LLM PR #20636, Description: one GEMM over the row-concatenated weight,
// its halves returned as dense [M, N_i] outputs.  Row n of a launch belongs to split
// i with off[i] <= n < off[i] + rows[i]; its value for token t goes to
// out[i][t * rows[i] + (n - off[i])], rounded once to the output type.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "stream_args.h"

namespace hsp {

// Where one output row lives: its element for token t is at base + t * stride.
struct OutRow {
    char *base;
    int64_t stride_bytes;
};

// The split that row n of the launch belongs to: the number of later splits whose
// first row is at or below n.  Every table entry is read at a constant index (no
// dynamic indexing into the kernel parameters, no loop-carried dependence).
__device__ __forceinline__ int split_of(const SplitTable &s, int n) {
    int i = 0;
#pragma unroll
    for (int j = 1; j < kMaxSplits; ++j) i += (j < s.count && n >= s.off[j]) ? 1 : 0;
    return i;
}

template <bool BF16_OUT>
__device__ __forceinline__ OutRow out_row(const SplitTable &s, int n) {
    const int i = split_of(s, n);
    constexpr int esz = BF16_OUT ? 2 : 4;
    OutRow o;
    o.base = static_cast<char *>(s.out[i]) + static_cast<int64_t>(n - s.off[i]) * esz;
    o.stride_bytes = static_cast<int64_t>(s.rows[i]) * esz;
    return o;
}

template <bool BF16_OUT>
__device__ __forceinline__ void store_tok(const OutRow &o, int tok, float v) {
    char *p = o.base + static_cast<int64_t>(tok) * o.stride_bytes;
    if constexpr (BF16_OUT)
        *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
    else
        *reinterpret_cast<float *>(p) = v;
}

}  // namespace hsp
