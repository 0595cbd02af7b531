// prefetch.cuh -- L2 prefetch of caller-named tensors (weights of later kernels).
//
// TensorRT-LLM PR #20502 (GLM-5.2 decode target), glmFusedAGemm commit message:
// ahead of its grid-dependency wait, the GLM fused-A kernel has its CTAs share out
// 16 KB L2 bulk prefetches of as many as four caller tensors (the weights the step's
// following kernels will need).  Here chunk c of the concatenated ranges goes to CTA
// (c mod CTAs), lane-parallel inside the calling warp.  The streaming kernel issues
// them after its own weight and token copies (measured: ahead of the token copies
// they delay the first stage), the tensor-memory kernel before its grid wait.
#pragma once

#include <stdint.h>

#include "ptx.cuh"
#include "stream_args.h"

namespace hsp {

__device__ __forceinline__ void prefetch_ranges_l2(const PrefetchList &pf, int cta, int ctas, int lane) {
    int64_t base_chunk = 0;
    for (int i = 0; i < pf.count; ++i) {
        const int64_t chunks = static_cast<int64_t>((pf.bytes[i] + kPrefetchChunk - 1) / kPrefetchChunk);
        // first chunk of range i owned by this CTA, then every ctas-th
        int64_t c = ((cta - base_chunk) % ctas + ctas) % ctas;
        for (c += static_cast<int64_t>(lane) * ctas; c < chunks; c += static_cast<int64_t>(ctas) * 32) {
            const uint64_t off = static_cast<uint64_t>(c) * kPrefetchChunk;
            const uint64_t left = pf.bytes[i] - off;
            bulk_prefetch_l2(pf.ptr[i] + off, static_cast<uint32_t>(left < kPrefetchChunk ? left : kPrefetchChunk));
        }
        base_chunk += chunks;
    }
}

}  // namespace hsp
