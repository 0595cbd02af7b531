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
// The finishing CTA's reads of the workspace are issued together rather than one
// dependent load per loop trip: the per-CTA sums of squares are first copied into
// `scratch` (shared memory, scratch_floats floats, free at this point) by all threads
// and then added in CTA order from there, and each thread loads kNormBatch parked
// values and gammas before it scales and stores them.  (A dependent load per trip put
// one L2 round trip per CTA of the split, ~100 at wq_a, on the critical path.)
//
// The workspace's first 256 bytes hold the arrival counters [kMaxSplits] (arrivals in
// the low 16 bits, arrivals of CTAs that gave up a wait in the high 16): zero before
// the first call, and every call, one that timed out included, leaves them at zero.
//
// Returns true when this thread stored an output (the caller fences before its
// trigger).  A flag returned by value, not through a reference: a reference would
// put the caller's flag in local memory, and its local store would then sit in
// front of the caller's release fence.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

constexpr int kNormBatch = 8;  // scalar path: values per thread in flight
constexpr int kNormItems = 4;  // vector path: 8-column items per thread in flight

template <bool BF16_OUT, int kSlots, int kXRows>
__device__ __noinline__ bool norm_epilogue(const StreamArgs &a, float *red, int *finish, int row0, int rows_here,
                                           bool aborted, int tid, float *scratch, int scratch_floats) {
    // Every argument this function reads is copied into registers first: `a` is the
    // kernel's parameter block seen through a generic pointer, and a store through
    // another generic pointer (the workspace, the outputs) would otherwise make the
    // compiler read it again after every store.
    bool stored = false;
    __syncthreads();
    const NormArgs &nm = a.norm;
    const int bx = blockIdx.x;
    const int M = a.M, nsplit = a.splits.count;
    const int nthreads = static_cast<int>(blockDim.x);
    float *const __restrict__ partial = nm.partial;
    if (!aborted) {
        for (int e = tid; e < nsplit * M; e += nthreads) {
            const int i = e / M, tok = e - i * M;
            const int cols = nm.cols[i], first = nm.cta_first[i], count = nm.cta_count[i];
            if (cols == 0 || bx < first || bx >= first + count) continue;
            const int off = a.splits.off[i];
            const int lo = max(off - row0, 0);
            const int hi = min(off + cols - row0, rows_here);
            float ss = 0.f;
            for (int slot = lo; slot < hi; ++slot) {
                const float v = red[slot * kXRows + tok];
                ss = fmaf(v, v, ss);
            }
            partial[nm.part_off[i] + (bx - first) * M + tok] = ss;
        }
    }
    // The arrival below is an acquire-release atomic after a CTA barrier: its release
    // half is cumulative over the barrier, so it publishes every thread's parked values
    // and sums; for the last arrival its acquire half, followed by the next barrier,
    // makes every other CTA's values visible to all threads of this CTA.
    __syncthreads();
    if (tid < nsplit) {
        // Every CTA of the split arrives, also one that gave up a wait: it adds 1 + 2^16
        // instead of 1, so the last arrival sees in the same atomic whether any CTA of
        // the split gave up, and the counter always returns to zero for the next call.
        const int i = tid;
        const int cols = nm.cols[i], first = nm.cta_first[i], count = nm.cta_count[i];
        int last = 0;
        if (cols > 0 && bx >= first && bx < first + count) {
            const unsigned inc = aborted ? 0x10001u : 1u;
            const unsigned old = atom_add_acq_rel_gpu(&nm.counter[i], inc);
            if ((old & 0xffffu) == static_cast<unsigned>(count - 1)) last = ((old + inc) >> 16) != 0u ? 2 : 1;
        }
        finish[i] = last;
    }
    __syncthreads();
    for (int i = 0; i < nsplit; ++i) {
        if (finish[i] == 0) continue;
        if (finish[i] == 2) {  // a CTA of the split gave up: no outputs, counters reset
            if (tid == 0) nm.counter[i] = 0u;
            continue;
        }
        const int c = nm.cols[i];
        const int count = nm.cta_count[i];
        const int np = count * M;
        const float eps = nm.eps;
        const float *const __restrict__ parts = partial + nm.part_off[i];
        const float *const __restrict__ vals = nm.vals + nm.vals_off[i];
        const void *const gamma = nm.gamma[i];
        char *const __restrict__ out = static_cast<char *>(a.splits.out[i]);
        const int64_t stride = a.splits.rows[i];
        const bool staged = np + M <= scratch_floats;  // [count][M] sums, then [M] scales
        float *scale = staged ? scratch + np : red;    // red: this CTA's own sums are in the workspace by now
        const int n = c * M;
        // Eight columns per item when every address allows 16-byte output stores and
        // 32-byte value loads (normalized widths of the pages' splits are multiples of 64).
        const bool vec = BF16_OUT && (c % 8) == 0 && (stride % 8) == 0 && (nm.vals_off[i] % 8) == 0 &&
                         ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(gamma)) & 15u) == 0;
        const int c8 = c >> 3, items = vec ? c8 * M : 0;
        // This thread's first kNormItems items are requested before the sums of squares
        // are added, so their loads overlap the staging and the sums below.
        float4 va[kNormItems], vb[kNormItems];
        uint4 gv[kNormItems];
        auto load_items = [&](int base) {
#pragma unroll
            for (int j = 0; j < kNormItems; ++j) {
                const int it = base + j * nthreads;
                if (it < items) {
                    const int tok = it / c8, col = (it - tok * c8) * 8;
                    va[j] = __ldcg(reinterpret_cast<const float4 *>(vals + tok * c + col));
                    vb[j] = __ldcg(reinterpret_cast<const float4 *>(vals + tok * c + col + 4));
                    gv[j] = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(gamma) + col);
                }
            }
        };
        // The per-CTA sums of squares head the chain to the scales: their loads go out
        // first, then this thread's first items, which overlap the staging and the sums
        // (items first put ~100 KB of value loads ahead of them).
        constexpr int kPartBatch = 4;
        float pv[kPartBatch];
        if (staged) {
#pragma unroll
            for (int j = 0; j < kPartBatch; ++j) {
                const int e = tid + j * nthreads;
                pv[j] = e < np ? __ldcg(&parts[e]) : 0.f;
            }
        }
        load_items(tid);
        __syncthreads();
        if (staged) {
#pragma unroll
            for (int j = 0; j < kPartBatch; ++j) {
                const int e = tid + j * nthreads;
                if (e < np) scratch[e] = pv[j];
            }
            for (int e = tid + kPartBatch * nthreads; e < np; e += nthreads) scratch[e] = __ldcg(&parts[e]);
            __syncthreads();
        }
        if (staged) {
            // warp w < M adds token w's sums: lane l takes CTAs l, l + 32, ... in order,
            // then the lanes are added by a fixed butterfly
            const int warp = tid >> 5, lane = tid & 31;
            for (int tok = warp; tok < M; tok += nthreads >> 5) {
                float ss = 0.f;
                for (int k = lane; k < count; k += 32) ss += scratch[k * M + tok];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (lane == 0) scale[tok] = 1.0f / sqrtf(ss / static_cast<float>(c) + eps);
            }
        } else if (tid < M) {
            float ss = 0.f;
            for (int k = 0; k < count; ++k) ss += __ldcg(&parts[k * M + tid]);
            scale[tid] = 1.0f / sqrtf(ss / static_cast<float>(c) + eps);
        }
        __syncthreads();
        for (int base = tid; base < items; base += kNormItems * nthreads) {
#pragma unroll
            for (int j = 0; j < kNormItems; ++j) {
                const int it = base + j * nthreads;
                if (it < items) {
                    const int tok = it / c8, col = (it - tok * c8) * 8;
                    const float sc = scale[tok];
                    const float vv[8] = {va[j].x, va[j].y, va[j].z, va[j].w, vb[j].x, vb[j].y, vb[j].z, vb[j].w};
                    const uint32_t gw[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
                    uint32_t ow[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float g0 = __uint_as_float(gw[h] << 16), g1 = __uint_as_float(gw[h] & 0xffff0000u);
                        const __nv_bfloat16 b0 = __float2bfloat16_rn(vv[2 * h] * sc * g0);
                        const __nv_bfloat16 b1 = __float2bfloat16_rn(vv[2 * h + 1] * sc * g1);
                        ow[h] = static_cast<uint32_t>(__bfloat16_as_ushort(b0)) |
                                (static_cast<uint32_t>(__bfloat16_as_ushort(b1)) << 16);
                    }
                    *reinterpret_cast<uint4 *>(out + (static_cast<int64_t>(tok) * stride + col) * 2) =
                        make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    stored = true;
                }
            }
            if (base + kNormItems * nthreads < items) load_items(base + kNormItems * nthreads);
        }
        for (int e0 = vec ? n : tid; e0 < n; e0 += kNormBatch * nthreads) {
            float v[kNormBatch], g[kNormBatch];
#pragma unroll
            for (int j = 0; j < kNormBatch; ++j) {
                const int e = e0 + j * nthreads;
                v[j] = 0.f;
                g[j] = 0.f;
                if (e < n) {
                    const int col = e % c;
                    v[j] = __ldcg(&vals[e]);
                    if constexpr (BF16_OUT) g[j] = __bfloat162float(static_cast<const __nv_bfloat16 *>(gamma)[col]);
                    else g[j] = static_cast<const float *>(gamma)[col];
                }
            }
#pragma unroll
            for (int j = 0; j < kNormBatch; ++j) {
                const int e = e0 + j * nthreads;
                if (e < n) {
                    const int tok = e / c, col = e - tok * c;
                    const float y = v[j] * scale[tok] * g[j];
                    const int64_t idx = static_cast<int64_t>(tok) * stride + col;
                    if constexpr (BF16_OUT) reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(y);
                    else reinterpret_cast<float *>(out)[idx] = y;
                    stored = true;
                }
            }
        }
        __syncthreads();
        if (tid == 0) nm.counter[i] = 0u;  // ready for the next call
    }
    return stored;
}

}  // namespace hsp
