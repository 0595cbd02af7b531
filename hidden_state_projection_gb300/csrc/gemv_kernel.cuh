// gemv_kernel.cuh -- the fp32 register GEMV kernel (PROJ_FP32, 1 <= M <= 64).
//
// Same operation and split epilogue as the other kernels (TensorRT-LLM PR #20636,
// Description), for the fp32 projections the pages run at decode size: the indexer's
// wk ++ weights_proj (TensorRT-LLM PR #12055, Description: 128 + 64 rows of 7168) and
// the GLM router (TensorRT-LLM PR #20502, glmRouterGemm commit message: 256 experts x
// 6144, one CTA per expert, an FP32 GEMV).  Their few hundred rows leave every SM only
// 2 rows to stream; the streaming kernel split K over clusters of 4 CTAs for them and
// spent most of a call in its cluster set-up and reduction.  Here one CTA of sixteen
// warps owns R = ceil(N / SMs) rows and all of K, with no cluster:
//
//   * K is cut into 16-byte chunks of 4 floats; thread t takes chunks t, t + 512, ...
//     of every row, up to kGemvSteps chunks per row (K <= 8192);
//   * rows go in blocks of kGemvRows; a block's chunks are loaded straight into
//     registers (read-only path, no L1 allocation, L2 evict-first), two blocks in
//     flight: the first two before griddepcontrol.wait, at kernel entry;
//   * the tokens X[M, K] arrive after the grid-dependency wait as eight 1-D bulk copies
//     into shared memory, issued from a different piece in each CTA (contiguous rows;
//     thread t reads its own chunks, conflict free);
//   * each thread keeps one fp32 FMA chain per (row, token): its chunks in increasing
//     order, the 4 floats of a chunk in k order; the 32 lanes of a warp are then added
//     by a fixed transposing reduction and the 16 warps in warp order.  The order
//     depends on K only, so fused and per-projection launches, repeats and graph
//     replays give identical bits; the chains are at most 16 terms long, well inside
//     the fp32 tolerance;
//   * every storing thread fences, the CTA synchronises, and only then is the dependent
//     launch triggered (the trigger follows the stores).
//
// More tokens than shared memory holds (M * K * 4 > 192 KB, or M > 8) are cut into
// grid.y groups of ceil(M / grid.y) tokens (the last one ragged); the CTAs of one row
// slab and different groups read the same weight rows, the first from HBM and the others
// mostly from L2, so those loads keep the normal L2 priority.  A token's sums do not
// depend on its group: every output is one CTA's fixed-order sum over all of K.
//
// The one barrier wait (the token copy) is bounded; on expiry the kernel records
// PROJ_ERR_TIMEOUT, skips its stores, waits (bounded) for its copy and returns.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "prefetch.cuh"
#include "ptx.cuh"
#include "scatter.cuh"
#include "stream_args.h"

namespace hsp {

constexpr int kGemvWarps = 16;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvRows = 2;   // rows per block (two blocks in flight)
constexpr int kGemvSteps = 4;  // 16-byte chunks per thread and row: K <= 4 * 4 * 512 = 8192

__device__ __forceinline__ uint4 ldg_stream16(const char *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// L2 policy for weights that other CTAs (the other token groups) read again soon.
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__global__ void __launch_bounds__(kGemvThreads, 1) hsp_gemv_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ __align__(16) float xs[];     // [tokens of the group][K]
    __shared__ float part[kGemvWarps][kGemvRows][8];  // warp sums of a block [warp][row][token]
    __shared__ __align__(8) uint64_t xfull;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // token group: grid.y groups of ceil(M / grid.y) tokens, the last one ragged
    const int group = static_cast<int>((a.M + gridDim.y - 1) / gridDim.y);
    const int tok0 = static_cast<int>(blockIdx.y) * group;
    const int Mh = min(group, a.M - tok0);
    if (Mh < 1) {  // an empty group (the planner never makes one): nothing to do
        griddep_launch_dependents();
        return;
    }
    const int row0 = blockIdx.x * a.rows_per_cta;
    const int rows_here = min(a.rows_per_cta, a.n_rows - row0);
    const int nblk = (rows_here + kGemvRows - 1) / kGemvRows;
    const int chunks = static_cast<int>(a.row_bytes >> 4);
    const int K = chunks * 4;
    // with one group every weight is read once; with several the other groups' CTAs read
    // the same rows at about the same time, from L2
    const uint64_t policy = gridDim.y > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();

    uint4 buf0[kGemvRows][kGemvSteps], buf1[kGemvRows][kGemvSteps];
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    auto load_block = [&](uint4 (&buf)[kGemvRows][kGemvSteps], int b) {
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r) {
            const int row = b * kGemvRows + r;
            const char *p = a.w + static_cast<int64_t>(row0 + min(row, rows_here - 1)) * a.row_bytes;
#pragma unroll
            for (int s = 0; s < kGemvSteps; ++s) {
                const int c = tid + s * kGemvThreads;
                buf[r][s] = (row < rows_here && c < chunks) ? ldg_stream16(p + static_cast<int64_t>(c) * 16, policy) : zero;
            }
        }
    };
    load_block(buf0, 0);
    if (nblk > 1) load_block(buf1, 1);

    const uint32_t bar = smem_u32(&xfull);
    if (tid == 0) {
        mbar_init(bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (a.trigger_early) griddep_launch_dependents();  // option trigger_early (the tinygemm2 order)
    // The activations are written by the previous kernel on the stream.
    griddep_wait();
    const bool x_issued = a.skip_stage != 0;  // test hook: stage 0 of this kernel is its token copy
    if (tid == 0 && x_issued) {
        const uint32_t bytes = static_cast<uint32_t>(Mh) * static_cast<uint32_t>(a.row_bytes);
        mbar_arrive_expect_tx(bar, bytes);
        // Every CTA reads the same token bytes at about the same time: eight pieces, each
        // CTA starting at a different one, spread the requests over the L2 slices
        // (measured on GB300: indexer M = 4 5.32 -> 5.15 us, router M = 4 5.01 -> 4.90).
        constexpr uint32_t kPieces = 8;
        const uint32_t piece = (bytes + kPieces * 16 - 1) / (kPieces * 16) * 16;
        for (uint32_t q = 0; q < kPieces; ++q) {
            const uint32_t off = ((q + blockIdx.x) % kPieces) * piece;
            if (off >= bytes) continue;
            bulk_copy_g2s(smem_u32(xs) + off, a.x + static_cast<int64_t>(tok0) * a.row_bytes + off,
                          min(piece, bytes - off), bar);
        }
    }
    if (warp == kGemvWarps - 1 && a.prefetch.count > 0)
        prefetch_ranges_l2(a.prefetch, blockIdx.x, gridDim.x, lane);

    // bounded wait for the tokens (warp-wide)
    bool ok;
    {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 0;; ++it) {
            const bool done = mbar_try_wait(bar, 0u);
            if (__all_sync(0xffffffffu, done)) {
                ok = true;
                break;
            }
            int give_up = 0;
            if ((it & 7u) == 7u) give_up = (global_timer_ns() - t0 > a.wait_limit_ns) ? 1 : 0;
            if (__shfl_sync(0xffffffffu, give_up, 0)) {
                ok = false;
                break;
            }
        }
    }
    if (!ok && lane == 0) {
        atomicCAS(a.err_word, 0, kDeviceErrTimeout);
        abort_flag = 1;
    }

    bool stored = false;
    // Products, reductions and stores of block b from buf; then buf takes block b + 2.
    auto do_block = [&](uint4 (&buf)[kGemvRows][kGemvSteps], int b) {
        float acc[kGemvRows][8];
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
            for (int t = 0; t < 8; ++t) acc[r][t] = 0.f;
        if (ok) {
#pragma unroll
            for (int s = 0; s < kGemvSteps; ++s) {
                const int c = tid + s * kGemvThreads;
                if (c < chunks) {
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        if (t < Mh) {
                            const float4 xv = *reinterpret_cast<const float4 *>(xs + t * K + c * 4);
#pragma unroll
                            for (int r = 0; r < kGemvRows; ++r) {
                                const uint4 w = buf[r][s];
                                float v = acc[r][t];
                                v = fmaf(__uint_as_float(w.x), xv.x, v);
                                v = fmaf(__uint_as_float(w.y), xv.y, v);
                                v = fmaf(__uint_as_float(w.z), xv.z, v);
                                v = fmaf(__uint_as_float(w.w), xv.w, v);
                                acc[r][t] = v;
                            }
                        }
                    }
                }
            }
        }
        if (b + 2 < nblk) load_block(buf, b + 2);
        // Lanes of a warp by a fixed transposing reduction over all 16 (row, token) slots
        // (token slots past the group's tokens hold zeros): at offsets 16, 8, 4 and 2 each
        // lane keeps half of its values and adds the partner's copy of that half, so lane
        // l ends with slot (l >> 1) & 15 summed over 16 lanes; offset 1 adds the last pair.
        // 16 shuffles per lane for any token count (a butterfly per slot took 5 per slot:
        // 40 at four tokens).  Then the warps in order.
        static_assert(kGemvRows * 8 == 16, "the transposing reduction covers 16 slots");
        float v[16];
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
            for (int t = 0; t < 8; ++t) v[r * 8 + t] = acc[r][t];
        int n = 16;
#pragma unroll
        for (int o = 16; o >= 2; o >>= 1) {
            const bool upper = (lane & o) != 0;  // keep the upper half, send the lower
            n >>= 1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < n) {
                    const float keep = upper ? v[i + n] : v[i];
                    const float send = upper ? v[i] : v[i + n];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
        }
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        {
            const int slot = (lane >> 1) & 15, r = slot >> 3, t = slot & 7;
            if ((lane & 1) == 0 && t < Mh) part[warp][r][t] = v[0];
        }
        __syncthreads();
        if (abort_flag == 0 && tid < kGemvRows * Mh) {
            const int r = tid / Mh, t = tid - r * Mh;
            const int row = b * kGemvRows + r;
            if (row < rows_here) {
                float v = part[0][r][t];
#pragma unroll
                for (int w = 1; w < kGemvWarps; ++w) v += part[w][r][t];
                const int n = row0 + row;
                const int i = split_of(a.splits, n);
                float *o = static_cast<float *>(a.splits.out[i]);
                o[static_cast<int64_t>(tok0 + t) * a.splits.rows[i] + (n - a.splits.off[i])] = v;
                stored = true;
            }
        }
        __syncthreads();  // part is reused by the next block
    };
    for (int b = 0; b < nblk; b += 2) {
        do_block(buf0, b);
        if (b + 1 < nblk) do_block(buf1, b + 1);
    }

    if (abort_flag != 0 && tid == 0 && x_issued) {
        // the token copy may still be in flight: let it land before the CTA leaves
        const uint64_t t0 = global_timer_ns(), limit = a.wait_limit_ns / 16 + 1;
        while (!mbar_try_wait(bar, 0u) && global_timer_ns() - t0 < limit) {
        }
    }
    // Trigger the dependent launch only after every output store of this CTA is
    // performed: each storing thread fences, then the CTA synchronises.
    if (stored) fence_release_gpu();
    __syncthreads();
    griddep_launch_dependents();
}

}  // namespace hsp
