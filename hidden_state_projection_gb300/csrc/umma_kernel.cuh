// umma_kernel.cuh -- the tensor-memory (tcgen05) projection kernel for 9 <= M <= 64.
//
// Same operation and output scatter as the streaming kernel (TensorRT-LLM PR #20636,
// Description), for the token counts where the products no longer fit the legacy
// mma.sync issue rate.  One CTA of four warps owns a tile of 128 (or 64) weight rows
// and one K slice; its S K slices form a cluster.
//
//   * with the l2_prefetch option, warps 2-3 first bulk-prefetch the CTA's weight
//     segments (one contiguous run per row) into L2 (measured slower on GB300: off by
//     default);
//   * warp 0 lane 0 issues tensor copies (128-byte swizzle) of the weight box
//     [tile rows x 128 bytes], L2 evict-first, and the token box [16/32/64 tokens x
//     128 bytes] of each ring stage: one k-block per stage (2-D boxes), or two (3-D
//     boxes [2][rows][128 bytes], 256 contiguous bytes of every weight row per copy);
//     the weight boxes of the first two stages go out before griddepcontrol.wait,
//     token boxes after it (the GLM fused-A order of TensorRT-LLM PR #20502,
//     glmFusedAGemm commit message), then the rest of the first ring;
//   * warp 1 lane 0 issues four tcgen05.mma (M = the tile's weight rows, N = the token tile,
//     K = 16 bf16 or 8 tf32 each) per k-block, k-blocks in order, into one TMEM
//     accumulator and commits each stage back to the ring; a final commit marks the
//     accumulator ready;
//   * all four warps read the accumulator (warp w reads TMEM lanes 32w..32w+31: one
//     weight row per thread, or per lane < 16 for a 64-row tile), then either store
//     (S = 1) or stage the partials per
//     owner CTA and bulk-copy each owner's block into its receive buffer (a copy
//     between cluster shared memories, counted on the owner's mbarrier); the owner
//     adds the S slices in slice order and stores.  The sum of every
//     output is the tensor-core accumulation over K in order, then slices in order:
//     a function of (K, dtype, M bucket) only, never of the row's place in a tile or
//     of the tile's height (64- and 128-row tiles give the same bits, tested).
//   * the trigger follows a release fence in every storing thread (TensorRT-LLM PR
//     #20636, Description).
//
// Rows past the launch, tokens past M and k past K are zero-filled by the tensor
// copies.  Every barrier wait is bounded; on expiry the error word is set, work
// stops, the accumulator is still committed (so no MMA is in flight at exit), copies
// in flight are awaited (bounded) and TMEM is freed on every path.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "prefetch.cuh"
#include "ptx.cuh"
#include "scatter.cuh"
#include "stream_args.h"

namespace hsp {

constexpr int kUmmaThreads = 128;
// Stages whose weight box is requested before the grid-dependency wait (one or two
// k-blocks each); the rest of the first ring follows the first token boxes after the wait
// (measured on GB300 with one-k-block stages, graphs of back-to-back calls: the whole ring
// at entry 10.22 / 10.31 / 11.38 us at qk_indexer M = 16 / 32 / 64, two stages 9.84 /
// 10.09 / 11.22; wq_a++wkv M = 16 8.22 -> 7.90).  With two-k-block stages the ring is two
// stages, so the whole ring goes out before the wait (one stage instead: qk_indexer M = 16
// / 32 / 64 9.36 / 9.67 / 10.38 -> 9.50 / 9.79 / 10.47 us).
constexpr int kUmmaPreWaitStages = 2;

template <int NT>
struct UmmaCfg {
    static_assert(NT == 16 || NT == 32 || NT == 64, "token tile");
    static constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
};

__device__ __forceinline__ bool umma_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7u) == 7u && ((*abort_flag != 0) || (global_timer_ns() - t0 > limit_ns))) return false;
    }
}

template <int COMPUTE, int NT>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    hsp_umma_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                    const __grid_constant__ UmmaArgs a) {
    using C = UmmaCfg<NT>;
    constexpr int kBoxK = (COMPUTE == kMmaBf16) ? 64 : 32;  // elements per 128-byte k-block
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t ring = smem_u32(smem);
    constexpr int kPitch = NT + 4;  // row pitch (floats) of the reduction buffers
    // A stage is the weight box [tile rows][128 bytes] followed by the token box, so the
    // tile height (64 or 128 weight rows, the MMA's M) is what the token box leaves.
    const uint32_t w_box = a.stage_bytes - a.x_box_bytes;
    const int G = a.kb_per_stage == 2 ? 2 : 1;  // k-blocks per stage
    const int TR = static_cast<int>((w_box / G) >> 7);
    const uint32_t x_kb = a.x_box_bytes / G;    // one k-block of the token box
    const uint32_t red_bytes = static_cast<uint32_t>(TR) * kPitch * 4u;  // one partial per row of the tile
    const uint32_t ring_bytes = a.ring_stages * a.stage_bytes;
    float *recv = reinterpret_cast<float *>(smem + ring_bytes);  // K-slice partials of my rows (S > 1)
    const uint32_t recv_bytes = a.slices > 1 ? red_bytes : 0u;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + ring_bytes + recv_bytes);
    uint64_t *empty = full + a.ring_stages;
    uint64_t *accf = empty + a.ring_stages;
    uint64_t *recv_bar = accf + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(recv_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *issued = const_cast<int *>(abort_flag) + 1;  // k-blocks whose copies were issued
    float *staging = reinterpret_cast<float *>(smem);  // my partials, one block per owner (aliases the ring)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * TR;
    const int rows_here = min(TR, a.n_rows - row0);
    const int slice = blockIdx.y;
    const int kb0 = slice * a.kb_per_slice;
    const int nkb = max(0, min(a.kb_total, kb0 + a.kb_per_slice) - kb0);
    // Weights are read once per call: evict first, so that the tokens and outputs the
    // neighbouring kernels share stay in L2 (measured on GB300 at qk_indexer M = 64:
    // 11.98 -> 11.23 us per call; the first token boxes otherwise came from DRAM).
    const uint64_t w_policy = l2_policy_evict_first();
    // Stages of this slice (with two k-blocks per stage the planner makes every slice's
    // k-block count even, so no stage reaches past its slice).
    const int nst = (nkb + G - 1) / G;
    auto load_w = [&](int i, uint32_t dst, uint32_t fb) {
        if (G == 1) tma_load_2d_hint(dst, &tmap_w, (kb0 + i) * kBoxK, row0, fb, w_policy);
        else tma_load_3d_hint(dst, &tmap_w, 0, row0, kb0 + 2 * i, fb, w_policy);
    };
    auto load_x = [&](int i, uint32_t dst, uint32_t fb) {
        if (G == 1) tma_load_2d(dst, &tmap_x, (kb0 + i) * kBoxK, 0, fb);
        else tma_load_3d(dst, &tmap_x, 0, 0, kb0 + 2 * i, fb);
    };

    if (tid == 0) {
        for (int s = 0; s < a.ring_stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(recv_bar), 1);
        // every slice's block of my rows arrives on recv_bar: expect all of them now
        if (a.slices > 1) mbar_arrive_expect_tx(smem_u32(recv_bar), red_bytes);
        *abort_flag = 0;
        *issued = 0;
        mbar_fence_init();
        // The producer's first two weight boxes (stages) go out before the CTA barrier and
        // the TMEM allocation: they depend on nothing but the barriers initialised above.
        tma_prefetch_map(&tmap_w);
        tma_prefetch_map(&tmap_x);
        for (int i = 0; i < min(min(nst, a.ring_stages), kUmmaPreWaitStages); ++i) {
            if (i == a.skip_stage) continue;
            const uint32_t fb = smem_u32(&full[i]);
            mbar_expect_tx(fb, w_box);
            load_w(i, ring + i * a.stage_bytes, fb);
        }
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_d = *tmem_slot;
    if (a.trigger_early) griddep_launch_dependents();  // option trigger_early (the tinygemm2 order)
    // First half of a cluster barrier: the peers' receive barriers are initialised
    // before anyone pushes into them (the wait comes after the main loop).  The
    // initialising thread's fence.mbarrier_init.release.cluster, before the CTA
    // barrier, is the release; the arrival itself is relaxed, so that the copy
    // producer and the MMA issuer start without waiting on it.
    if (a.slices > 1) cluster_arrive_relaxed();

    if (warp >= 2 && a.prefetch_l2 && nkb > 0) {
        // One contiguous run per weight row: this slice's k-blocks of that row.
        const int64_t b0 = static_cast<int64_t>(kb0) * 128;
        const int64_t b1 = min(static_cast<int64_t>(kb0 + nkb) * 128, a.row_bytes);
        const uint32_t nbytes = static_cast<uint32_t>(b1 - b0);
        for (int r = (warp - 2) * 32 + lane; r < rows_here; r += 64)
            bulk_prefetch_l2(a.w + (row0 + r) * a.row_bytes + b0, nbytes);
    }

    // Weights of later kernels named by the caller: into L2, before the grid dependency.
    if (warp == 3 && a.prefetch.count > 0)
        prefetch_ranges_l2(a.prefetch, blockIdx.y * gridDim.x + blockIdx.x, gridDim.x * gridDim.y, lane);

    if (warp == 0 && lane == 0) {
        // ---------------- copy producer (its first weight boxes are already out) ----------------
        const int npre = min(nst, a.ring_stages);
        griddep_wait();
        for (int i = 0; i < npre; ++i) {
            if (i == a.skip_stage) continue;
            const uint32_t fb = smem_u32(&full[i]);
            if (i >= kUmmaPreWaitStages) {  // the rest of the first ring, after the first token boxes
                mbar_expect_tx(fb, w_box);
                load_w(i, ring + i * a.stage_bytes, fb);
            }
            mbar_arrive_expect_tx(fb, a.x_box_bytes);
            load_x(i, ring + i * a.stage_bytes + w_box, fb);
            *issued = i + 1;
        }
        for (int i = npre; i < nst; ++i) {
            const int slot = i % a.ring_stages;
            const uint32_t par = static_cast<uint32_t>((i / a.ring_stages) - 1) & 1u;
            if (!umma_wait(smem_u32(&empty[slot]), par, a.wait_limit_ns, abort_flag)) {
                atomicCAS(a.err_word, 0, kDeviceErrTimeout);
                *abort_flag = 1;
                break;
            }
            if (i == a.skip_stage) continue;
            const uint32_t fb = smem_u32(&full[slot]);
            mbar_arrive_expect_tx(fb, a.stage_bytes);
            load_w(i, ring + slot * a.stage_bytes, fb);
            load_x(i, ring + slot * a.stage_bytes + w_box, fb);
            *issued = i + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t kFmt = (COMPUTE == kMmaBf16) ? 1u : 2u;  // bf16 (kind::f16) / tf32 (kind::tf32)
        const uint32_t idesc = (1u << 4)                       // D: f32
                               | (kFmt << 7) | (kFmt << 10)    // A, B element type
                               | (static_cast<uint32_t>(NT >> 3) << 17)  // N
                               | (static_cast<uint32_t>(TR >> 4) << 24);  // M: the tile's weight rows
        for (int i = 0; i < nst; ++i) {
            const int slot = i % a.ring_stages;
            const uint32_t par = static_cast<uint32_t>(i / a.ring_stages) & 1u;
            if (!umma_wait(smem_u32(&full[slot]), par, a.wait_limit_ns, abort_flag)) {
                atomicCAS(a.err_word, 0, kDeviceErrTimeout);
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            // k-block g of the stage: the weight slab [TR][128 bytes] at g * TR * 128, the
            // token slab at w_box + g * x_kb (both 1024-byte aligned)
            for (int g = 0; g < G; ++g) {
                const uint32_t wa = ring + slot * a.stage_bytes + static_cast<uint32_t>(g * TR * 128);
                const uint32_t xa = ring + slot * a.stage_bytes + w_box + g * x_kb;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t ad = umma_desc_sw128(wa + k * 32);
                    const uint64_t bd = umma_desc_sw128(xa + k * 32);
                    if constexpr (COMPUTE == kMmaBf16)
                        umma_f16(tmem_d, ad, bd, idesc, (i | g | k) != 0 ? 1u : 0u);
                    else
                        umma_tf32(tmem_d, ad, bd, idesc, (i | g | k) != 0 ? 1u : 0u);
                }
            }
            umma_commit(smem_u32(&empty[slot]));
        }
        // Always committed, so that no MMA is in flight when the accumulator is read
        // or the tensor memory freed (also after a timeout).
        umma_commit(smem_u32(accf));
    }
    __syncwarp();

    // ---------------- epilogue ----------------
    // The MMA issuer alone polls for the accumulator; every other thread waits at the
    // CTA barrier, which costs no issue slots.  (With all 128 threads polling the
    // barrier through the main loop, the producer's and the MMA issuer's barrier and
    // tcgen05 instructions queued behind theirs: per-k-block stamps on GB300 showed
    // about 0.35 us per k-block whatever its size.)
    if (warp == 1 && lane == 0) {
        if (!umma_wait(smem_u32(accf), 0u, a.wait_limit_ns, abort_flag)) {
            atomicCAS(a.err_word, 0, kDeviceErrTimeout);
            *abort_flag = 1;
        }
    }
    __syncthreads();
    tc_fence_after_sync();
    const bool aborted = (*abort_flag != 0);
    const bool have_acc = !aborted && nkb > 0;  // an empty K slice contributes zeros
    if (*abort_flag != 0 && tid == 0) {
        // copies still in flight land before the shared memory is reused or freed
        const int n_iss = *issued;
        for (int i = max(0, n_iss - a.ring_stages); i < n_iss; ++i) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&full[i % a.ring_stages]), static_cast<uint32_t>(i / a.ring_stages) & 1u) &&
                   global_timer_ns() - t0 < a.wait_limit_ns / 16 + 1) {
            }
        }
    }
    __syncthreads();

    // Warp w reads TMEM lanes 32w .. 32w + 31.  An M = 128 accumulator keeps row i in lane
    // i; an M = 64 one keeps rows 16w .. 16w + 15 in lanes 32w .. 32w + 15 (the other
    // sixteen lanes of each quarter hold no rows).  Thread (w, l) owns row w * TR / 4 + l.
    const int rpw = TR >> 2;
    const bool has_row = lane < rpw;
    const int r = warp * rpw + lane;
    float v[NT];
    if (have_acc) {
#pragma unroll
        for (int c = 0; c < NT; c += 16) {
            float t[16];
            tmem_ld16(tmem_d + (static_cast<uint32_t>(warp * 32) << 16) + c, t);
#pragma unroll
            for (int q = 0; q < 16; ++q) v[c + q] = t[q];
        }
        tmem_wait_ld();
    } else {
#pragma unroll
        for (int c = 0; c < NT; ++c) v[c] = 0.f;
    }
    tc_fence_before_sync();

    griddep_wait();  // outputs may still be read by the previous kernel on the stream
    bool stored = false;
    constexpr bool kBf16Out = (COMPUTE == kMmaBf16);
    if (a.slices == 1) {
        if (!aborted && has_row && r < rows_here) {
            const OutRow o = out_row<kBf16Out>(a.splits, row0 + r);
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (t < a.M) store_tok<kBf16Out>(o, t, v[t]);
            stored = true;
        }
    } else {
        // Push model.  Each thread puts its row's partial into a local staging buffer
        // laid out as one contiguous block per owner CTA, [owner][row][token] with a
        // row pitch of NT + 4 floats.  One thread then bulk-copies block q into the
        // dedicated receive buffer of CTA q, completing on that CTA's receive barrier,
        // which has expected all S blocks since the kernel started.  Each owner waits
        // for its barrier and adds the S slices of its rows in slice order.
        const int per = TR / a.slices;
        const uint32_t block_bytes = static_cast<uint32_t>(per * kPitch * 4);
        if (has_row) {
            const int q = r / per, rr = r - q * per;
            float *dst = staging + q * per * kPitch + rr * kPitch;
#pragma unroll
            for (int c = 0; c < NT; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
        }
        fence_proxy_async_smem();   // staging writes -> the bulk copies that read them
        __syncthreads();
        cluster_wait();             // every peer's receive barrier is initialised
        if (tid == 0) {
            const uint32_t recv_local = smem_u32(recv), bar_local = smem_u32(recv_bar), src = smem_u32(staging);
            for (int q = 0; q < a.slices; ++q)
                bulk_s2s_cluster(cluster_map_shared(recv_local + slice * block_bytes, static_cast<uint32_t>(q)),
                                 src + q * block_bytes, block_bytes, cluster_map_shared(bar_local, static_cast<uint32_t>(q)));
        }
        // One thread polls for the peers' blocks, bounded by time only (not cut short by
        // an earlier timeout: no CTA may leave while copies into it are in flight); the
        // others wait at the CTA barrier.
        if (tid == 0) {
            const uint64_t t0 = global_timer_ns();
            bool done = false;
            for (uint32_t it = 0;; ++it) {
                if ((done = mbar_try_wait(smem_u32(recv_bar), 0u))) break;
                if ((it & 7u) == 7u && global_timer_ns() - t0 > a.wait_limit_ns) break;
            }
            if (!done) {
                atomicCAS(a.err_word, 0, kDeviceErrTimeout);
                *abort_flag = 1;
            }
        }
        __syncthreads();
        const bool got = *abort_flag == 0;
        // First half of the closing cluster barrier: my receive buffer is complete, so
        // every copy out of a peer's staging buffer into mine has landed.  The wait
        // comes last, after the trigger: no CTA leaves while a bulk copy may still read
        // its staging buffer, yet the peers' sums, stores and fences overlap it.  The
        // barrier only keeps the CTAs resident (the data moved by copies that complete on
        // mbarriers), so the arrival carries no release ordering: a release arrival here
        // waited 0.3-1.9 us (0.7 us on average) at qk_indexer M = 64 on GB300.
        cluster_arrive_relaxed();
        if (!aborted && got) {
            constexpr int kT4 = NT / 4;
            // consecutive threads take consecutive rows of the same four tokens
            for (int e = tid; e < per * kT4; e += kUmmaThreads) {
                const int t4 = (e / per) * 4, rr = e - (e / per) * per;
                const int row = slice * per + rr;
                if (row >= rows_here || t4 >= a.M) continue;
                float4 part[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (q < a.slices) part[q] = *reinterpret_cast<const float4 *>(recv + (q * per + rr) * kPitch + t4);
                float4 acc = part[0];
#pragma unroll
                for (int q = 1; q < 16; ++q)
                    if (q < a.slices) {
                        acc.x += part[q].x;
                        acc.y += part[q].y;
                        acc.z += part[q].z;
                        acc.w += part[q].w;
                    }
                const float o4[4] = {acc.x, acc.y, acc.z, acc.w};
                const OutRow o = out_row<kBf16Out>(a.splits, row0 + row);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (t4 + j < a.M) store_tok<kBf16Out>(o, t4 + j, o4[j]);
                stored = true;
            }
        }
    }
    if (stored) fence_release_gpu();
    tc_fence_before_sync();
    __syncthreads();
    // Every output store of this CTA is performed: trigger the dependent launch.
    griddep_launch_dependents();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_d, C::kTmemCols);
    }
    if (a.slices > 1) cluster_wait();
}

}  // namespace hsp
