// stream_kernel.cuh -- the weight-streaming projection kernel.
//
// Computes, for the rows [row0, row0 + R) of one launch's weight map and all M
// tokens,  y[m][n] = sum_k x[m][k] * w[n][k]  with fp32 accumulation, rounds once
// and scatters every row into the output of the projection it belongs to
// (TensorRT-LLM PR #20636, Description: one GEMM over the row-concatenated
// weight, halves returned as dense [M, N_i] outputs).
//
// Structure of one CTA (the design of the pages' GLM fused-A kernel -- weights
// staged by tensor copies before the grid-dependency wait, activations after
// it, warp sums added in warp order and rounded once; TensorRT-LLM PR #20502,
// glmFusedAGemm commit message -- re-drawn for TMA rings and clusters):
//
//   * warp kNCW (the producer) issues 2-D TMA copies of 128-byte-wide boxes of
//     W (R rows) and X (8*MT token rows) into a ring of shared-memory stages;
//     the W boxes of the first ring's worth of stages go out before
//     griddepcontrol.wait, the X boxes only after it;
//   * consumer warp (wr, wk) takes box wk of every stage, for its RT 16-row
//     tiles, and accumulates in registers: mma.sync bf16 / tf32, or fp32 FMA;
//   * the WK warp partials of each output are added in warp order, then (S > 1)
//     the S CTAs of a cluster, each holding one K slice, add their partials in
//     slice order through distributed shared memory;
//   * the sum is rounded once and stored; every storing thread fences, the CTA
//     synchronises, and only then is the dependent launch triggered (the trigger
//     follows the stores, the robust order TensorRT-LLM PR #20636, Description,
//     recommends).
//
// Determinism: the summation order of an output depends only on (K, the element
// type, WK, S) -- never on the row count, the row's position in a tile, the grid
// or the arrival order -- so fused and per-projection launches, repeated runs
// and graph replays give identical bits.
//
// Every wait on a shared-memory barrier is bounded (globaltimer); on expiry the
// kernel records PROJ_ERR_TIMEOUT in the device error word, stops computing,
// skips its stores, waits (bounded) for its own copies still in flight, and
// returns through the same barriers as a normal exit.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"
#include "stream_args.h"

namespace hsp {

template <int COMPUTE, int MT, int RT, int WR, int WK>
struct StreamCfg {
    static constexpr int kCompute = COMPUTE;
    static constexpr int kNCW = WR * WK;                 // consumer warps
    static constexpr int kThreads = (kNCW + 1) * 32;     // + producer warp
    static constexpr int kSlots = WR * RT * 16;          // row slots per CTA
    static constexpr int kXRows = 8 * MT;                // token rows per X box
    static constexpr int kEsz = (COMPUTE == kMmaBf16) ? 2 : 4;
    static constexpr int kBoxK = 128 / kEsz;             // K elements per box
    static_assert(WR * WK == 8, "eight consumer warps");
    static_assert(MT == 1 || MT % 2 == 0, "token tiles: 1 or even");
};

// Byte offset of 16-byte chunk c of row r inside a box written by TMA with
// 128-byte swizzling (box base 1024-byte aligned): chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// Warp-wide bounded wait on one barrier phase.  True when the phase completed;
// false when the limit ran out or another warp already gave up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile int *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        int give_up = 0;
        if ((it & 7u) == 7u) give_up = (*abort_flag != 0) || (global_timer_ns() - t0 > limit_ns);
        if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
}

// Single-thread bounded wait (producer lane).
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                            volatile int *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7u) == 7u && ((*abort_flag != 0) || (global_timer_ns() - t0 > limit_ns)))
            return false;
    }
}

__device__ __forceinline__ void record_timeout(int *err_word, volatile int *abort_flag) {
    atomicCAS(err_word, 0, kDeviceErrTimeout);
    *abort_flag = 1;
}

// ---- inner products on one staged box ------------------------------------

// Tensor-core box: 4 k-steps (k16 for bf16, k8 for tf32) over the warp's row tiles.
template <class C, int RT, int MT>
__device__ __forceinline__ void box_mma(uint32_t wbox, uint32_t xbox, int wr, int lane,
                                        float (&acc)[RT][MT][4]) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t b[MT][2];
        if constexpr (MT == 1) {
            const int tok = lane & 7, c = 2 * ks + ((lane >> 3) & 1);
            ldsm_x2(xbox + swz(tok, c), b[0][0], b[0][1]);
        } else {
#pragma unroll
            for (int j = 0; j < MT; j += 2) {
                const int tok = (j + (lane >> 4)) * 8 + (lane & 7);
                const int c = 2 * ks + ((lane >> 3) & 1);
                ldsm_x4(xbox + swz(tok, c), b[j][0], b[j][1], b[j + 1][0], b[j + 1][1]);
            }
        }
        if constexpr (C::kCompute == kMmaTf32) {
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                b[j][0] = to_tf32(b[j][0]);
                b[j][1] = to_tf32(b[j][1]);
            }
        }
#pragma unroll
        for (int t = 0; t < RT; ++t) {
            const int r = wr * RT * 16 + t * 16 + (lane & 15);
            const int c = 2 * ks + (lane >> 4);
            uint32_t a[4];
            ldsm_x4(wbox + swz(r, c), a[0], a[1], a[2], a[3]);
            if constexpr (C::kCompute == kMmaTf32) {
#pragma unroll
                for (int q = 0; q < 4; ++q) a[q] = to_tf32(a[q]);
#pragma unroll
                for (int j = 0; j < MT; ++j) mma_tf32_1688(acc[t][j], a, b[j][0], b[j][1]);
            } else {
#pragma unroll
                for (int j = 0; j < MT; ++j) mma_bf16_16816(acc[t][j], a, b[j][0], b[j][1]);
            }
        }
    }
}

// FP32 FMA box, few tokens (MT == 1): lane = (row group g = lane/8, chunk c = lane%8).
// Each lane owns rows wr*RT*16 + g + 4i (i < 4RT) for all 8 token rows and the
// 4 consecutive k of chunk c; the 8 chunk lanes are added by a fixed butterfly
// at the end.  acc[i][t]: row i, token t.
template <class C, int RT>
__device__ __forceinline__ void box_fma_ksplit(uint32_t wbox, uint32_t xbox, int wr, int lane,
                                               int M, float (&acc)[4 * RT][8]) {
    const int c = lane & 7, g = lane >> 3;
    float4 xv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) xv[t] = lds128(xbox + swz(t, c));
#pragma unroll
    for (int i = 0; i < 4 * RT; ++i) {
        const float4 wv = lds128(wbox + swz(wr * RT * 16 + g + 4 * i, c));
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < M) {
                acc[i][t] = fmaf(wv.x, xv[t].x, acc[i][t]);
                acc[i][t] = fmaf(wv.y, xv[t].y, acc[i][t]);
                acc[i][t] = fmaf(wv.z, xv[t].z, acc[i][t]);
                acc[i][t] = fmaf(wv.w, xv[t].w, acc[i][t]);
            }
        }
    }
}

// FP32 FMA box, many tokens (MT >= 2): lane = (row lane rl = lane%4, token lane
// tl = lane/4); rows wr*RT*16 + rl + 4i (i < 4RT), tokens tl + 8j (j < MT); each
// output is one sequential fma chain over k.
template <class C, int RT, int MT>
__device__ __forceinline__ void box_fma_outer(uint32_t wbox, uint32_t xbox, int wr, int lane,
                                              float (&acc)[4 * RT][MT]) {
    const int rl = lane & 3, tl = lane >> 2;
#pragma unroll 2
    for (int c = 0; c < 8; ++c) {
        float4 wv[4 * RT], xv[MT];
#pragma unroll
        for (int i = 0; i < 4 * RT; ++i) wv[i] = lds128(wbox + swz(wr * RT * 16 + rl + 4 * i, c));
#pragma unroll
        for (int j = 0; j < MT; ++j) xv[j] = lds128(xbox + swz(tl + 8 * j, c));
#pragma unroll
        for (int i = 0; i < 4 * RT; ++i)
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                acc[i][j] = fmaf(wv[i].x, xv[j].x, acc[i][j]);
                acc[i][j] = fmaf(wv[i].y, xv[j].y, acc[i][j]);
                acc[i][j] = fmaf(wv[i].z, xv[j].z, acc[i][j]);
                acc[i][j] = fmaf(wv[i].w, xv[j].w, acc[i][j]);
            }
    }
}

// ---- output scatter -------------------------------------------------------

template <int COMPUTE>
__device__ __forceinline__ void store_out(const StreamArgs &a, int n, int tok, float v) {
    int i = 0;
#pragma unroll 1
    while (i + 1 < a.splits.count && n >= a.splits.off[i + 1]) ++i;
    const int64_t idx = static_cast<int64_t>(tok) * a.splits.rows[i] + (n - a.splits.off[i]);
    if constexpr (COMPUTE == kMmaBf16) {
        static_cast<__nv_bfloat16 *>(a.splits.out[i])[idx] = __float2bfloat16_rn(v);
    } else {
        static_cast<float *>(a.splits.out[i])[idx] = v;
    }
}

// ---- the kernel -------------------------------------------------------------

template <int COMPUTE, int MT, int RT, int WR, int WK>
__global__ void __launch_bounds__(StreamCfg<COMPUTE, MT, RT, WR, WK>::kThreads, 1)
    hsp_stream_kernel(const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ StreamArgs a) {
    using C = StreamCfg<COMPUTE, MT, RT, WR, WK>;
    constexpr int kSlots = C::kSlots, kXRows = C::kXRows, kBoxK = C::kBoxK;

    extern __shared__ uint8_t smem_raw[];
    // Align the ring to 1024 bytes in the shared window (swizzle atom).
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t ring = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.ring_bytes);
    uint64_t *empty = full + a.ring_stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + a.ring_stages);
    int *armed = const_cast<int *>(abort_flag) + 1;  // last stage armed in each slot

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * a.rows_per_cta;
    const int g0 = blockIdx.y * a.stages_per_slice;
    const int nst = max(0, min(a.stages_total, g0 + a.stages_per_slice) - g0);
    const uint32_t x_region = WK * a.w_box_bytes;  // X boxes follow the W boxes in a stage

    if (tid == 0) {
        for (int s = 0; s < a.ring_stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), C::kNCW);
            armed[s] = -1;
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    float acc_mma[(COMPUTE == kFmaFp32) ? 1 : RT][(COMPUTE == kFmaFp32) ? 1 : MT][4];
    float acc_fk[(COMPUTE == kFmaFp32 && MT == 1) ? 4 * RT : 1][8];
    float acc_fo[(COMPUTE == kFmaFp32 && MT > 1) ? 4 * RT : 1][MT];
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc_mma) / sizeof(float)); ++i) (&acc_mma[0][0][0])[i] = 0.f;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc_fk) / sizeof(float)); ++i) (&acc_fk[0][0])[i] = 0.f;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc_fo) / sizeof(float)); ++i) (&acc_fo[0][0])[i] = 0.f;

    if (warp == C::kNCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            tma_prefetch_map(&tmap_w);
            tma_prefetch_map(&tmap_x);
            const int npre = min(nst, a.ring_stages);
            // Weights of the first ring's worth of stages: before the grid dependency.
            for (int i = 0; i < npre; ++i) {
                const int g = g0 + i;
                if (g == a.skip_stage) continue;
                const int nb = min(WK, a.kboxes - g * WK);
                const uint32_t fb = smem_u32(&full[i]);
                const uint32_t base = ring + i * a.stage_bytes;
                mbar_expect_tx(fb, nb * a.w_tx_bytes);
                for (int j = 0; j < nb; ++j)
                    tma_load_2d(base + j * a.w_box_bytes, &tmap_w, (g * WK + j) * kBoxK, row0, fb);
            }
            // Activations are written by the previous kernel on the stream.
            griddep_wait();
            for (int i = 0; i < npre; ++i) {
                const int g = g0 + i;
                if (g == a.skip_stage) continue;
                const int nb = min(WK, a.kboxes - g * WK);
                const uint32_t fb = smem_u32(&full[i]);
                const uint32_t base = ring + i * a.stage_bytes + x_region;
                mbar_arrive_expect_tx(fb, nb * a.x_tx_bytes);
                for (int j = 0; j < nb; ++j)
                    tma_load_2d(base + j * a.x_box_bytes, &tmap_x, (g * WK + j) * kBoxK, 0, fb);
                armed[i] = i;
            }
            for (int i = npre; i < nst; ++i) {
                const int slot = i % a.ring_stages;
                const uint32_t par = static_cast<uint32_t>((i / a.ring_stages) - 1) & 1u;
                if (!thread_wait(smem_u32(&empty[slot]), par, a.wait_limit_ns, abort_flag)) {
                    record_timeout(a.err_word, abort_flag);
                    break;
                }
                const int g = g0 + i;
                if (g == a.skip_stage) continue;
                const int nb = min(WK, a.kboxes - g * WK);
                const uint32_t fb = smem_u32(&full[slot]);
                const uint32_t base = ring + slot * a.stage_bytes;
                mbar_arrive_expect_tx(fb, nb * (a.w_tx_bytes + a.x_tx_bytes));
                for (int j = 0; j < nb; ++j)
                    tma_load_2d(base + j * a.w_box_bytes, &tmap_w, (g * WK + j) * kBoxK, row0, fb);
                for (int j = 0; j < nb; ++j)
                    tma_load_2d(base + x_region + j * a.x_box_bytes, &tmap_x, (g * WK + j) * kBoxK,
                                0, fb);
                armed[slot] = i;
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers ----------------
        const int wk = warp % WK, wr = warp / WK;
        const bool has_rows = wr * RT * 16 < a.rows_per_cta;
        for (int i = 0; i < nst; ++i) {
            const int slot = i % a.ring_stages;
            const uint32_t par = static_cast<uint32_t>(i / a.ring_stages) & 1u;
            if (!warp_wait(smem_u32(&full[slot]), par, a.wait_limit_ns, abort_flag)) {
                if (lane == 0) record_timeout(a.err_word, abort_flag);
                break;
            }
            const int b = (g0 + i) * WK + wk;
            if (b < a.kboxes && has_rows) {
                const uint32_t wbox = ring + slot * a.stage_bytes + wk * a.w_box_bytes;
                const uint32_t xbox = ring + slot * a.stage_bytes + x_region + wk * a.x_box_bytes;
                if constexpr (COMPUTE == kFmaFp32) {
                    if constexpr (MT == 1)
                        box_fma_ksplit<C, RT>(wbox, xbox, wr, lane, a.M, acc_fk);
                    else
                        box_fma_outer<C, RT, MT>(wbox, xbox, wr, lane, acc_fo);
                } else {
                    box_mma<C, RT, MT>(wbox, xbox, wr, lane, acc_mma);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
        }
    }

    // All ring reads are done (or abandoned).  [A]
    __syncthreads();
    const bool aborted = (*abort_flag != 0);
    if (aborted) {
        // Let copies still in flight land before the ring is reused or freed.
        if (warp == C::kNCW && lane == 0) {
            const uint64_t limit = a.wait_limit_ns / 16 + 1;
            for (int s = 0; s < a.ring_stages; ++s) {
                const int i = armed[s];
                if (i < 0) continue;
                const uint32_t par = static_cast<uint32_t>(i / a.ring_stages) & 1u;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_u32(&full[s]), par) && global_timer_ns() - t0 < limit) {
                }
            }
        }
        __syncthreads();
    }

    // ---- per-warp partials -> red[wk][slot][tok] (aliases the ring) ----
    float *red = reinterpret_cast<float *>(smem);
    if (warp < C::kNCW && !aborted) {
        const int wk = warp % WK, wr = warp / WK;
        if constexpr (COMPUTE == kFmaFp32) {
            if constexpr (MT == 1) {
                const int c = lane & 7, g = lane >> 3;
#pragma unroll
                for (int i = 0; i < 4 * RT; ++i)
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        float v = acc_fk[i][t];
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        if (c == 0) red[(wk * kSlots + wr * RT * 16 + g + 4 * i) * kXRows + t] = v;
                    }
            } else {
                const int rl = lane & 3, tl = lane >> 2;
#pragma unroll
                for (int i = 0; i < 4 * RT; ++i)
#pragma unroll
                    for (int j = 0; j < MT; ++j)
                        red[(wk * kSlots + wr * RT * 16 + rl + 4 * i) * kXRows + tl + 8 * j] = acc_fo[i][j];
            }
        } else {
#pragma unroll
            for (int t = 0; t < RT; ++t)
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    const int s0 = wr * RT * 16 + t * 16 + (lane >> 2);
                    const int t0 = j * 8 + 2 * (lane & 3);
                    float *p0 = red + (wk * kSlots + s0) * kXRows + t0;
                    float *p1 = red + (wk * kSlots + s0 + 8) * kXRows + t0;
                    p0[0] = acc_mma[t][j][0];
                    p0[1] = acc_mma[t][j][1];
                    p1[0] = acc_mma[t][j][2];
                    p1[1] = acc_mma[t][j][3];
                }
        }
    }
    __syncthreads();

    // Outputs may still be read by the previous kernel on the stream.
    griddep_wait();

    // ---- warp partials added in warp order; single-slice CTAs store here ----
    const int rows_here = min(a.rows_per_cta, a.n_rows - row0);
    if (!aborted) {
        for (int e = tid; e < kSlots * kXRows; e += C::kThreads) {
            const int tok = e / kSlots, slot = e - tok * kSlots;
            if (tok >= a.M || slot >= rows_here) continue;
            float v = red[slot * kXRows + tok];
#pragma unroll
            for (int q = 1; q < WK; ++q) v += red[(q * kSlots + slot) * kXRows + tok];
            if (a.slices == 1)
                store_out<COMPUTE>(a, row0 + slot, tok, v);
            else
                red[slot * kXRows + tok] = v;
        }
    }

    if (a.slices > 1) {
        // ---- K slices of the cluster added in slice order (DSMEM) ----
        cluster_sync_all();
        if (!aborted) {
            const int per = kSlots / a.slices;
            const int my = static_cast<int>(blockIdx.y);
            const uint32_t red_local = smem_u32(red);
            for (int e = tid; e < per * kXRows; e += C::kThreads) {
                const int tok = e / per, slot = my * per + (e - tok * per);
                if (tok >= a.M || slot >= rows_here) continue;
                const uint32_t off = red_local + static_cast<uint32_t>((slot * kXRows + tok) * 4);
                float v = ld_shared_cluster_f32(cluster_map_shared(off, 0));
                for (int q = 1; q < a.slices; ++q)
                    v += ld_shared_cluster_f32(cluster_map_shared(off, static_cast<uint32_t>(q)));
                store_out<COMPUTE>(a, row0 + slot, tok, v);
            }
        }
        cluster_sync_all();  // no CTA leaves while a peer may still read its partials
    }

    // Trigger the dependent launch only after every output store of this CTA.
    __threadfence();
    __syncthreads();
    griddep_launch_dependents();
}

}  // namespace hsp
