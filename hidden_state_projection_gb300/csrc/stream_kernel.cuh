// stream_kernel.cuh -- the weight-streaming projection kernel.
//
// Computes, for the rows [row0, row0 + R) of one launch's weight rows and all M
// tokens,  y[m][n] = sum_k x[m][k] * w[n][k]  with fp32 accumulation, rounds once
// and scatters every row into the output of the projection it belongs to
// (TensorRT-LLM PR #20636, Description: one GEMM over the row-concatenated
// weight, halves returned as dense [M, N_i] outputs).
//
// Structure of one CTA (after the pages' GLM fused-A kernel -- weights copied
// in before the grid-dependency wait, activations after it, warp sums added in
// warp order and rounded once; TensorRT-LLM PR #20502, glmFusedAGemm commit
// message -- re-drawn for bulk-copy rings and clusters on sm_103a):
//
//   * a ring of shared-memory stages is filled by the copy engine.  When a row is a
//     whole number of 128-byte units (every workload of the pages), one thread of
//     the ninth warp issues TWO 3-D tensor copies per stage: the weight box
//     [stage_units][R rows][128 bytes] and the token box [stage_units][M][128 bytes],
//     both with the 128-byte swizzle, so that the eight rows an ldmatrix phase
//     reads sit in eight different bank groups.  The copy engine accepts about one
//     copy per 55 cycles per SM, so one large box per stage replaces the R + M
//     row copies of the other layout and leaves the stages short (small compute
//     tail after the last byte).  (fp32 FMA above 8 tokens: one weight box per
//     unit, [R rows][128 bytes], so that every unit starts on the same swizzle
//     phase, and token boxes 8 * MT rows high.)  Otherwise (a ragged last unit)
//     each weight row and token row of a stage is one 1-D bulk copy of a contiguous
//     segment, rows padded to a pitch of 16 mod 128 bytes, issued lane-parallel by
//     all nine warps.  Weight copies of the first stages (tensor layout: two, one
//     with token tiles; bulk layout: the first ring's worth) are issued before
//     griddepcontrol.wait, token copies only after it; a slot is refilled once
//     every consumer has released it;
//   * consumer warp (wr, wk) takes every k-unit u (128 bytes of K) of a stage
//     with u mod WK == wk, for its RT 16-row tiles, and accumulates in registers
//     (mma.sync bf16 / tf32, or fp32 FMA); fp32 FMA with more than 8 tokens instead
//     gives warp wk the 16-byte chunk wk of every unit, for all row slots of the CTA
//     (equal shares for any unit count, large register tiles);
//   * the WK warp partials of each output are added in warp order, then (S > 1)
//     the S CTAs of a cluster, each holding one K slice, add their partials in
//     slice order through distributed shared memory;
//   * the sum is rounded once and stored; every storing thread fences, the CTA
//     synchronises, and only then is the dependent launch triggered (the trigger
//     follows the stores, the robust order TensorRT-LLM PR #20636, Description,
//     recommends).
//
// Determinism: the summation order of an output depends only on (K, the element
// type, WK, S) -- never on the row count, the stage width, the row's position in a
// tile, the grid or the arrival order -- so fused and per-projection launches,
// repeated runs and graph replays give identical bits.
//
// Fragment reads of rows past the CTA's last weight row, and of token rows past M,
// are clamped to the last real row; their results are never stored.  The tensor
// copies zero-fill rows and units past the tensor; a final partial k-unit (bulk
// layout only) is zero-filled in shared memory before use.
//
// Every wait on a shared-memory barrier is bounded (globaltimer); on expiry the
// kernel records PROJ_ERR_TIMEOUT in the device error word, stops computing,
// skips its stores, waits (bounded) for its own copies still in flight, and
// returns through the same barriers as a normal exit.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "norm_epilogue.cuh"
#include "prefetch.cuh"
#include "ptx.cuh"
#include "scatter.cuh"
#include "stream_args.h"

namespace hsp {

template <int COMPUTE, int MT, int RT, int WR, int WK>
struct StreamCfg {
    static constexpr int kCompute = COMPUTE;
    static constexpr int kNCW = WR * WK;                 // consumer warps
    static constexpr int kNW = kNCW + 1;                 // + one issue-only warp
    static constexpr int kThreads = kNW * 32;
    static constexpr int kSlots = WR * RT * 16;          // row slots per CTA
    static constexpr int kXRows = 8 * MT;                // token slots
    static_assert(WR * WK == 8, "eight consumer warps");
    static_assert(MT == 1 || MT % 2 == 0, "token tiles: 1 or even");
};

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

// Shared-memory view of one stage, addressed by (row, unit of the stage, 16-byte
// chunk of the unit).  Reads past the real rows are clamped to the last one.
template <bool TENSOR>
struct StageView;

// Bulk layout: weight rows [0, R) then token rows, each `pitch` bytes apart.
template <>
struct StageView<false> {
    uint32_t w, x;     // shared addresses of weight row 0 / token row 0
    uint32_t pitch;
    int rmax, tmax;    // last real weight row / token row
    __device__ __forceinline__ uint32_t wa(int r, int ul, int c) const {
        return w + static_cast<uint32_t>(min(r, rmax)) * pitch + static_cast<uint32_t>(ul * kUnitBytes + c * 16);
    }
    __device__ __forceinline__ uint32_t xa(int t, int ul, int c) const {
        return x + static_cast<uint32_t>(min(t, tmax)) * pitch + static_cast<uint32_t>(ul * kUnitBytes + c * 16);
    }
};

// Tensor layout: line L = unit * rows + row of 128 bytes; chunk c of line L is stored
// at chunk c ^ (L mod 8) (the copy engine's 128-byte swizzle; both boxes start on a
// 1024-byte boundary).
template <>
struct StageView<true> {
    uint32_t w, x;
    int wrows, xrows;  // box rows: R and M
    int rmax, tmax;
    __device__ __forceinline__ uint32_t wa(int r, int ul, int c) const {
        const int L = ul * wrows + min(r, rmax);
        return w + static_cast<uint32_t>(L * kUnitBytes + ((c ^ (L & 7)) << 4));
    }
    __device__ __forceinline__ uint32_t xa(int t, int ul, int c) const {
        const int L = ul * xrows + min(t, tmax);
        return x + static_cast<uint32_t>(L * kUnitBytes + ((c ^ (L & 7)) << 4));
    }
};

// ---- inner products on one 128-byte k-unit (unit `ul` of the stage) ----

// Tensor cores: 4 k-steps (k16 for bf16, k8 for tf32) over the warp's row tiles.
// All fragment loads of a batch of k-steps are issued before its products, so
// their shared-memory latencies overlap (the whole unit for up to two token
// tiles, two k-steps at a time for more).  With one token tile (M <= 8) the even
// and odd k-steps feed two accumulator chains (acc[0], acc[1]) that are added at
// the end: half the dependent MMA latency.  With more token tiles the tiles
// themselves are independent chains.
template <class C, int RT, int MT, int NCH, class V>
__device__ __forceinline__ void unit_mma(const V &v, int ul, int wr, int lane, float (&acc)[NCH][RT][MT][4]) {
    constexpr int kBatch = (MT >= 4) ? 2 : 4;
    constexpr int kMask = NCH - 1;
#pragma unroll
    for (int k0 = 0; k0 < 4; k0 += kBatch) {
        uint32_t b[kBatch][MT][2];
        uint32_t a[kBatch][RT][4];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int cb = 2 * (k0 + q) + ((lane >> 3) & 1);   // 16-byte chunk of the token rows
            if constexpr (MT == 1) {
                ldsm_x2(v.xa(lane & 7, ul, cb), b[q][0][0], b[q][0][1]);
            } else {
#pragma unroll
                for (int j = 0; j < MT; j += 2) {
                    const int tok = (j + (lane >> 4)) * 8 + (lane & 7);
                    ldsm_x4(v.xa(tok, ul, cb), b[q][j][0], b[q][j][1], b[q][j + 1][0], b[q][j + 1][1]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int ca = 2 * (k0 + q) + (lane >> 4);          // 16-byte chunk of the weight rows
#pragma unroll
            for (int t = 0; t < RT; ++t)
                ldsm_x4(v.wa(wr * RT * 16 + t * 16 + (lane & 15), ul, ca), a[q][t][0], a[q][t][1], a[q][t][2],
                        a[q][t][3]);
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int ks = k0 + q;
            if constexpr (C::kCompute == kMmaTf32) {
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    b[q][j][0] = to_tf32(b[q][j][0]);
                    b[q][j][1] = to_tf32(b[q][j][1]);
                }
#pragma unroll
                for (int t = 0; t < RT; ++t) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) a[q][t][e] = to_tf32(a[q][t][e]);
#pragma unroll
                    for (int j = 0; j < MT; ++j) mma_tf32_1688(acc[ks & kMask][t][j], a[q][t], b[q][j][0], b[q][j][1]);
                }
            } else {
#pragma unroll
                for (int t = 0; t < RT; ++t)
#pragma unroll
                    for (int j = 0; j < MT; ++j) mma_bf16_16816(acc[ks & kMask][t][j], a[q][t], b[q][j][0], b[q][j][1]);
            }
        }
    }
}

// FMA, few tokens (MT == 1), fp32 or bf16 elements: lane = (row group g = lane/8,
// 16-byte chunk c = lane%8).  Each lane owns rows wr*RT*16 + g + 4i (i < 4RT) for
// the first TOK token slots and the 4 (fp32) or 8 (bf16) consecutive k of chunk c;
// the 8 chunk lanes are added by a fixed butterfly at the end.  Only tokens below M
// are loaded and multiplied.  acc[i][t]: row i, token t.
__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[8]) {
    // bf16 pairs: the low half is the first element (the top 16 bits of an fp32)
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xFFFF0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xFFFF0000u);
    f[4] = __uint_as_float(u.z << 16);
    f[5] = __uint_as_float(u.z & 0xFFFF0000u);
    f[6] = __uint_as_float(u.w << 16);
    f[7] = __uint_as_float(u.w & 0xFFFF0000u);
}

template <class C, int RT, int TOK, class V>
__device__ __forceinline__ void unit_fma_ksplit(const V &v, int ul, int wr, int lane, int M, float (&acc)[4 * RT][8]) {
    constexpr int E = (C::kCompute == kFmaBf16) ? 8 : 4;  // elements per 16-byte chunk
    const int c = lane & 7, g = lane >> 3;
    float xf[TOK][E];
#pragma unroll
    for (int t = 0; t < TOK; ++t)
        if (t < M) unpack16(lds128u(v.xa(t, ul, c)), xf[t]);
#pragma unroll
    for (int i = 0; i < 4 * RT; ++i) {
        float wf[E];
        unpack16(lds128u(v.wa(wr * RT * 16 + g + 4 * i, ul, c)), wf);
#pragma unroll
        for (int t = 0; t < TOK; ++t)
            if (t < M) {
#pragma unroll
                for (int e = 0; e < E; ++e) acc[i][t] = fmaf(wf[e], xf[t][e], acc[i][t]);
            }
    }
}

// FP32 FMA, more than 8 tokens: warp wk takes the 16-byte chunk wk (4 consecutive k)
// of EVERY unit, so the eight warps share any unit count equally.  Lane = (row lane
// rl = lane % LR, token lane tl = lane / LR); it owns rows rl + LR*i (i < RPL) and
// tokens tl + (32/LR)*j (j < TPL), an RPL x TPL register tile: per unit RPL + TPL
// 16-byte shared loads feed 4*RPL*TPL FMAs (8 x 8 at 64 tokens: 16 loads per 256 FMAs;
// 12 x 8 with three row tiles;
// measured on GB300 ~70% of the FMA pipe on a resident stage, against ~53% for one
// unit per warp with 4 x 8 tiles).  Each output of a warp is one sequential fma chain
// over its chunks in increasing k.
template <int RPL, int TPL, int LR, class V>
__device__ __forceinline__ void unit_fma_chunk(const V &v, int ul, int c, int lane, float (&acc)[RPL][TPL]) {
    constexpr int TS = 32 / LR;
    const int rl = lane % LR, tl = lane / LR;
    float4 wv[RPL], xv[TPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) wv[i] = lds128(v.wa(rl + LR * i, ul, c));
#pragma unroll
    for (int j = 0; j < TPL; ++j) xv[j] = lds128(v.xa(tl + TS * j, ul, c));
#pragma unroll
    for (int i = 0; i < RPL; ++i)
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
            acc[i][j] = fmaf(wv[i].x, xv[j].x, acc[i][j]);
            acc[i][j] = fmaf(wv[i].y, xv[j].y, acc[i][j]);
            acc[i][j] = fmaf(wv[i].z, xv[j].z, acc[i][j]);
            acc[i][j] = fmaf(wv[i].w, xv[j].w, acc[i][j]);
        }
}

// The same products on the chunk layout's tensor-copy stage: unit rows kSlots (weights)
// and kXRows (tokens) lines apart, both multiples of 8, so that line rl + LR*i has the
// swizzle phase rl + LR*i mod 8 = (rl mod 8) + 4*(i odd, LR = 4) in every unit.  w0 / w1
// (x0 / x1) address the lane's first even / odd row (token) of this unit, chunk swizzled;
// the other rows follow at compile-time offsets.
template <int RPL, int TPL, int LR>
__device__ __forceinline__ void unit_fma_chunk_sw(uint32_t w0, uint32_t w1, uint32_t x0, uint32_t x1,
                                                  float (&acc)[RPL][TPL]) {
    constexpr int TS = 32 / LR;
    float4 wv[RPL], xv[TPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) wv[i] = lds128(((i & 1) ? w1 : w0) + static_cast<uint32_t>(i * LR * kUnitBytes));
#pragma unroll
    for (int j = 0; j < TPL; ++j) xv[j] = lds128(((j & 1) ? x1 : x0) + static_cast<uint32_t>(j * TS * kUnitBytes));
#pragma unroll
    for (int i = 0; i < RPL; ++i)
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
            acc[i][j] = fmaf(wv[i].x, xv[j].x, acc[i][j]);
            acc[i][j] = fmaf(wv[i].y, xv[j].y, acc[i][j]);
            acc[i][j] = fmaf(wv[i].z, xv[j].z, acc[i][j]);
            acc[i][j] = fmaf(wv[i].w, xv[j].w, acc[i][j]);
        }
}

// Zero the bytes [valid, 128) of one k-unit in every loaded row (the tail of K;
// bulk layout only: the tensor layout is used only when K has no partial unit).
__device__ __forceinline__ void zero_unit_tail(const StageView<false> &v, int ul, uint32_t valid, int lane) {
    const int chunks = static_cast<int>((128u - valid) >> 4);
    const int rows = v.rmax + 1 + v.tmax + 1;
    for (int idx = lane; idx < rows * chunks; idx += 32) {
        const int r = idx / chunks, c = idx - r * chunks;
        const uint32_t base = (r <= v.rmax) ? v.wa(r, ul, 0) : v.xa(r - v.rmax - 1, ul, 0);
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + valid + c * 16), "r"(0u)
                     : "memory");
    }
    __syncwarp();
}

// ---- the kernel -------------------------------------------------------------

// NORM: the RMSNorm epilogue is compiled in (only bf16 instances with one token
// tile carry it; the others have no call, parked-value branch or flag of it).
template <int COMPUTE, int MT, int RT, int WR, int WK, bool TENSOR, bool NORM>
__global__ void __launch_bounds__(StreamCfg<COMPUTE, MT, RT, WR, WK>::kThreads, 1)
    hsp_stream_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                      const __grid_constant__ StreamArgs a) {
    using C = StreamCfg<COMPUTE, MT, RT, WR, WK>;
    constexpr int kSlots = C::kSlots, kXRows = C::kXRows;
    // fp32 FMA above 8 tokens: one 16-byte chunk of every unit per warp (unit_fma_chunk).
    // With tensor copies its stage holds each unit's weight rows at a stride of kSlots
    // lines (one copy per unit) and its token rows at a stride of kXRows lines (token
    // rows past M zero-filled), so that a lane's swizzle phases do not change from unit
    // to unit.
    constexpr bool kChunk = (COMPUTE == kFmaFp32 && MT > 1);
    static_assert(!kChunk || (WR == 1 && WK == 8), "chunk layout: eight K warps over all row slots");
    constexpr int kLR = (MT == 8) ? 4 : 8;   // row lanes
    constexpr int kTS = 32 / kLR;            // token lanes
    constexpr int kTPL = kXRows / kTS;       // tokens per lane
    constexpr int kRPL = kSlots / kLR;       // rows per lane
    // Row pitch (floats) of the partial-sum buffer red[warp][slot][token].  The combine
    // loop reads one token of 32 consecutive rows per warp instruction (chunk layout: 32
    // consecutive tokens of one row), so the pitch is one more than the token slots --
    // 32 banks (a pitch of 8 * MT read one bank 8- to 32-fold).  The chunk layout's lanes
    // each write a tile of rows rl + kLR*i and tokens tl + kTS*j: with a pitch of
    // kXRows + kTS (rl * pitch + tl covers 32 banks) those writes are conflict-free too.
    constexpr int kXP = kChunk ? kXRows + kTS : kXRows + 1;
    // Row pitch of the K-slice reduction's staging and receive blocks: a multiple of
    // four floats, so that each owner's block is a whole number of 16-byte chunks (the
    // unit of a bulk copy between cluster shared memories).
    constexpr int kSP = kXRows + 4;

    // The ring starts on a 1024-byte boundary (the swizzle pattern of the tensor
    // layout repeats every 1024 bytes).
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t ring = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.ring_bytes);
    uint64_t *empty = full + a.ring_stages;
    uint64_t *recv_bar = empty + a.ring_stages;  // the K-slice partials of my rows (S > 1)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(recv_bar + 1);
    int *armed = const_cast<int *>(abort_flag) + 1;  // last stage armed in each slot
    // (then kMaxSplits ints for the RMSNorm epilogue's "finish this split" flags)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * a.rows_per_cta;
    const int rows_here = min(a.rows_per_cta, a.n_rows - row0);
    const int slice = blockIdx.y;
    const int u_slice0 = slice * a.units_per_slice;
    const int u_slice1 = min(a.units_total, u_slice0 + a.units_per_slice);
    const int nst = max(0, (u_slice1 - u_slice0 + a.stage_units - 1) / a.stage_units);
    const int npre = min(nst, a.ring_stages);
    // The tensor layout has one producer thread (one arrival per phase); in the bulk
    // layout every warp issues a share of each stage and arrives once.
    constexpr uint32_t kFullCount = TENSOR ? 1u : static_cast<uint32_t>(C::kNW);
    const bool producer = TENSOR && warp == C::kNCW && lane == 0;

    const uint64_t w_policy = l2_policy_evict_first();
    // Tensor layout: weight stages requested before the grid-dependency wait.  The rest of
    // the first ring goes out after the wait, behind the first stages' token boxes: with
    // the whole ring requested at entry the DRAM serves every CTA's stages interleaved and
    // each CTA's first stage lands late (measured on GB300, graphs of back-to-back calls:
    // two stages instead of the full ring took qk_indexer M = 1 / 8 from 7.96 / 8.34 to
    // 7.53 / 7.59 us and glm_fused_a M = 1 / 8 from 8.53 / 9.03 to 8.25 / 8.59; with token
    // tiles one stage did best, fp32 M = 16 6.66 -> 6.49 us, tf32 M = 64 8.67 -> 8.45).
    constexpr int kPreWaitStages = (MT == 1) ? 2 : 1;
    // every stage's box holds the same bytes (units past the tensor are zero-filled)
    const uint32_t stage_tx =
        static_cast<uint32_t>((a.rows_per_cta + (kChunk ? kXRows : a.M)) * a.stage_units * kUnitBytes);
    // ---------------- tensor layout: one producer thread, two boxes per stage ----------------
    // (chunk layout: one weight box per unit, [R][128 bytes], kSlots lines apart)
    auto tensor_w = [&](int i, int slot) {
        if constexpr (kChunk) {
            for (int k = 0; k < a.stage_units; ++k)
                tma_load_3d_hint(ring + slot * a.stage_bytes + static_cast<uint32_t>(k * kSlots * kUnitBytes), &tmap_w,
                                 0, row0, u_slice0 + i * a.stage_units + k, smem_u32(&full[slot]), w_policy);
        } else {
            tma_load_3d_hint(ring + slot * a.stage_bytes, &tmap_w, 0, row0, u_slice0 + i * a.stage_units,
                             smem_u32(&full[slot]), w_policy);
        }
    };
    auto tensor_x = [&](int i, int slot) {
        tma_load_3d(ring + slot * a.stage_bytes + a.x_off, &tmap_x, 0, 0, u_slice0 + i * a.stage_units,
                    smem_u32(&full[slot]));
    };

    // The barriers are initialised by the producer (tensor layout) or by thread 0.
    if (TENSOR ? producer : tid == 0) {
        for (int s = 0; s < a.ring_stages; ++s) {
            mbar_init(smem_u32(&full[s]), kFullCount);
            mbar_init(smem_u32(&empty[s]), C::kNCW);
            armed[s] = -1;
        }
        mbar_init(smem_u32(recv_bar), 1);
        // every slice's block of my rows arrives on recv_bar: expect all of them now
        if (a.slices > 1) mbar_arrive_expect_tx(smem_u32(recv_bar), static_cast<uint32_t>(kSlots * kSP * 4));
        *abort_flag = 0;
        mbar_fence_init();
        if constexpr (TENSOR) {
            // Weights of the first ring's worth of stages: before the grid dependency,
            // and before the CTA barrier (they need nothing but the barriers above).
            tma_prefetch_map(&tmap_w);
            tma_prefetch_map(&tmap_x);
            for (int i = 0; i < min(npre, kPreWaitStages); ++i) {
                if (i == a.skip_stage) continue;
                mbar_arrive_expect_tx(smem_u32(&full[i]), stage_tx);
                tensor_w(i, i);
                armed[i] = i;
            }
        }
    }
    __syncthreads();
    if (a.trigger_early) griddep_launch_dependents();  // option trigger_early (the tinygemm2 order)

    constexpr bool kFma = (COMPUTE == kFmaFp32 || COMPUTE == kFmaBf16);
    constexpr int kChains = (!kFma && MT == 1) ? 2 : 1;
    float acc_mma[kChains][kFma ? 1 : RT][kFma ? 1 : MT][4];
    float acc_fk[(kFma && MT == 1) ? 4 * RT : 1][8];
    float acc_fo[kChunk ? kRPL : 1][kChunk ? kTPL : 1];
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc_mma) / sizeof(float)); ++i) (&acc_mma[0][0][0][0])[i] = 0.f;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc_fk) / sizeof(float)); ++i) (&acc_fk[0][0])[i] = 0.f;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(acc_fo) / sizeof(float)); ++i) (&acc_fo[0][0])[i] = 0.f;

    // ---------------- bulk layout: copy issue by every warp, lane-parallel ----------------
    // Warp `warp` copies weight rows r = warp + 9 l and token rows t = warp + 9 l;
    // lane l issues the copy of its row, after lane 0 has raised the stage's
    // expected byte count by the warp's share.  Each warp arrives once per phase.
    const char *wrow0 = a.w + static_cast<int64_t>(row0) * a.row_bytes;
    auto span = [&](int i, int64_t &byte0, uint32_t &nbytes) {
        const int u0 = u_slice0 + i * a.stage_units;
        const int u1 = min(u0 + a.stage_units, u_slice1);
        byte0 = static_cast<int64_t>(u0) * kUnitBytes;
        const int64_t end = min(static_cast<int64_t>(u1) * kUnitBytes, a.row_bytes);
        nbytes = static_cast<uint32_t>(end - byte0);
    };
    const int my_rows = rows_here > warp ? (rows_here - warp + C::kNW - 1) / C::kNW : 0;
    const int my_toks = a.M > warp ? (a.M - warp + C::kNW - 1) / C::kNW : 0;
    // lanes past 32 loop (a CTA has at most 128 rows and 64 tokens)
    auto issue_w = [&](int slot, int64_t byte0, uint32_t nbytes, uint32_t fb) {
        const uint32_t base = ring + slot * a.stage_bytes;
        for (int l = lane; l < my_rows; l += 32) {
            const int r = warp + C::kNW * l;
            bulk_load_hint(base + r * a.pitch, wrow0 + r * a.row_bytes + byte0, nbytes, fb, w_policy);
        }
    };
    auto issue_x = [&](int slot, int64_t byte0, uint32_t nbytes, uint32_t fb) {
        const uint32_t base = ring + slot * a.stage_bytes + a.x_off;
        for (int l = lane; l < my_toks; l += 32) {
            const int t = warp + C::kNW * l;
            bulk_load(base + t * a.pitch, a.x + t * a.row_bytes + byte0, nbytes, fb);
        }
    };
    // Weights of the first ring's worth of stages (bulk layout): before the grid dependency.
    if constexpr (!TENSOR) {
        for (int i = 0; i < npre; ++i) {
            if (i == a.skip_stage) continue;
            int64_t b0;
            uint32_t nb;
            span(i, b0, nb);
            if (lane == 0 && my_rows > 0) mbar_expect_tx(smem_u32(&full[i]), static_cast<uint32_t>(my_rows) * nb);
            __syncwarp();
            issue_w(i, b0, nb, smem_u32(&full[i]));
        }
    }
    // Activations are written by the previous kernel on the stream.
    griddep_wait();
    if constexpr (TENSOR) {
        if (producer)
            for (int i = 0; i < npre; ++i) {
                if (i == a.skip_stage) continue;
                if (i >= kPreWaitStages) {  // the rest of the first ring, after its predecessors' tokens
                    mbar_arrive_expect_tx(smem_u32(&full[i]), stage_tx);
                    tensor_w(i, i);
                    armed[i] = i;
                }
                tensor_x(i, i);
            }
    } else {
        for (int i = 0; i < npre; ++i) {
            if (i == a.skip_stage) continue;
            int64_t b0;
            uint32_t nb;
            span(i, b0, nb);
            if (lane == 0) {
                mbar_arrive_expect_tx(smem_u32(&full[i]), static_cast<uint32_t>(my_toks) * nb);
                if (warp == 0) armed[i] = i;
            }
            __syncwarp();
            issue_x(i, b0, nb, smem_u32(&full[i]));
        }
    }
    __syncwarp();
    // Weights of later kernels named by the caller: into L2, after this CTA's own
    // copies (the copy engine serves requests in order; prefetches queued ahead of
    // the token copies would hold up the first stage).
    if (warp == C::kNCW && a.prefetch.count > 0)
        prefetch_ranges_l2(a.prefetch, blockIdx.y * gridDim.x + blockIdx.x, gridDim.x * gridDim.y, lane);

    const int wk = warp % WK, wr = warp / WK;
    const bool consumer = warp < C::kNCW;
    const bool has_rows = consumer && wr * RT * 16 < rows_here;
    if constexpr (TENSOR) {
        // ---------------- tensor layout: the producer refills released slots ----------------
        if (producer) {
            for (int j = npre; j < nst; ++j) {
                const int slot = j % a.ring_stages;
                const uint32_t par = static_cast<uint32_t>((j / a.ring_stages) - 1) & 1u;
                if (!thread_wait(smem_u32(&empty[slot]), par, a.wait_limit_ns, abort_flag)) {
                    record_timeout(a.err_word, abort_flag);
                    break;
                }
                if (j == a.skip_stage) continue;
                mbar_arrive_expect_tx(smem_u32(&full[slot]), stage_tx);
                tensor_w(j, slot);
                tensor_x(j, slot);
                armed[slot] = j;
            }
        }
        __syncwarp();  // the producer's warp reconverges before the barriers below
    }
    // ---------------- consume stage i (bulk layout: then refill its slot with stage i + ring) ----------------
    for (int i = 0; i < nst; ++i) {
        const int slot = i % a.ring_stages;
        const uint32_t par = static_cast<uint32_t>(i / a.ring_stages) & 1u;
        if (consumer) {
            if (!warp_wait(smem_u32(&full[slot]), par, a.wait_limit_ns, abort_flag)) {
                if (lane == 0) record_timeout(a.err_word, abort_flag);
                break;
            }
            const int u0 = u_slice0 + i * a.stage_units;
            const int u1 = min(u0 + a.stage_units, u_slice1);
            StageView<TENSOR> v;
            v.w = ring + slot * a.stage_bytes;
            v.x = v.w + a.x_off;
            if constexpr (TENSOR) {
                v.wrows = a.rows_per_cta;
                v.xrows = a.M;
            } else {
                v.pitch = a.pitch;
            }
            v.rmax = rows_here - 1;
            v.tmax = a.M - 1;
            bool zeroed = false;
            if constexpr (kChunk) {
                // chunk wk of every unit of the stage, in increasing order; a chunk past the
                // end of the row (bulk layout, ragged last unit) adds nothing and is skipped
                // (K * 4 is a multiple of 16: a chunk is wholly inside the row or past it)
                if (has_rows) {
                    if constexpr (TENSOR) {
                        // lane offsets of its first even / odd row and token line (chunk wk,
                        // swizzled); rows past R and tokens past M hold data never stored
                        const int rl = lane % kLR, tl = lane / kLR;
                        const uint32_t wb0 = static_cast<uint32_t>(rl * kUnitBytes + ((wk ^ (rl & 7)) << 4));
                        const uint32_t wb1 = static_cast<uint32_t>(rl * kUnitBytes + ((wk ^ ((rl + kLR) & 7)) << 4));
                        const uint32_t xb0 = static_cast<uint32_t>(tl * kUnitBytes + ((wk ^ (tl & 7)) << 4));
                        const uint32_t xb1 = static_cast<uint32_t>(tl * kUnitBytes + ((wk ^ ((tl + kTS) & 7)) << 4));
#pragma unroll 2
                        for (int u = u0; u < u1; ++u) {
                            const uint32_t uw = v.w + static_cast<uint32_t>((u - u0) * kSlots * kUnitBytes);
                            const uint32_t ux = v.x + static_cast<uint32_t>((u - u0) * kXRows * kUnitBytes);
                            unit_fma_chunk_sw<kRPL, kTPL, kLR>(uw + wb0, uw + wb1, ux + xb0, ux + xb1, acc_fo);
                        }
                    } else {
#pragma unroll 2
                        for (int u = u0; u < u1; ++u) {
                            if (static_cast<int64_t>(u) * kUnitBytes + wk * 16 >= a.row_bytes) continue;
                            unit_fma_chunk<kRPL, kTPL, kLR>(v, u - u0, wk, lane, acc_fo);
                        }
                    }
                }
            } else {
                // units of this warp: u = u0 + j with u mod WK == wk, in increasing order
                for (int u = u0 + ((wk - u0 % WK) % WK + WK) % WK; u < u1; u += WK) {
                    const int ul = u - u0;
                    if constexpr (!TENSOR) {
                        const int64_t valid = a.row_bytes - static_cast<int64_t>(u) * kUnitBytes;
                        if (valid < kUnitBytes) {
                            zero_unit_tail(v, ul, static_cast<uint32_t>(valid), lane);
                            zeroed = true;
                        }
                    }
                    if (!has_rows) continue;
                    if constexpr (COMPUTE == kFmaBf16) {
                        unit_fma_ksplit<C, RT, 2>(v, ul, wr, lane, a.M, acc_fk);
                    } else if constexpr (COMPUTE == kFmaFp32) {
                        unit_fma_ksplit<C, RT, 8>(v, ul, wr, lane, a.M, acc_fk);  // MT == 1
                    } else {
                        unit_mma<C, RT, MT, kChains>(v, ul, wr, lane, acc_mma);
                    }
                }
            }
            if (zeroed) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
        }
        if constexpr (!TENSOR) {
            const int j = i + a.ring_stages;
            if (j < nst) {
                // every consumer has released the slot: issue this warp's share of stage j
                if (!warp_wait(smem_u32(&empty[slot]), par, a.wait_limit_ns, abort_flag)) {
                    if (lane == 0) record_timeout(a.err_word, abort_flag);
                    break;
                }
                if (j != a.skip_stage) {
                    int64_t b0;
                    uint32_t nb;
                    span(j, b0, nb);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(smem_u32(&full[slot]), static_cast<uint32_t>(my_rows + my_toks) * nb);
                        if (warp == 0) armed[slot] = j;
                    }
                    __syncwarp();
                    issue_w(slot, b0, nb, smem_u32(&full[slot]));
                    issue_x(slot, b0, nb, smem_u32(&full[slot]));
                }
                __syncwarp();
            }
        }
    }

    // All ring reads are done (or abandoned).
    __syncthreads();
    const bool aborted = (*abort_flag != 0);
    if (aborted) {
        // Let copies still in flight land before the ring is reused or freed.
        if (warp == 0 && lane == 0) {
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

    // ---- per-warp partials -> red[wk][slot][tok], row pitch kXP (aliases the ring) ----
    float *red = reinterpret_cast<float *>(smem);
    if (warp < C::kNCW && !aborted) {
        const int wk = warp % WK, wr = warp / WK;
        if constexpr (kFma) {
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
                        if (c == 0) red[(wk * kSlots + wr * RT * 16 + g + 4 * i) * kXP + t] = v;
                    }
            } else {
                const int rl = lane % kLR, tl = lane / kLR;
#pragma unroll
                for (int i = 0; i < kRPL; ++i)
#pragma unroll
                    for (int j = 0; j < kTPL; ++j) red[(wk * kSlots + rl + kLR * i) * kXP + tl + kTS * j] = acc_fo[i][j];
            }
        } else {
#pragma unroll
            for (int t = 0; t < RT; ++t)
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    const int s0 = wr * RT * 16 + t * 16 + (lane >> 2);
                    const int t0 = j * 8 + 2 * (lane & 3);
                    float *p0 = red + (wk * kSlots + s0) * kXP + t0;
                    float *p1 = red + (wk * kSlots + s0 + 8) * kXP + t0;
                    float d[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        d[q] = acc_mma[0][t][j][q];
                        if constexpr (kChains == 2) d[q] += acc_mma[kChains - 1][t][j][q];
                    }
                    p0[0] = d[0];
                    p0[1] = d[1];
                    p1[0] = d[2];
                    p1[1] = d[3];
                }
        }
    }
    __syncthreads();

    // Outputs may still be read by the previous kernel on the stream.
    griddep_wait();

    // ---- warp partials added in warp order; single-slice CTAs store here ----
    constexpr bool kBf16Out = (COMPUTE == kMmaBf16 || COMPUTE == kFmaBf16);
    float *stage = red + WK * kSlots * kXP;  // K slices: [owner][row][token], pitch kSP
    float *recv = stage + kSlots * kSP;      // K slices: [slice][my row][token], pitch kSP
    bool stored = false;
    if (!aborted) {
        for (int e = tid; e < kSlots * kXRows; e += C::kThreads) {
            // (chunk layout: consecutive threads on consecutive tokens of one row)
            const int tok = kChunk ? e % kXRows : e / kSlots;
            const int slot = kChunk ? e / kXRows : e % kSlots;
            if (tok >= a.M || slot >= rows_here) continue;
            float v = red[slot * kXP + tok];
#pragma unroll
            for (int q = 1; q < WK; ++q) v += red[(q * kSlots + slot) * kXP + tok];
            if (a.slices == 1) {
                const int n = row0 + slot;
                const int i = split_of(a.splits, n);
                if (NORM && n - a.splits.off[i] < a.norm.cols[i]) {
                    // normalized column: parked in fp32 for the split's last CTA
                    a.norm.vals[a.norm.vals_off[i] + static_cast<int64_t>(tok) * a.norm.cols[i] +
                                (n - a.splits.off[i])] = v;
                    red[slot * kXP + tok] = v;
                } else {
                    store_tok<kBf16Out>(out_row<kBf16Out>(a.splits, n), tok, v);
                    stored = true;
                }
            } else {
                stage[slot * kSP + tok] = v;  // my partial of this row, staged for its owner
            }
        }
    }
    if constexpr (NORM)
        stored |= norm_epilogue<kBf16Out, kSlots, kXP>(a, red, armed + a.ring_stages, row0, rows_here, aborted, tid,
                                                       red + kSlots * kXP,
                                                       static_cast<int>(a.ring_bytes / 4) - kSlots * kXP);

    if (a.slices > 1) {
        // ---- K slices of the cluster added in slice order ----
        // Push model with bulk copies: each CTA has staged its combined partial P[slot][tok]
        // as one contiguous block per owner CTA (owner q holds slots [q * per, (q + 1) * per));
        // one thread copies block q into recv[slice] of CTA q (a copy between cluster
        // shared memories, counted in bytes on q's recv_bar, which has expected all S
        // blocks since the kernel started).  Each owner then adds the S slices of its
        // rows in slice order.  stage and recv sit after the partials in the ring, which
        // every CTA has left once the first cluster barrier is passed; its arrival needs
        // no release ordering (the ring's last reads were consumed before the CTA
        // barrier above, its copies landed before they were waited on).  The staging
        // writes reach the copy engine through the proxy fence and the CTA barrier.
        const int per = kSlots / a.slices;
        const uint32_t block_bytes = static_cast<uint32_t>(per * kSP * 4);
        fence_proxy_async_smem();
        __syncthreads();
        cluster_arrive_relaxed();
        cluster_wait();
        if (tid == 0) {
            const uint32_t recv_local = smem_u32(recv), bar_local = smem_u32(recv_bar), src = smem_u32(stage);
            for (int q = 0; q < a.slices; ++q)
                bulk_s2s_cluster(cluster_map_shared(recv_local + slice * block_bytes, static_cast<uint32_t>(q)),
                                 src + q * block_bytes, block_bytes, cluster_map_shared(bar_local, static_cast<uint32_t>(q)));
        }
        // Every block addressed to this CTA lands before it reads them or exits: the wait
        // is bounded by time only (not cut short by an earlier timeout of this CTA).
        {
            const uint64_t t0 = global_timer_ns();
            bool got = false;
            for (uint32_t it = 0;; ++it) {
                got = mbar_try_wait(smem_u32(recv_bar), 0u);
                if (__all_sync(0xffffffffu, got)) break;
                int give_up = 0;
                if ((it & 7u) == 7u) give_up = (global_timer_ns() - t0 > a.wait_limit_ns) ? 1 : 0;
                if (__shfl_sync(0xffffffffu, give_up, 0)) break;
            }
            if (!got && lane == 0) record_timeout(a.err_word, abort_flag);
        }
        // First half of the closing cluster barrier: my receive buffer is complete, so
        // every copy out of a peer's staging block into mine has landed.  The wait comes
        // last, after the trigger: no CTA leaves while a copy may still read its staging
        // block.  Relaxed: the data moved by copies that complete on mbarriers.
        cluster_arrive_relaxed();
        if (!aborted && *abort_flag == 0) {
            for (int e = tid; e < per * kXRows; e += C::kThreads) {
                const int tok = e / per, rr = e - tok * per;
                const int slot = slice * per + rr;
                if (tok >= a.M || slot >= rows_here) continue;
                float v = recv[rr * kSP + tok];
                for (int q = 1; q < a.slices; ++q) v += recv[(q * per + rr) * kSP + tok];
                store_tok<kBf16Out>(out_row<kBf16Out>(a.splits, row0 + slot), tok, v);
                stored = true;
            }
        }
    }

    // Trigger the dependent launch only after every output store of this CTA is
    // performed: each storing thread fences, then the CTA synchronises.
    if (stored) fence_release_gpu();
    __syncthreads();
    griddep_launch_dependents();
    if (a.slices > 1) cluster_wait();
}

}  // namespace hsp
