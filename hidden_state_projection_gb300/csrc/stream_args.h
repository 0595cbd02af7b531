// stream_args.h -- launch arguments shared by the host planner and the kernels.
#pragma once

#include <stdint.h>

namespace hsp {

enum Compute : int { kMmaBf16 = 0, kMmaTf32 = 1, kFmaFp32 = 2, kFmaBf16 = 3 };

constexpr int kMaxSplits = 8;
constexpr int kDeviceErrTimeout = 7;  // same value as PROJ_ERR_TIMEOUT
constexpr int kUnitBytes = 128;       // one k-unit: 128 bytes of a row (64 bf16 or 32 fp32)
constexpr int kMaxPrefetch = 4;       // caller tensors prefetched into L2 by one call
constexpr uint32_t kPrefetchChunk = 16384;

// Global ranges a call prefetches into L2 for later kernels (16-byte aligned,
// sizes multiples of 16), cut into 16 KB chunks spread over the CTAs.
struct PrefetchList {
    int32_t count;
    const char *ptr[kMaxPrefetch];
    uint64_t bytes[kMaxPrefetch];
};

// Output scatter: row n of the launch (0-based in its weight rows) belongs to
// split i with off[i] <= n < off[i] + rows[i]; element (token t, row n) goes to
// out[i][t * rows[i] + (n - off[i])].
struct SplitTable {
    int32_t count;
    int32_t off[kMaxSplits];
    int32_t rows[kMaxSplits];
    void *out[kMaxSplits];
};

// RMSNorm epilogue (q_norm / kv_norm of the projections' consumers): split i's
// first cols[i] columns are normalized per token, y * rsqrt(mean(y^2) + eps) * gamma,
// from the fp32 sums, and rounded once.  The mean spans CTAs, so the CTAs meeting a
// normalized split park their fp32 values and per-token sums of squares in a
// workspace; the last of them to arrive (an arrival counter per split) adds the sums
// in CTA order, normalizes every value of the split and stores it, then clears the
// counter.  Single-slice (S = 1) launches only.
struct NormArgs {
    int32_t active;                 // 1: some split is normalized
    float eps;
    int32_t cols[kMaxSplits];       // normalized leading columns of split i (0: none)
    const void *gamma[kMaxSplits];  // [cols[i]] elements of the data type
    int64_t vals_off[kMaxSplits];   // float offset of split i's [M][cols[i]] block in vals
    int32_t part_off[kMaxSplits];   // float offset of split i's [cta_count[i]][M] block in partial
    int32_t cta_first[kMaxSplits];  // first CTA (grid.x index) holding a normalized row of split i
    int32_t cta_count[kMaxSplits];  // CTAs holding normalized rows of split i
    float *vals;                    // workspace
    float *partial;                 // workspace
    unsigned *counter;              // workspace: [kMaxSplits] arrivals, [kMaxSplits] abort flags; zero between calls
};

// K is cut into units of 128 bytes.  Unit u is summed by warp (u mod WK) of the
// CTA that owns its K slice (slice s holds units [s*units_per_slice, ...)); a
// ring stage carries stage_units consecutive units of every row of the CTA and
// of every token.  Only the unit -> warp -> slice map decides the summation
// order; the stage width, the row count and the stage layout do not.
//
// Two stage layouts, one per copy engine use:
//   tensor (rows a multiple of 128 bytes): one 3-D tensor copy per stage for the
//     weights and one for the tokens, each a box [stage_units][rows][128 bytes]
//     with the 128-byte swizzle (16-byte chunk c of line L stored at c ^ (L mod 8));
//     the token box starts x_off bytes (a multiple of 1024) after the weight box.
//     (fp32 FMA above 8 tokens: one weight box [R][128 bytes] per unit, unit k at
//     k * slots lines, and token boxes of 8 * MT rows, the rows past M zero-filled);
//   bulk (any other K): one 1-D bulk copy per row and stage, rows at `pitch`
//     (16 mod 128) bytes; the token rows start x_off = R * pitch after the weights.
struct StreamArgs {
    const char *w;             // first weight row of the launch, [n_rows, K] row-major
    const char *x;             // activations, [M, K] row-major
    int64_t row_bytes;         // K * element size (a multiple of 16)
    int32_t n_rows;            // rows of the launch
    int32_t rows_per_cta;      // R
    int32_t M;                 // tokens
    int32_t units_total;       // ceil(row_bytes / 128)
    int32_t units_per_slice;   // units of one K slice
    int32_t stage_units;       // units per ring stage
    int32_t stages_per_slice;  // ceil(units_per_slice / stage_units)
    int32_t ring_stages;       // shared-memory ring depth
    int32_t slices;            // S (cluster size along grid.y)
    uint32_t pitch;            // bulk layout: shared-memory row pitch (stage_units*128 + 16)
    uint32_t stage_bytes;      // bytes of one stage (weights + tokens)
    uint32_t ring_bytes;       // ring_stages * stage_bytes, at least the reduction buffer
    uint32_t x_off;            // bytes from a stage's start to its first token row
    int32_t skip_stage;        // test hook: this stage of every slice is never loaded (-1: off)
    int32_t trigger_early;     // option: trigger dependents at kernel start (default: after the stores)
    uint64_t wait_limit_ns;    // bound of every barrier wait
    int *err_word;             // device error word (PROJ_ERR_TIMEOUT on expiry)
    SplitTable splits;
    PrefetchList prefetch;
    NormArgs norm;
};

// Tensor-memory path (9 <= M <= 64): a CTA owns a 128-row weight tile and one
// K slice of `kb_per_slice` 128-byte k-blocks; the S slices of a row tile form a
// cluster and add their partials in slice order.
struct UmmaArgs {
    const char *w;             // first weight row of the launch (for the L2 prefetch)
    int64_t row_bytes;         // K * element size
    int32_t n_rows;            // rows of the launch
    int32_t M;                 // tokens
    int32_t kb_total;          // ceil(row_bytes / 128)
    int32_t kb_per_slice;      // k-blocks of one K slice
    int32_t slices;            // S (cluster size along grid.y)
    int32_t ring_stages;
    uint32_t stage_bytes;      // weight boxes (tile rows * 128 per k-block) + x_box_bytes, a multiple of 1024
    uint32_t x_box_bytes;      // token rows (16, 32 or 64) * 128 per k-block of the stage
    int32_t prefetch_l2;       // 1: bulk-prefetch the CTA's weight segments into L2 first
    int32_t skip_stage;        // test hook: this k-block of every slice is never loaded (-1: off)
    int32_t trigger_early;     // option: trigger dependents at kernel start (default: after the stores)
    int32_t kb_per_stage;      // k-blocks per ring stage: 1 (2-D boxes) or 2 (one 3-D box each of weights and tokens)
    uint64_t wait_limit_ns;
    int *err_word;
    SplitTable splits;
    PrefetchList prefetch;
};

}  // namespace hsp
