// stream_args.h -- launch arguments shared by the host planner and the kernels.
#pragma once

#include <stdint.h>

namespace hsp {

enum Compute : int { kMmaBf16 = 0, kMmaTf32 = 1, kFmaFp32 = 2 };

constexpr int kMaxSplits = 8;
constexpr int kDeviceErrTimeout = 7;  // same value as PROJ_ERR_TIMEOUT

// Output scatter: row n of the launch (0-based in its weight map) belongs to
// split i with off[i] <= n < off[i] + rows[i]; element (token t, row n) goes to
// out[i][t * rows[i] + (n - off[i])].
struct SplitTable {
    int32_t count;
    int32_t off[kMaxSplits];
    int32_t rows[kMaxSplits];
    void *out[kMaxSplits];
};

struct StreamArgs {
    int32_t n_rows;            // rows of the launch's weight map
    int32_t rows_per_cta;      // R (the W box height)
    int32_t M;                 // tokens
    int32_t kboxes;            // ceil(K / box width)
    int32_t stages_total;      // ceil(kboxes / WK)
    int32_t stages_per_slice;  // stages owned by one K slice
    int32_t ring_stages;       // shared-memory ring depth
    int32_t slices;            // S (cluster size along grid.y)
    uint32_t stage_bytes;      // WK * (w_box_bytes + x_box_bytes)
    uint32_t w_box_bytes;      // shared footprint of one W box (row slots * 128)
    uint32_t x_box_bytes;      // 8 * MT * 128
    uint32_t w_tx_bytes;       // bytes one W box delivers (R * 128)
    uint32_t x_tx_bytes;       // bytes one X box delivers (8 * MT * 128)
    uint32_t ring_bytes;       // ring_stages * stage_bytes, at least the reduction buffer
    int32_t skip_stage;        // test hook: this global stage is never loaded (-1: off)
    int32_t pad_;
    uint64_t wait_limit_ns;    // bound of every barrier wait
    int *err_word;             // device error word (PROJ_ERR_TIMEOUT on expiry)
    SplitTable splits;
};

}  // namespace hsp
