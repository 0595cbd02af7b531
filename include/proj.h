/*
 * proj.h -- C ABI of the fused hidden-state projection library (libhsp_proj.so).
 *
 * The operation (TensorRT-LLM PR #20636, "DeepSeek-V4.1 wq_a/wkv via tinygemm2",
 * Description): several projections that read the same hidden state have their
 * weights row-concatenated into one matrix W_cat; one GEMM
 *
 *     Y[M, N_total] = X[M, K] . W_cat[N_total, K]^T        (fp32 accumulate)
 *
 * streams W_cat once, and Y is returned as one dense [M, N_i] output per
 * projection (rows off_i .. off_i + N_i - 1 of W_cat, off_i = N_0 + ... + N_{i-1}).
 * The FP32 variant follows TensorRT-LLM PR #12055 ("Fuse indexer wk +
 * weights_proj into single GEMM in TF32"), Description; the widened four-way
 * split follows TensorRT-LLM PR #8771 ("Fuse QK down_proj with indexer K +
 * weight_proj"), Walkthrough; the single rounding of the FP32 sums follows
 * TensorRT-LLM PR #20502 (GLM-5.2 decode target), glmFusedAGemm commit message.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory and keeps no pointer after the call returns.
 *   - x is [M, K] row-major dense, w_cat is [N_total, K] row-major dense and
 *     outs[i] is [M, N_i] row-major dense.  Element type: bf16 for PROJ_BF16,
 *     fp32 for PROJ_FP32 and PROJ_TF32 (inputs and outputs alike).
 *   - x and w_cat must be 16-byte aligned, every outs[i] aligned to its element
 *     size, and K * element size must be a multiple of 16 bytes (the row pitch of
 *     a tensor copy).  Outputs must not overlap the inputs or each other.
 *   - M == 0 is an empty batch: the call succeeds and touches nothing.
 *   - Host arrays (n_splits, outs, ws, n_rows) are read synchronously, before
 *     the call returns.
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and is
 *     asynchronous; errors found on the host are returned immediately, launch
 *     failures map to PROJ_ERR_CUDA.  No entry point throws or aborts.
 *   - The library never computes on the CPU: there is no fallback path.
 */
#ifndef HSP_PROJ_H
#define HSP_PROJ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (a pointer to the driver's stream object). */
typedef struct CUstream_st *proj_stream_t;

typedef enum {
    PROJ_BF16 = 0, /* x, w, outs bf16; tensor-core products, fp32 accumulate, one RNE rounding */
    PROJ_FP32 = 1, /* x, w, outs fp32; fp32 fused multiply-add on the CUDA cores */
    PROJ_TF32 = 2  /* x, w, outs fp32; operands rounded to tf32 for the tensor cores, fp32 accumulate */
} proj_dtype;

typedef enum {
    PROJ_OK = 0,
    PROJ_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad option value */
    PROJ_ERR_UNSUPPORTED_SHAPE = 2, /* M outside 1..PROJ_MAX_M, splits not summing, K too small ... */
    PROJ_ERR_MISALIGNED = 3,        /* pointer or row pitch not 16-byte aligned */
    PROJ_ERR_UNSUPPORTED_DTYPE = 4,
    PROJ_ERR_DEVICE = 5,            /* current device is not compute capability 10.3 */
    PROJ_ERR_CUDA = 6,              /* a CUDA runtime/driver call failed */
    PROJ_ERR_TIMEOUT = 7            /* a kernel's bounded wait ran out (see proj_check_device_error) */
} proj_status;

#define PROJ_MAX_SPLITS 8
#define PROJ_MAX_M 64
#define PROJ_MAX_PREFETCH 4

/* A global range to bring into L2 (proj_fused_gemm_prefetch). */
typedef struct {
    const void *ptr;  /* device pointer, 16-byte aligned */
    uint64_t bytes;   /* a multiple of 16 */
} proj_prefetch_range;

/* Process-wide options (proj_set_options).  Zero-initialised = defaults. */
typedef struct {
    /* 1 (default): launch with programmatic stream serialization, so the kernel's
     * weight loads overlap the tail of the previous kernel on the stream; the
     * activations are read only after griddepcontrol.wait, and the completion
     * trigger is issued after the last output store (TensorRT-LLM PR #20636,
     * Description, discusses the hazard of triggering before the stores).
     * 0: plain stream-ordered launches.  -1 in a set call = leave unchanged. */
    int32_t pdl;
    /* Limit of every in-kernel wait on a shared-memory barrier, in microseconds.
     * 0 = default (1,000,000 us).  When a wait runs out the kernel records
     * PROJ_ERR_TIMEOUT in a device error word, skips its stores and returns. */
    int32_t wait_limit_us;
    /* Test hook, 0 = off.  When > 0, the weight stream of every CTA leaves out
     * its stage number (value - 1), so its consumers' waits run out: used only
     * to test the timeout path (in the register-ring and register GEMV kernels,
     * stage 0 is the token copy).  Never faults: nothing is read or written out of
     * bounds and every wait is bounded. */
    int32_t skip_stage_plus1;
    /* Kernel for bf16 with 9 <= M <= 64: 0 (default) and 2 = the tensor-memory kernel
     * (tcgen05.mma into TMEM); 1 = the streaming mma.sync kernel (the one that also
     * serves M <= 8, tf32 and fp32).  For PROJ_TF32 at every M: 0 (default) and 1 = the
     * streaming kernel, 2 = the tensor-memory kernel (kind::tf32; slower on GB300 for
     * the pages' tf32 shapes).  All give results within tolerance; each is bitwise
     * self-consistent (fused = separate, run to run). */
    int32_t large_m_path;
    /* 1: the tensor-memory kernel first prefetches each CTA's weight rows into L2 as
     * contiguous runs.  0 (default): no prefetch (measured slower on GB300). */
    int32_t l2_prefetch;
    /* 0 (default): the dependent launch is triggered after every output store is
     * performed.  1: it is triggered at kernel start, before any output store (the order
     * TensorRT-LLM PR #20636, Description, describes for tinygemm2).  Correct only when
     * every kernel launched after this one with programmatic stream serialization calls
     * griddepcontrol.wait before it reads the outputs (all of this library's kernels
     * do); a dependent that reads without waiting can see stale values, which the PDL
     * ordering test uses as its positive control.  Measured on GB300 with back-to-back
     * calls: 0.7-1.5 us less per call (wq_a++wkv M = 8: 5.45 -> 4.60 us). */
    int32_t trigger_early;
    /* bf16 with M <= 2: 0 (default) = mma.sync like 3 <= M <= 8; 1 = fp32 FMA on the
     * CUDA cores.  Both within tolerance, each bitwise self-consistent. */
    int32_t small_m_path;
    /* Register kernels.  bf16, M <= 8 and K a multiple of 64: 0 (default) = the
     * register-ring kernel (sixteen warps load the weights straight into registers, the
     * tokens arrive as one tensor copy) when a row has at most 80 k-units of 128 bytes
     * (K <= 5120), the streaming kernel otherwise; 2 = the register-ring kernel up to 128
     * k-units (K <= 8192).  PROJ_FP32 with K <= 8192: 0 = the register GEMV kernel (a CTA
     * owns a slab of rows and all of K, no K slices) when the M tokens fit one CTA (at
     * most 8 and M * K * 4 <= 192 KB), the streaming kernel otherwise; 2 = the register
     * GEMV kernel up to M = 64, the tokens in groups that fit, one group per CTA along
     * grid.y (slower than the streaming kernel on GB300 at most such M).
     * 1 = the streaming kernel for both.  All within tolerance, each bitwise
     * self-consistent (fused = separate, run to run, graph = eager). */
    int32_t reg_path;
} proj_options;

/* Kernel geometry chosen for one launch (proj_describe_plan). */
typedef struct {
    int32_t bucket;        /* 0: M <= 8, 1: 9 <= M <= 32, 2: 33 <= M <= 64 */
    int32_t compute;       /* 0 bf16 tensor cores, 1 tf32 tensor cores, 2 fp32 FMA, 3 bf16 data with fp32 FMA */
    int32_t rows_per_cta;  /* R: output rows owned by one CTA */
    int32_t row_ctas;      /* CTAs along the rows (grid.x) */
    int32_t slices;        /* S: K slices = CTAs per cluster (grid.y) */
    int32_t k_warps;       /* WK: warps sharing one row tile, each on its own k boxes */
    int32_t row_warps;     /* WR */
    int32_t row_tiles;     /* RT: 16-row MMA tiles per warp */
    int32_t token_tiles;   /* MT: 8-token tiles */
    int32_t ring_stages;   /* shared-memory ring depth */
    int32_t stage_bytes;
    int32_t smem_bytes;    /* dynamic shared memory per CTA */
    int32_t k_per_stage;   /* elements of K per ring stage */
    int32_t stages_total;  /* ring stages of one K slice */
    int32_t threads;       /* threads per CTA (consumer warps + 1 producer warp) */
    int32_t units_per_slice; /* 128-byte k-units per K slice (fixes the summation order with k_warps) */
    int32_t engine;          /* 0 streaming mma.sync / FMA kernel, 1 tensor-memory (tcgen05) kernel,
                              * 2 register-ring kernel (bf16, M <= 8: ring_stages = k-units in flight per
                              * warp, stages_total = k-units per warp, stage_bytes = 0),
                              * 3 fp32 register GEMV (M <= 64: ring_stages = row blocks in flight,
                              * stages_total = row blocks of two rows, token_tiles = token groups
                              * along grid.y, stage_bytes = 0) */
    int32_t tensor_copies;   /* streaming kernel: 1 = one 3-D tensor copy per stage for the weights
                              * and one for the tokens (rows a multiple of 128 bytes), 0 = one 1-D
                              * bulk copy per row and stage (any other K); register-ring kernel: 1
                              * (the tokens arrive as one tensor copy) */
    int32_t reserved[2];
} proj_plan_info;

/*
 * proj_fused_gemm -- the fused projection (TensorRT-LLM PR #20636, Description: the
 * two projections become one GEMM over the row-concatenated weight; here for any M in
 * 1..PROJ_MAX_M).  One kernel launch streams every row of w_cat
 * once and writes outs[i][m * n_splits[i] + r] = round(sum_k x[m,k] * w_cat[off_i + r, k]).
 *   x          device [M, K]
 *   w_cat      device [N_total, K], N_total = sum(n_splits)
 *   n_splits   host   [num_splits], each >= 1
 *   num_splits 1..PROJ_MAX_SPLITS
 *   outs       host array of num_splits device pointers, outs[i] is [M, n_splits[i]]
 *   M          1..PROJ_MAX_M tokens;  K >= 1
 * The result of every output row depends only on (x, its weight row, M's bucket,
 * K, dtype): it is bitwise identical to proj_separate_gemm, run to run, and under
 * CUDA-graph replay.
 */
proj_status proj_fused_gemm(const void *x, const void *w_cat, const int32_t *n_splits,
                            int32_t num_splits, void *const *outs, int32_t M, int32_t K,
                            proj_dtype dtype, proj_stream_t stream);

/*
 * proj_fused_gemm_prefetch -- proj_fused_gemm that also prefetches up to
 * PROJ_MAX_PREFETCH caller-named global ranges into L2 (TensorRT-LLM PR #20502,
 * glmFusedAGemm commit message: ahead of its grid-dependency wait, the GLM fused-A
 * kernel has its CTAs share out 16 KB L2 bulk prefetches of as many as four caller
 * tensors, the weights the step's following kernels will need; here the streaming
 * kernel issues them right after its own copies).  The ranges are only read as a hint:
 * the outputs are bitwise those of proj_fused_gemm.  Ranges must stay allocated
 * until the call has completed on the stream.
 */
proj_status proj_fused_gemm_prefetch(const void *x, const void *w_cat, const int32_t *n_splits,
                                     int32_t num_splits, void *const *outs, int32_t M, int32_t K,
                                     proj_dtype dtype, const proj_prefetch_range *ranges,
                                     int32_t num_ranges, proj_stream_t stream);

/*
 * proj_fused_gemm_rmsnorm -- proj_fused_gemm followed, in the same kernel, by the
 * RMSNorm its consumers apply (TensorRT-LLM PR #20636, Description: the q_norm /
 * kv_norm RMSNorms read the wq_a / wkv outputs; PR #20502, glm_mla_kv_half_append
 * commit message: the kv_a_proj output's 512 latent columns, not its RoPE part, are
 * normalised).
 * For split i with c = norm_cols[i] > 0, every token m and r < c:
 *     outs[i][m, r] = round(y[m, r] / sqrt(mean_{j < c} y[m, j]^2 + eps) * gammas[i][r])
 * with y the fp32 sums of the projection (one rounding per output); columns r >= c,
 * and splits with norm_cols[i] == 0, are the plain projection, bitwise those of
 * proj_fused_gemm.
 *   norm_cols  host [num_splits], each in [0, n_splits[i]]
 *   gammas     host array of num_splits device pointers; gammas[i] is [norm_cols[i]]
 *              of the data type (may be NULL where norm_cols[i] == 0)
 *   eps        finite, >= 0
 *   workspace  device, 16-byte aligned, at least proj_rmsnorm_workspace_bytes(...)
 *              bytes, owned by the caller.  Zero it once before its first use; every
 *              call, one that reported PROJ_ERR_TIMEOUT included, leaves it ready for
 *              the next (its counters back at zero).  Calls that share a workspace
 *              must not overlap on the GPU.
 * PROJ_BF16 with 1 <= M <= 8 only (PROJ_ERR_UNSUPPORTED_DTYPE / _SHAPE otherwise).
 * Bitwise identical run to run and under CUDA-graph replay.
 */
proj_status proj_fused_gemm_rmsnorm(const void *x, const void *w_cat, const int32_t *n_splits,
                                    int32_t num_splits, const int32_t *norm_cols,
                                    const void *const *gammas, float eps, void *const *outs,
                                    int32_t M, int32_t K, proj_dtype dtype, void *workspace,
                                    size_t workspace_bytes, proj_stream_t stream);

/* Workspace bytes proj_fused_gemm_rmsnorm needs for this shape (host only; 0 when the
 * shape is not supported, with proj_last_error_string saying why). */
size_t proj_rmsnorm_workspace_bytes(int32_t M, int32_t K, const int32_t *n_splits,
                                    int32_t num_splits, const int32_t *norm_cols,
                                    proj_dtype dtype);

/*
 * proj_fused_gemm_rmsnorm_static -- proj_fused_gemm_rmsnorm for callers that cannot
 * allocate device memory.  The pages have no counterpart; it exists for callers
 * that have no workspace to pass: code under an inference runtime that owns all
 * device memory through its own pool and forbids side allocations, plugins that
 * receive only the tensors of one operation, and latency-critical paths where
 * cudaMalloc's implicit device synchronisation is not acceptable.  It allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library call): the workspace is
 * a fixed 1 MiB array compiled into this library, present in the memory of every GPU
 * that loads it until the process exits.  The caller still passes inputs and outputs,
 * with the meaning and limits of proj_fused_gemm_rmsnorm.
 *   - The first call made in a context looks up the array's device address there
 *     (cudaGetSymbolAddress); make that first call before any stream capture.  A
 *     device reset (cudaDeviceReset) or another context on the device gives the array
 *     a new address, which the next call in that context looks up again (so that call,
 *     too, belongs outside a capture).
 *   - Every call shares the one array and finds the last call's contents in it.  The
 *     part that must start at zero (the arrival counters) is zero when the library is
 *     loaded, and every call, one that reported PROJ_ERR_TIMEOUT included, leaves it at
 *     zero; nothing is cleared per call, so a call is one kernel launch, chained to the
 *     previous kernel on the stream like proj_fused_gemm_rmsnorm.  Calls that overlap
 *     on the GPU race on the array: issue them on one stream, or order them.
 *   - Shapes whose workspace (proj_rmsnorm_workspace_bytes) exceeds 1 MiB are refused
 *     with PROJ_ERR_UNSUPPORTED_SHAPE and a message that gives both sizes.
 */
proj_status proj_fused_gemm_rmsnorm_static(const void *x, const void *w_cat, const int32_t *n_splits,
                                           int32_t num_splits, const int32_t *norm_cols,
                                           const void *const *gammas, float eps, void *const *outs,
                                           int32_t M, int32_t K, proj_dtype dtype, proj_stream_t stream);

/*
 * proj_fused_gemm_host -- proj_fused_gemm for a caller whose tokens and results live in
 * host memory (a decode step that receives the hidden state from the host and hands the
 * projections back to it).  Enqueued on `stream`, in this order: x_host copied into
 * x_dev (M * K elements), the fused projection from x_dev into outs_dev (exactly
 * proj_fused_gemm: same kernel, same bits), one device-to-host copy of each outs_dev[i]
 * into outs_host[i].  When x_host is page-locked memory that the device can address
 * (cudaHostAlloc memory under unified addressing), the token copy is a small staging
 * kernel that reads it over the host link, launched with programmatic dependent launch
 * like the projection (2 kernel launches per call); otherwise it is one host-to-device
 * cudaMemcpyAsync.  An outs_host[i] in such memory is likewise written by the kernel
 * directly, and outs_dev[i] is left untouched.  The call returns once everything is
 * enqueued; synchronise the stream before reading outs_host, and do not change x_host
 * before the stream has passed the call.
 *   x_host     host [M, K]; page-locked (cudaHostAlloc / pinned) for the copies to be
 *              asynchronous, pageable memory makes the copy synchronous
 *   outs_host  host array of num_splits host pointers, outs_host[i] is [M, N_i]
 *   x_dev      device [M, K] staging buffer, 16-byte aligned, owned by the caller
 *   outs_dev   host array of num_splits device pointers, outs_dev[i] is [M, N_i]
 * Other arguments, limits and errors as proj_fused_gemm; a failed copy returns
 * PROJ_ERR_CUDA.  The library allocates nothing: both staging buffers are the caller's.
 */
proj_status proj_fused_gemm_host(const void *x_host, const void *w_cat, const int32_t *n_splits,
                                 int32_t num_splits, void *const *outs_host, int32_t M, int32_t K,
                                 proj_dtype dtype, void *x_dev, void *const *outs_dev,
                                 proj_stream_t stream);

/*
 * Host plans -- proj_fused_gemm_host bound once to fixed buffers and recorded as one CUDA
 * graph (the token copy, the fused projection, the device-to-host copies), so
 * that a loop repeating the step (decode) costs one graph launch per step on the host.
 * proj_host_plan_create takes the arguments of proj_fused_gemm_host (x_host and every
 * outs_host[i] must be page-locked: the recording refuses pageable memory with
 * PROJ_ERR_CUDA) and records the work with the options in force at that moment (PDL,
 * engine switches).  The buffers must stay allocated until the plan is destroyed.
 * proj_host_plan_launch enqueues one step on `stream` (same bits as proj_fused_gemm);
 * synchronise the stream before reading the host outputs.  proj_host_plan_destroy
 * releases the graph; NULL is accepted.  The plan is host state only: no device memory
 * is allocated by the library.  A plan may be launched from one thread at a time.
 * Cost: a plan step is slower on the GPU than calling proj_fused_gemm_host directly
 * (measured on GB300 at wq_a++wkv M = 8: 13.3-14.9 us against 6.7-6.9 us per step in a
 * loop on one stream), because a graph launch costs more than the two kernel launches it
 * replaces and consecutive graph launches are not chained by programmatic dependent
 * launch.  Prefer the direct call in a loop; a plan only saves host-side argument work.
 */
typedef struct proj_host_plan proj_host_plan;

proj_status proj_host_plan_create(const void *x_host, const void *w_cat, const int32_t *n_splits,
                                  int32_t num_splits, void *const *outs_host, int32_t M, int32_t K,
                                  proj_dtype dtype, void *x_dev, void *const *outs_dev,
                                  proj_host_plan **plan);
proj_status proj_host_plan_launch(proj_host_plan *plan, proj_stream_t stream);
proj_status proj_host_plan_destroy(proj_host_plan *plan);

/*
 * proj_separate_gemm -- one launch per projection over its row range of the same
 * w_cat (TensorRT-LLM PR #20636, Description: "2-8 tokens: one tinygemm2 per
 * projection").  Same arguments and outputs as proj_fused_gemm, bitwise equal to it.
 */
proj_status proj_separate_gemm(const void *x, const void *w_cat, const int32_t *n_splits,
                               int32_t num_splits, void *const *outs, int32_t M, int32_t K,
                               proj_dtype dtype, proj_stream_t stream);

/*
 * proj_pack_weights -- build W_cat by copying the projection weights one after
 * another (TensorRT-LLM PR #20636, Description: post_load_weights copies wq_a and
 * wkv into one row-concatenated tensor and rebinds the per-projection weights as
 * views of it).  ws[i] is a device [n_rows[i], K] dense matrix; w_cat receives them
 * in order, rows [sum_{j<i} n_rows[j], sum_{j<=i} n_rows[j]).
 *   ws       host array of num device pointers, each 16-byte aligned (may be NULL
 *            where n_rows[i] == 0)
 *   n_rows   host [num], each >= 0 (a part of 0 rows copies nothing)
 *   num      1..PROJ_MAX_SPLITS
 *   K        elements per row; K * element size must be a multiple of 16 bytes
 *            (PROJ_ERR_MISALIGNED otherwise, like the projection calls)
 *   w_cat    device, 16-byte aligned, owned by the caller and at least
 *            sum(n_rows) * K elements long: the library cannot check the size of
 *            the caller's buffer, so a shorter one is overrun
 * One copy kernel enqueued on `stream` (none when every part is skipped), without
 * programmatic dependent launch: it starts after earlier work on the stream and a
 * projection call enqueued after it reads the new weights.  Re-running it into the
 * same w_cat refreshes the weights in place (a checkpoint reload).  A ws[i] that is
 * exactly its own rows of w_cat (already packed, or a view written through) is
 * skipped; a ws[i] that overlaps w_cat anywhere else is refused with
 * PROJ_ERR_INVALID_ARG before anything is enqueued.
 */
proj_status proj_pack_weights(const void *const *ws, const int32_t *n_rows, int32_t num,
                              int32_t K, proj_dtype dtype, void *w_cat, proj_stream_t stream);

/*
 * proj_pack_check -- 1 if `w` is exactly the view of rows [row_off, row_off + n_rows)
 * of w_cat (so a reload through `w` updates the fused weight; TensorRT-LLM PR
 * #20636, Description: a replaced Parameter is no longer a view), else 0.
 * Pure pointer arithmetic on the host.
 */
int proj_pack_check(const void *w, const void *w_cat, int64_t row_off, int32_t n_rows,
                    int32_t n_total, int32_t K, proj_dtype dtype);

/*
 * proj_supported -- host-side query: 1 if (M, K, n_total, dtype) is served,
 * 0 otherwise (the shape gate; TensorRT-LLM PR #20502, dense-MLP and fused-A
 * commit messages: a host query answers whether the kernels serve a shape).
 */
int proj_supported(int32_t M, int32_t K, int32_t n_total, proj_dtype dtype);

/* proj_describe_plan -- the geometry a launch over n_rows rows would use (host only). */
proj_status proj_describe_plan(int32_t M, int32_t K, int32_t n_rows, proj_dtype dtype,
                               proj_plan_info *info);

proj_status proj_set_options(const proj_options *opt);
proj_status proj_get_options(proj_options *opt);

/*
 * proj_check_device_error -- synchronizes `stream`, then reads and clears the
 * device error word of the current device.  Returns PROJ_ERR_TIMEOUT if any
 * kernel since the last check gave up a bounded wait, PROJ_ERR_CUDA if the
 * stream reported an error, else PROJ_OK.
 */
proj_status proj_check_device_error(proj_stream_t stream);

/* Number of kernels this library has launched in the process (all devices). */
uint64_t proj_launch_count(void);

/* Message of the last error returned on the calling thread ("" if none). */
const char *proj_last_error_string(void);

/* Library version string. */
const char *proj_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HSP_PROJ_H */
