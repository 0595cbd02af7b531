// proj_api.cu -- the C ABI (include/proj.h): validation, the M-bucketed planner,
// the weight packer and the launch wrapper.
//
// Dispatch (TensorRT-LLM PR #20636, Description: one fused call at one token,
// one call per projection at 2-8 tokens, a different GEMM above): here every M in
// 1..64 has both a fused and a per-projection entry point, and M picks the
// kernel geometry:
//   bucket 0, M <= 8      : 1 token tile;  warps split K 8 ways, no K slices
//   bucket 1, 9 <= M <= 32: 2 or 4 token tiles; 2 row warps x 4 K warps, S K slices
//   bucket 2, 33 <= M <= 64: 8 token tiles; 2 row warps x 4 K warps, S K slices
// bf16 with M <= 8 and rows of at most 80 k-units of 128 bytes (K <= 5120) runs the
// register-ring kernel instead (sixteen warps split K, weights straight into
// registers), and fp32 with M <= 8 the register GEMV kernel (no K slices), both
// measured faster on GB300 there.
// The K-split (warps WK, slices S, box width) is a function of (K, dtype,
// bucket) only, so an output row is summed in the same order whatever the
// number of rows in the launch -- the property that makes the fused and the
// separate calls bitwise equal.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "proj.h"
#include "stream_args.h"

namespace {

using hsp::LaunchReq;
using hsp::StreamArgs;

constexpr int kSmemLimit = 232448;          // per-block dynamic shared memory on sm_103
constexpr int kUmmaSmemBudget = 110 * 1024;  // tensor-memory kernel: ring + receive buffer, two CTAs per SM
constexpr int kUmmaTrioSmemBudget = 74 * 1024;  // the same at three CTAs per SM
constexpr int kSmemReserve = 1024 + 1024;   // ring alignment slack (1024 for the swizzle) + barriers + flags
constexpr int kStageWeightBytes = 65536;    // tensor layout: weight bytes per ring stage
constexpr int kMaxRingStages = 32;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

thread_local char g_last_error[512] = "";
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_opt_pdl{1};
std::atomic<int> g_opt_wait_us{0};
std::atomic<int> g_opt_skip_stage_plus1{0};
std::atomic<int> g_opt_large_m_path{0};
std::atomic<int> g_opt_l2_prefetch{0};
std::atomic<int> g_opt_trigger_early{0};
std::atomic<int> g_opt_small_m_path{0};
std::atomic<int> g_opt_reg_path{0};

}  // namespace

// Device error word: a kernel whose bounded wait runs out stores PROJ_ERR_TIMEOUT here.
__device__ int g_hsp_device_error;

namespace hsp {
// Sets the text proj_last_error_string returns (for entry points in other files).
proj_status set_last_error(proj_status st, const char *msg) {
    snprintf(g_last_error, sizeof g_last_error, "%s", msg);
    return st;
}
}  // namespace hsp

namespace {

proj_status fail(proj_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
proj_status fail(proj_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

proj_status ok() {
    g_last_error[0] = '\0';
    return PROJ_OK;
}

proj_status cuda_fail(cudaError_t e, const char *what) {
    return fail(PROJ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_size(proj_dtype dt) { return dt == PROJ_BF16 ? 2 : 4; }

bool dtype_valid(int dt) { return dt == PROJ_BF16 || dt == PROJ_FP32 || dt == PROJ_TF32; }

// ---- per-device facts ------------------------------------------------------

struct DeviceInfo {
    int sms = 0;
    int cc_ok = 0;
    int *err_word = nullptr;
    int cluster_ctas[17] = {0};  // CTAs co-resident in clusters of 1, 2, 4, 8, 16 (index = size)
    int pair_ctas[17] = {0};     // the same at two CTAs per SM (the tensor-memory kernel's footprint)
    int trio_ctas[17] = {0};     // and at three (its 64-row tiles at 9-32 tokens)
};

// Stand-in kernel for the co-residency query.  Default shape: the streaming kernels,
// one CTA of 288 threads and ~200 KB of shared memory per SM.
__global__ void hsp_cluster_probe_kernel(int *p) {
    if (p && threadIdx.x == 0x7fffffff) p[0] = 1;
}

int co_resident_ctas(int cluster, int fallback, int threads = 288, int smem = 200 * 1024) {
    if (cluster > 8 &&
        cudaFuncSetAttribute(hsp_cluster_probe_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        (void)cudaGetLastError();
        return fallback;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, static_cast<unsigned>(cluster * 16), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = static_cast<unsigned>(cluster);
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(hsp_cluster_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, hsp_cluster_probe_kernel, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return fallback;
    }
    return n * cluster;
}

std::mutex g_dev_mu;
DeviceInfo g_dev[64];
bool g_dev_ready[64] = {};
uint64_t g_dev_ctx[64] = {};  // context the entry of g_dev was made in

}  // namespace

namespace hsp {
// Unique id of the CUDA context current on the calling thread, 0 when none is current
// (or the driver cannot tell).  Device addresses of this library's __device__ symbols
// belong to one context: a reset device (cudaDeviceReset) or another context on the
// same device gets new ones, so every per-device cache of such an address is keyed by
// this id as well.
uint64_t current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
        } else {
            (void)cudaGetLastError();
        }
    });
    if (!get_cur || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_cur(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? static_cast<uint64_t>(id) : 0;
}
}  // namespace hsp

namespace {

proj_status device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PROJ_ERR_DEVICE, "device ordinal %d out of range", dev);
    // No current context yet (first call, or right after a reset) counts as a change:
    // the lookup below creates it, and the entry is then tagged with its id.
    const uint64_t ctx = hsp::current_context_id();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ready[dev] || ctx == 0 || ctx != g_dev_ctx[dev]) {
        DeviceInfo d;
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.cc_ok = (major == 10 && minor == 3);
        d.cluster_ctas[1] = d.sms;
        if (d.cc_ok) {
            d.cluster_ctas[2] = co_resident_ctas(2, d.sms);
            d.cluster_ctas[4] = co_resident_ctas(4, d.sms);
            d.cluster_ctas[8] = co_resident_ctas(8, d.sms * 3 / 4);
            d.cluster_ctas[16] = co_resident_ctas(16, d.sms * 2 / 3);
            for (int c = 1; c <= 16; c *= 2) {
                d.pair_ctas[c] = co_resident_ctas(c, d.cluster_ctas[c], hsp::kUmmaThreadsHost, kUmmaSmemBudget);
                d.trio_ctas[c] = co_resident_ctas(c, d.pair_ctas[c], hsp::kUmmaThreadsHost, kUmmaTrioSmemBudget);
            }
            void *p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_hsp_device_error)) != cudaSuccess)
                return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
            d.err_word = static_cast<int *>(p);
        }
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
        g_dev_ctx[dev] = hsp::current_context_id();
    }
    *out = g_dev[dev];
    if (!out->cc_ok)
        return fail(PROJ_ERR_DEVICE, "device %d is not compute capability 10.3 (GB300, sm_103a)", dev);
    return PROJ_OK;
}

// ---- planner -----------------------------------------------------------------

struct Plan {
    proj_plan_info info;
    int compute, bucket, MT, RT, WR, WK, S, R, grid_x;
    int units_total, units_per_slice, stage_units, stages_per_slice, ring_stages;
    int tensor;  // 3-D tensor copies (rows a multiple of 128 bytes) or 1-D bulk copies
    int chunk;   // fp32 FMA above 8 tokens: K warps on 16-byte chunks of every unit
    int pitch, stage_bytes, x_off, ring_bytes, smem;
};

int ceil_div(int a, int b) { return (a + b - 1) / b; }

proj_status check_shape(int32_t M, int32_t K, int64_t n_total, int dt) {
    if (!dtype_valid(dt)) return fail(PROJ_ERR_UNSUPPORTED_DTYPE, "dtype %d is not PROJ_BF16/FP32/TF32", dt);
    if (M < 0 || K < 0 || n_total < 0) return fail(PROJ_ERR_INVALID_ARG, "negative size (M=%d K=%d N=%lld)", M, K, (long long)n_total);
    if (M > PROJ_MAX_M) return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "M=%d exceeds %d tokens", M, PROJ_MAX_M);
    if (K == 0) return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "K must be at least 1");
    if ((static_cast<int64_t>(K) * elem_size(static_cast<proj_dtype>(dt))) % 16 != 0)
        return fail(PROJ_ERR_MISALIGNED, "row pitch K*%d bytes (K=%d) is not a multiple of 16", elem_size(static_cast<proj_dtype>(dt)), K);
    if (n_total > (int64_t(1) << 30) || K > (1 << 24))
        return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "N_total=%lld or K=%d too large", (long long)n_total, K);
    return PROJ_OK;
}

// Geometry of one launch over n_rows weight rows.
//   - bucket, WK, S and units_per_slice depend on (M's bucket, K, dtype) only:
//     they fix which warp and which K slice sums every 128-byte unit of K, hence
//     the summation order of every output;
//   - R (rows per CTA) spreads the rows over the SMs.  With tensor copies (rows a
//     multiple of 128 bytes) a stage holds ~16 KB of weights, so the compute left
//     after the last byte lands is short; with bulk copies the stage width is the
//     widest that still leaves two ring stages in shared memory (long contiguous
//     row segments per copy).  Neither changes the order.
void make_plan(int M, int K, int n_rows, proj_dtype dt, const int *cluster_ctas, Plan *p) {
    memset(p, 0, sizeof *p);
    const int esz = elem_size(dt);
    p->compute = dt == PROJ_BF16 ? hsp::kMmaBf16 : (dt == PROJ_TF32 ? hsp::kMmaTf32 : hsp::kFmaFp32);
    // Opt-in for one or two tokens: fp32 FMA on the CUDA cores instead of an
    // 8-token-wide mma.sync (measured slower on GB300: 8.4 vs 6.4 us for wq_a++wkv M=1).
    if (dt == PROJ_BF16 && M <= 2 && g_opt_small_m_path.load() == 1) p->compute = hsp::kFmaBf16;
    p->bucket = M <= 8 ? 0 : (M <= 32 ? 1 : 2);
    // Bucket 2 splits K four ways like bucket 1: with 4 row warps x 2 K warps the
    // indexer's 192 rows (28 per CTA) left half the warps without rows (measured on
    // GB300, indexer M = 64: fp32 14.6 -> 14.4 us, tf32 9.9 -> 9.5 us).
    static const int WRs[3] = {1, 2, 2}, WKs[3] = {8, 4, 4};
    // fp32 FMA above 8 tokens: eight K warps, each on one 16-byte chunk of every unit,
    // over all row slots of the CTA (balanced for any unit count; measured on GB300,
    // the FMA loop on a resident stage went from ~53% to ~70% of the FMA pipe at 64
    // tokens and from ~34% to ~56% at 16)
    const bool chunk = p->compute == hsp::kFmaFp32 && p->bucket > 0;
    p->chunk = chunk;
    p->WR = chunk ? 1 : WRs[p->bucket];
    p->WK = chunk ? 8 : WKs[p->bucket];
    p->MT = p->bucket == 0 ? 1 : (p->bucket == 2 ? 8 : (M <= 16 ? 2 : 4));
    const int64_t row_bytes = static_cast<int64_t>(K) * esz;
    p->units_total = static_cast<int>((row_bytes + hsp::kUnitBytes - 1) / hsp::kUnitBytes);
    // K slices (clusters) only for the larger token buckets, where one CTA's
    // token rows of X would not fit next to a useful weight stage otherwise.
    const int per_warp = ceil_div(p->units_total, p->WK);
    p->S = 1;
    if (p->bucket > 0 && esz == 4 && p->units_total >= 128) {
        // fp32 rows of 16 KB and more with many tokens: every row tile re-reads its K
        // slice of all token rows, so slices must be short -- sixteen of them (tf32 at
        // 9-32 tokens: eight, its mma.sync products leave the reduction the larger part;
        // measured on GB300, indexer M = 9 / 16 / 32 5.47 / 5.59 / 7.00 -> 5.34 / 5.45 /
        // 6.65 us, router M = 16 6.30 -> 6.02; fp32 FMA stays faster with sixteen)
        p->S = (dt == PROJ_TF32 && p->bucket == 1) ? 8 : 16;
    } else if (p->bucket > 0) {
        if (per_warp >= 16) p->S = 4;
        else if (per_warp >= 4) p->S = 2;
    } else if (esz == 4 && per_warp >= 16) {
        // fp32 rows are twice as long: few rows per CTA would leave most SMs idle and
        // long per-warp chains; eight K slices per row instead (fixed per K and dtype;
        // measured on GB300 against four: tf32 indexer M = 1 / 4 / 8 5.17 / 5.18 / 5.41 ->
        // 4.89 / 4.89 / 5.11 us, fp32 indexer M = 7 / 8 6.84 / 6.88 -> 6.01 / 6.03; two
        // and sixteen were slower)
        p->S = 8;
    }
    // Units per slice: a multiple of WK when that leaves no slice empty (balanced
    // warps), else the plain share.  S stays a power of two (it must divide the
    // CTA's row slots for the cluster reduction).
    auto slice_units = [&](int S) {
        const int plain = ceil_div(p->units_total, S);
        if (chunk) return plain;  // every warp has a chunk of every unit already
        const int rounded = ceil_div(plain, p->WK) * p->WK;
        return (S - 1) * rounded < p->units_total ? rounded : plain;
    };
    p->units_per_slice = slice_units(p->S);
    while (p->S > 1 && (p->S - 1) * p->units_per_slice >= p->units_total) {  // no empty slice
        p->S /= 2;
        p->units_per_slice = slice_units(p->S);
    }
    // (the chunk layout: up to four 16-row tiles, three at 33-64 tokens -- the lane's
    // register tile is (slots / 4) x 8 there, 12 x 8 at three tiles; measured on GB300,
    // router 256 x 6144 at M = 33 / 48 / 64: 18.95 / 19.13 / 19.61 us with two tiles (its
    // CTAs in two waves) -> 13.82 / 13.96 / 14.40 with three; the indexer keeps two)
    const int max_rows = chunk ? (p->MT == 8 ? 48 : 64) : p->WR * 2 * 16;
    // rows per CTA: spread over the CTAs that can be resident at once (clusters of
    // S leave some SMs of a GPC idle)
    const int resident = cluster_ctas[p->S] > 0 ? cluster_ctas[p->S] : cluster_ctas[1];
    p->R = ceil_div(n_rows * p->S, resident);
    if (p->R < 1) p->R = 1;
    if (p->R > max_rows) p->R = max_rows;
    p->RT = chunk ? ceil_div(p->R, 16) : (p->R > p->WR * 16 ? 2 : 1);
    const int slots = p->WR * p->RT * 16;
    p->grid_x = ceil_div(n_rows, p->R);
    // partial sums of the warps
    // (rows of 8 * MT + 1 floats, padded against bank conflicts), plus (K slices) the
    // staging and receive blocks of the cluster reduction (rows of 8 * MT + 4 floats)
    // (chunk layout: rows of 8 * MT + 32 / row lanes floats, its lanes' tiles write
    // conflict-free)
    const int xp = chunk ? 8 * p->MT + (p->MT == 8 ? 8 : 4) : 8 * p->MT + 1;
    const int red_bytes = p->WK * slots * xp * 4 + (p->S > 1 ? 2 * slots * (8 * p->MT + 4) * 4 : 0);
    const int budget = kSmemLimit - kSmemReserve;
    const int Us = p->units_per_slice;
    p->tensor = (row_bytes % hsp::kUnitBytes) == 0;
    if (p->tensor) {
        // Stages of su units, su dividing the slice (no box reaches into the next
        // slice), a multiple of WK where possible (every warp gets the same share),
        // holding about kStageWeightBytes of weights.  One weight box and one token
        // box per stage, each rounded up to 1024 bytes.
        auto box = [](int rows, int su) { return ceil_div(rows * su * hsp::kUnitBytes, 1024) * 1024; };
        // The chunk layout keeps every unit's weight rows kSlots lines apart (one box per
        // unit) and its token rows 8 * MT lines apart (rows past M zero-filled).
        auto wbox_bytes = [&](int su) { return chunk ? su * slots * hsp::kUnitBytes : box(p->R, su); };
        auto xbox_bytes = [&](int su) { return chunk ? su * 8 * p->MT * hsp::kUnitBytes : box(M, su); };
        auto choose = [&](int stage_weight_bytes) {
            const int target = std::max(1, stage_weight_bytes / (p->R * hsp::kUnitBytes));
            // the divisor of the slice nearest the target (the larger one on a tie), at
            // most half the slice: at least two stages, so loads and products overlap
            int su = 0;
            for (int d = 1; d <= std::max(1, Us / 2); ++d)
                if (Us % d == 0 && (su == 0 || std::abs(d - target) <= std::abs(su - target))) su = d;
            for (;;) {
                const int stage = wbox_bytes(su) + xbox_bytes(su);
                const int nst = ceil_div(Us, su);
                int ring = std::min(std::min(nst, budget / stage), kMaxRingStages);
                if (ring >= std::min(2, nst) || su == 1) {
                    p->stage_units = su;
                    p->stages_per_slice = nst;
                    p->ring_stages = ring;
                    p->pitch = 0;
                    p->stage_bytes = stage;
                    p->x_off = wbox_bytes(su);
                    return;
                }
                int d = su - 1;  // next smaller divisor of the slice
                while (d > 1 && Us % d != 0) --d;
                su = d;
            }
        };
        choose(kStageWeightBytes);
        // When the token rows of a stage crowd the ring down to fewer than three of
        // several stages (M = 8 at hidden 6144 / 7168), half-size stages keep more of
        // the slice in flight: measured on GB300, qk_indexer M = 8 8.93 -> 8.55 us,
        // glm_fused_a M = 8 9.53 -> 9.15 us; at M = 1 the 64 KB stages stay faster.
        // The stage width does not enter the summation order.
        if (p->ring_stages < 3 && p->stages_per_slice > p->ring_stages) choose(kStageWeightBytes / 2);
    } else {
        const int first = Us >= 2 * p->WK ? 2 : 1;
        for (int nst = first; nst <= Us; ++nst) {
            int su = ceil_div(Us, nst);
            if (su > p->WK) su = ceil_div(su, p->WK) * p->WK;
            const int n_eff = ceil_div(Us, su);
            const int pitch = su * hsp::kUnitBytes + 16;
            const int stage = (p->R + M) * pitch;
            int ring = budget / stage;
            if (ring > n_eff) ring = n_eff;
            if (ring > kMaxRingStages) ring = kMaxRingStages;
            if (ring >= (n_eff >= 2 ? 2 : 1)) {
                p->stage_units = su;
                p->stages_per_slice = n_eff;
                p->ring_stages = ring;
                p->pitch = pitch;
                p->stage_bytes = stage;
                p->x_off = p->R * pitch;
                break;
            }
        }
    }
    p->ring_bytes = p->ring_stages * p->stage_bytes;
    if (p->ring_bytes < red_bytes) p->ring_bytes = red_bytes;
    p->ring_bytes = ceil_div(p->ring_bytes, 128) * 128;
    // ring, full/empty barriers, receive barrier, abort flag, armed[ring], RMSNorm flags[8], slack
    p->smem = 1024 + p->ring_bytes + 2 * p->ring_stages * 8 + 8 + 8 + 4 * p->ring_stages + 4 * hsp::kMaxSplits + 64;
    proj_plan_info &i = p->info;
    i.bucket = p->bucket;
    i.compute = p->compute;
    i.rows_per_cta = p->R;
    i.row_ctas = p->grid_x;
    i.slices = p->S;
    i.k_warps = p->WK;
    i.row_warps = p->WR;
    i.row_tiles = p->RT;
    i.token_tiles = p->MT;
    i.ring_stages = p->ring_stages;
    i.stage_bytes = p->stage_bytes;
    i.smem_bytes = p->smem;
    i.k_per_stage = p->stage_units * hsp::kUnitBytes / esz;
    i.stages_total = p->stages_per_slice;
    i.threads = hsp::kThreadsPerCta;
    i.units_per_slice = p->units_per_slice;
    i.tensor_copies = p->tensor;
}

// ---- tensor maps (tensor-memory kernel only) ---------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

struct MapEntry {
    uint64_t ptr;
    int rank, dtype;
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    bool used;
    CUtensorMap map;
};
constexpr int kMapCache = 256;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

// Tiled tensor map (128-byte swizzle, zero fill past the tensor), cached per
// (pointer, shape, box).  dims[0] is the innermost extent in elements; strides[i]
// is the byte stride of dimension i + 1.
proj_status encode_map(const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                       proj_dtype dt, CUtensorMap *out) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            (void)cudaGetLastError();
    });
    if (!g_encode) return fail(PROJ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    MapEntry key{};
    key.ptr = reinterpret_cast<uint64_t>(ptr);
    key.rank = rank;
    key.dtype = static_cast<int>(dt);
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides[i];
    }
    auto same = [&](const MapEntry &m) {
        if (!m.used || m.ptr != key.ptr || m.rank != key.rank || m.dtype != key.dtype) return false;
        for (int i = 0; i < rank; ++i) {
            if (m.dims[i] != key.dims[i] || m.box[i] != key.box[i]) return false;
            if (i + 1 < rank && m.strides[i] != key.strides[i]) return false;
        }
        return true;
    };
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        for (int i = 0; i < kMapCache; ++i)
            if (same(g_maps[i])) {
                *out = g_maps[i].map;
                return PROJ_OK;
            }
    }
    CUtensorMap map;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = g_encode(&map, dt == PROJ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), d, st, b, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PROJ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): rank %d, dims [%llu %llu %llu], box [%u %u %u]",
                    static_cast<int>(r), rank, (unsigned long long)d[0], (unsigned long long)(rank > 1 ? d[1] : 0),
                    (unsigned long long)(rank > 2 ? d[2] : 0), b[0], rank > 1 ? b[1] : 0u, rank > 2 ? b[2] : 0u);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        key.used = true;
        key.map = map;
        g_maps[g_map_next] = key;
        g_map_next = (g_map_next + 1) % kMapCache;
    }
    *out = map;
    return PROJ_OK;
}

// 2-D map of a row-major [d1, d0] tensor, box [box1, box0].
proj_status encode_map(const void *ptr, uint64_t d0, uint64_t d1, uint32_t box0, uint32_t box1, proj_dtype dt,
                       CUtensorMap *out) {
    const uint64_t dims[2] = {d0, d1};
    const uint64_t strides[1] = {d0 * static_cast<uint64_t>(elem_size(dt))};
    const uint32_t box[2] = {box0, box1};
    return encode_map(ptr, 2, dims, strides, box, dt, out);
}

// ---- tensor-memory plan ----------------------------------------------------

// bf16 with 9 <= M <= 64: the tensor-memory kernel.  Measured on GB300 (µs, streaming /
// tensor memory with its first 128-row tiles): qk_indexer M = 9 / 12 / 16: 10.2 / 10.9,
// 10.7 / 10.9, 11.0 / 10.9; wq_a++wkv: 8.1 / 8.8, 8.3 / 8.8, 8.5 / 8.8; glm_fused_a (2752
// rows): 16.7 / 10.6, 18.0 / 10.6, 18.6 / 10.6 -- the streaming kernel's 64-row CTAs over
// four K slices need 172 CTAs, a second wave.  The tensor-memory kernel has no such cliff,
// and its 64-row tiles with two-k-block stages since took qk_indexer M = 12 / 16 to 9.33 /
// 9.35, wq_a++wkv M = 16 to 7.47 and glm_fused_a M = 9 / 16 to 8.88 / 8.90, so it takes
// every M >= 9; option large_m_path 1 / 2 forces one of them.
constexpr int kStreamMaxM = 8;
// PROJ_TF32 runs the tensor-memory kernel (kind::tf32, the fp32 operands read as tf32)
// only when large_m_path is 2.  Measured on GB300 (µs, streaming mma.sync / tcgen05 over
// 16 K slices): indexer 192 x 7168 at M = 1 / 4 / 16 / 64: 5.37 / 9.12, 5.60 / 9.61,
// 5.91 / 9.61, 9.48 / 9.90; router 256 x 6144 at M = 1 / 4 / 16: 5.54 / 9.07, 5.58 /
// 9.09, 6.40 / 9.07.  So the streaming kernel stays the default at every M.
bool use_umma(int M, proj_dtype dt) {
    const int o = g_opt_large_m_path.load();
    if (dt == PROJ_TF32) return o == 2;
    if (M <= 8 || dt != PROJ_BF16) return false;
    return o == 2 || (o == 0 && M > kStreamMaxM);
}

struct UPlan {
    proj_plan_info info;
    int compute, NT, S, TR, kb_total, kb_per_slice, tiles, ring, stage_bytes, x_box, smem, G;
};

// K slices and k-blocks per slice depend on (K, dtype) only (the summation order).  The
// ring is sized so that two CTAs fit on an SM (the next call's CTAs start beside this
// call's last ones).  The tile height, the MMA's M, does not change any output bit
// (tested): 64 weight rows when all the 64-row tiles times the slices fit one wave at two
// CTAs per SM (pair_ctas), or at three when the 64-row plan's shared memory allows three
// (trio_ctas: 16 or 32 tokens; measured on GB300, glm_fused_a 2752 x 6144 at M = 9 / 16 /
// 32 9.61 / 9.60 / 9.97 -> 8.88 / 8.90 / 9.34 us, the 2784-row cell at M = 16 9.79 ->
// 9.08), else 128.  Measured on GB300 (µs, 128-row / 64-row tiles with
// two-k-block stages, 8 slices): qk_indexer M = 12 / 16 / 24 / 32: 9.87 / 9.87 / 10.31 /
// 10.32 -> 9.33 / 9.35 / 9.80 / 9.82, wq_a++wkv M = 16 / 32 7.93 / 8.21 -> 7.47 / 7.71; at
// 64 tokens 64-row tiles won from the start (qk_indexer 13.8 -> 12.1 with one-k-block
// stages).  Four slices with 64-row tiles and one CTA per SM (36 clusters of 4 fill 144
// SMs) were slower: 14.8 - 15.7 µs for qk_indexer at every M.
void make_umma_plan(int M, int K, int n_rows, proj_dtype dt, const int *pair_ctas, const int *trio_ctas, UPlan *p) {
    memset(p, 0, sizeof *p);
    const int64_t row_bytes = static_cast<int64_t>(K) * elem_size(dt);
    p->compute = dt == PROJ_BF16 ? hsp::kMmaBf16 : hsp::kMmaTf32;
    p->NT = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    p->kb_total = static_cast<int>((row_bytes + 127) / 128);
    p->S = p->kb_total >= 64 ? 8 : (p->kb_total >= 32 ? 4 : (p->kb_total >= 8 ? 2 : 1));
    // tf32 rows are twice as long in bytes; their projections (the indexer's 192 rows,
    // the router's 256) have few rows: sixteen slices of the long rows give the grid
    // enough CTAs.  A function of (K, dtype) only, like every slice count.
    if (dt == PROJ_TF32 && p->kb_total >= 128) p->S = 16;
    p->kb_per_slice = ceil_div(p->kb_total, p->S);
    while (p->S > 1 && (p->S - 1) * p->kb_per_slice >= p->kb_total) {
        --p->S;
        p->kb_per_slice = ceil_div(p->kb_total, p->S);
    }
    const int wave2 = pair_ctas[p->S] > 0 ? pair_ctas[p->S] : pair_ctas[1];
    const int wave3 = trio_ctas[p->S] > 0 ? trio_ctas[p->S] : wave2;
    const int tiles64 = ceil_div(n_rows, 64) * p->S;
    // Stage shape, ring and shared memory for tiles of TR weight rows.
    auto size_for = [&](int TR) {
        p->TR = TR;
        p->tiles = ceil_div(n_rows, p->TR);
        // Two k-blocks per stage (one 3-D box of weights, 256 contiguous bytes of each row,
        // and one of tokens) for the 64-row tiles: measured on GB300, qk_indexer M = 64
        // 10.95 -> 10.37 us, wq_a++wkv M = 64 8.75 -> 8.21 (with 128-row tiles at 16-32
        // tokens it was mixed, qk_indexer M = 32 10.08 -> 10.34).  Only where rows are whole
        // k-blocks and the slices' and the total k-block counts are even: no stage then
        // reaches past its slice or adds a zero-filled k-block, so the products and their
        // order, hence every output bit, are those of one k-block per stage.
        p->G = (p->TR == 64 && row_bytes % 128 == 0 && p->kb_total % 2 == 0 && p->kb_per_slice % 2 == 0) ? 2 : 1;
        p->x_box = p->G * p->NT * 128;
        p->stage_bytes = p->G * p->TR * 128 + p->x_box;
        // receive buffer of the cluster reduction (dedicated); the staging buffer aliases
        // the ring.  Two CTAs per SM: ring + receive buffer within ~110 KB (64-row tiles
        // at 16 or 32 tokens stay under 74 KB, three per SM).
        const int red_bytes = p->TR * (p->NT + 4) * 4;
        const int recv_bytes = p->S > 1 ? red_bytes : 0;
        int ring = (kUmmaSmemBudget - recv_bytes) / p->stage_bytes;
        // 64-row tiles: four k-blocks in flight (four one-k-block stages or two of two)
        // rather than all that fit (measured on GB300 with one-k-block stages, qk_indexer
        // M = 33 / 48 / 64 10.99 / 10.98 / 11.18 -> 10.69 / 10.70 / 10.92 us, wq_a++wkv M = 64
        // 8.93 -> 8.71; with two-k-block stages at 16 / 32 tokens, two stages against the four
        // or five that fit: qk_indexer 10.29 / 10.03 -> 9.35 / 9.82).  The ring depth does not
        // change any output bit.
        if (p->TR == 64 && ring > 4 / p->G) ring = 4 / p->G;
        if (ring < 2) ring = 2;
        const int stages = p->kb_per_slice / p->G;
        if (ring > stages) ring = stages < 2 ? 2 : stages;
        while (p->S > 1 && ring * p->stage_bytes < red_bytes) ++ring;
        p->ring = ring;
        p->smem = 1024 + ring * p->stage_bytes + recv_bytes + (2 * ring + 2) * 8 + 16 + 64;
    };
    size_for(64);
    if (tiles64 > wave2 && (p->smem > kUmmaTrioSmemBudget || tiles64 > wave3)) size_for(128);
    proj_plan_info &i = p->info;
    i.bucket = M <= 8 ? 0 : (M <= 32 ? 1 : 2);
    i.compute = p->compute;
    i.rows_per_cta = p->TR;
    i.row_ctas = p->tiles;
    i.slices = p->S;
    i.k_warps = 1;
    i.row_warps = 4;
    i.row_tiles = 1;
    i.token_tiles = p->NT / 8;
    i.ring_stages = p->ring;
    i.stage_bytes = p->stage_bytes;
    i.smem_bytes = p->smem;
    i.k_per_stage = p->G * 128 / elem_size(dt);
    i.stages_total = p->kb_per_slice / p->G;
    i.threads = hsp::kUmmaThreadsHost;
    i.units_per_slice = p->kb_per_slice;
    i.engine = 1;
}

proj_status launch_umma_rows(const DeviceInfo &dev, const void *x, const void *w, int n_rows, int M, int K,
                             proj_dtype dt, const hsp::SplitTable &splits, const hsp::PrefetchList &pf,
                             cudaStream_t stream) {
    UPlan p;
    make_umma_plan(M, K, n_rows, dt, dev.pair_ctas, dev.trio_ctas, &p);
    hsp::UmmaLaunchReq r{};
    const uint32_t boxk = 128u / static_cast<uint32_t>(elem_size(dt));
    proj_status st;
    if (p.G == 2) {
        // [k-blocks][rows][128 bytes] (row stride row_bytes, k-block stride 128 bytes),
        // boxes [2][tile rows or token tile][128 bytes]
        const uint64_t rb = static_cast<uint64_t>(K) * elem_size(dt);
        const uint64_t strides[2] = {rb, 128u};
        const uint64_t wdims[3] = {boxk, static_cast<uint64_t>(n_rows), static_cast<uint64_t>(p.kb_total)};
        const uint64_t xdims[3] = {boxk, static_cast<uint64_t>(M), static_cast<uint64_t>(p.kb_total)};
        const uint32_t wbox[3] = {boxk, static_cast<uint32_t>(p.TR), 2u};
        const uint32_t xbox[3] = {boxk, static_cast<uint32_t>(p.NT), 2u};
        st = encode_map(w, 3, wdims, strides, wbox, dt, &r.tmap_w);
        if (st != PROJ_OK) return st;
        st = encode_map(x, 3, xdims, strides, xbox, dt, &r.tmap_x);
        if (st != PROJ_OK) return st;
    } else {
        st = encode_map(w, static_cast<uint64_t>(K), static_cast<uint64_t>(n_rows), boxk, static_cast<uint32_t>(p.TR), dt,
                        &r.tmap_w);
        if (st != PROJ_OK) return st;
        st = encode_map(x, static_cast<uint64_t>(K), static_cast<uint64_t>(M), boxk, static_cast<uint32_t>(p.NT), dt,
                        &r.tmap_x);
        if (st != PROJ_OK) return st;
    }
    r.compute = p.compute;
    r.NT = p.NT;
    r.grid = dim3(static_cast<unsigned>(p.tiles), static_cast<unsigned>(p.S), 1);
    r.smem_bytes = p.smem;
    r.pdl = g_opt_pdl.load();
    r.stream = stream;
    hsp::UmmaArgs &a = r.args;
    a.w = static_cast<const char *>(w);
    a.row_bytes = static_cast<int64_t>(K) * elem_size(dt);
    a.n_rows = n_rows;
    a.M = M;
    a.kb_total = p.kb_total;
    a.kb_per_slice = p.kb_per_slice;
    a.slices = p.S;
    a.ring_stages = p.ring;
    a.stage_bytes = static_cast<uint32_t>(p.stage_bytes);
    a.x_box_bytes = static_cast<uint32_t>(p.x_box);
    a.kb_per_stage = p.G;
    a.prefetch_l2 = g_opt_l2_prefetch.load();
    a.trigger_early = g_opt_trigger_early.load();
    a.skip_stage = g_opt_skip_stage_plus1.load() - 1;
    const int wus = g_opt_wait_us.load();
    a.wait_limit_ns = wus > 0 ? static_cast<uint64_t>(wus) * 1000ull : kDefaultWaitNs;
    a.err_word = dev.err_word;
    a.splits = splits;
    a.prefetch = pf;
    cudaError_t e = hsp::launch_umma(r);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch (tensor-memory path)");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PROJ_OK;
}

// ---- register-ring plan (bf16, M <= 8) -------------------------------------

// The register-ring kernel serves bf16 with M <= 8 when a row is a whole number of
// 128-byte k-units and, by default, at most kRegAutoUnits of them: then the sixteen
// warps hold a CTA's whole share of the weights in flight at once (measured on GB300,
// wq_a++wkv K = 5120: 5.41 / 5.62 / 5.76 us at M = 1 / 4 / 8 against 6.10 / 6.10 /
// 6.18 us for the streaming kernel; at K = 7168 it is no faster).  Option reg_path 1
// turns it off, 2 uses it up to kRegMaxUnits.  The choice depends on (M, K, dtype)
// only, so fused and per-projection launches run the same kernel.
constexpr int kRegAutoUnits = 80;
constexpr int kRegMaxUnits = 128;

bool use_reg(int M, int K, proj_dtype dt) {
    if (dt != PROJ_BF16 || M < 1 || M > 8) return false;
    const int64_t row_bytes = static_cast<int64_t>(K) * 2;
    if (row_bytes % hsp::kUnitBytes != 0) return false;
    const int o = g_opt_reg_path.load();
    if (o == 1) return false;
    if (M <= 2 && g_opt_small_m_path.load() == 1) return false;  // the opt-in CUDA-core path
    return row_bytes / hsp::kUnitBytes <= (o == 2 ? kRegMaxUnits : kRegAutoUnits);
}

struct RegPlan {
    int R, grid, units, smem;
};

void make_reg_plan(int M, int K, int n_rows, int sms, RegPlan *p) {
    p->units = static_cast<int>(static_cast<int64_t>(K) * 2 / hsp::kUnitBytes);
    p->R = std::min(16, std::max(1, ceil_div(n_rows, std::max(1, sms))));
    p->grid = ceil_div(n_rows, p->R);
    p->smem = p->units * M * hsp::kUnitBytes + 1024;
}

void reg_plan_info(int M, int K, const RegPlan &p, proj_plan_info *i) {
    memset(i, 0, sizeof *i);
    i->bucket = 0;
    i->compute = hsp::kMmaBf16;
    i->rows_per_cta = p.R;
    i->row_ctas = p.grid;
    i->slices = 1;
    i->k_warps = 16;
    i->row_warps = 1;
    i->row_tiles = 1;
    i->token_tiles = 1;
    i->ring_stages = hsp::kRegDepthHost;  // k-units in flight per warp
    i->stage_bytes = 0;
    i->smem_bytes = p.smem;
    i->k_per_stage = hsp::kUnitBytes / 2;
    i->stages_total = ceil_div(p.units, 16);  // k-units per warp
    i->threads = hsp::kRegThreadsHost;
    i->units_per_slice = p.units;
    i->engine = 2;
    i->tensor_copies = 1;  // the tokens arrive as one tensor copy
    (void)M;
    (void)K;
}

proj_status launch_reg_rows(const DeviceInfo &dev, const void *x, const void *w, int n_rows, int M, int K,
                            const hsp::SplitTable &splits, const hsp::PrefetchList &pf, cudaStream_t stream,
                            const hsp::NormArgs *norm) {
    RegPlan p;
    make_reg_plan(M, K, n_rows, dev.sms, &p);
    hsp::RegLaunchReq r{};
    // tokens as [units][M][128 bytes] (row stride row_bytes, unit stride 128 bytes), one box
    const uint64_t row_bytes = static_cast<uint64_t>(K) * 2;
    const uint64_t xdims[3] = {64u, static_cast<uint64_t>(M), static_cast<uint64_t>(p.units)};
    const uint64_t strides[2] = {row_bytes, 128u};
    const uint32_t xbox[3] = {64u, static_cast<uint32_t>(M), static_cast<uint32_t>(p.units)};
    proj_status st = encode_map(x, 3, xdims, strides, xbox, PROJ_BF16, &r.tmap_x);
    if (st != PROJ_OK) return st;
    r.grid = dim3(static_cast<unsigned>(p.grid), 1, 1);
    r.smem_bytes = p.smem;
    r.pdl = g_opt_pdl.load();
    r.stream = stream;
    StreamArgs &a = r.args;
    a.w = static_cast<const char *>(w);
    a.x = static_cast<const char *>(x);
    a.row_bytes = static_cast<int64_t>(row_bytes);
    a.n_rows = n_rows;
    a.rows_per_cta = p.R;
    a.M = M;
    a.units_total = p.units;
    a.units_per_slice = p.units;
    a.slices = 1;
    a.skip_stage = g_opt_skip_stage_plus1.load() - 1;
    a.trigger_early = g_opt_trigger_early.load();
    const int wus = g_opt_wait_us.load();
    a.wait_limit_ns = wus > 0 ? static_cast<uint64_t>(wus) * 1000ull : kDefaultWaitNs;
    a.err_word = dev.err_word;
    a.splits = splits;
    a.prefetch = pf;
    if (norm) a.norm = *norm;
    cudaError_t e = hsp::launch_reg(r);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch (register-ring path)");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PROJ_OK;
}

// ---- fp32 register GEMV plan (PROJ_FP32) ---------------------------------------

// Tokens one GEMV CTA holds in shared memory: at most 8, within 192 KB.
int gemv_group_cap(int K) {
    const int64_t cap = hsp::kGemvMaxTokenBytes / (static_cast<int64_t>(K) * 4);
    return static_cast<int>(std::min<int64_t>(8, cap));
}

// PROJ_FP32 with K <= 8192 and at most gemv_group_cap(K) tokens runs the register GEMV
// kernel: one CTA per slab of rows and all of K, no clusters (measured on GB300: indexer
// wk ++ weights_proj 192 x 7168 and the GLM router 256 x 6144; numbers in the design
// notes).  Option reg_path 2 also sends more tokens (up to 64) to it, cut into token
// groups along grid.y: every group's CTAs read all of their tokens and their rows'
// weights again, and on GB300 that lost to the streaming kernel's K slices at every
// M > 8 but one (so it is not the default).  Option reg_path 1 turns the kernel off.
// The choice depends on (M, K, dtype) only.
bool use_gemv(int M, int K, proj_dtype dt) {
    if (dt != PROJ_FP32 || M < 1 || M > 64 || K > 8192) return false;
    const int path = g_opt_reg_path.load();
    if (path == 1) return false;
    const int cap = gemv_group_cap(K);
    return cap >= 1 && (M <= cap || path == 2);
}

struct GemvPlan {
    int R, grid, groups, group_tokens, smem;
};

// Token groups: G = ceil(M / cap), each of ceil(M / G) tokens (so no group is empty);
// row slabs: as many as fit beside G groups in one wave of one CTA per SM.
void make_gemv_plan(int M, int K, int n_rows, int sms, GemvPlan *p) {
    const int cap = std::max(1, gemv_group_cap(K));
    p->groups = ceil_div(M, cap);
    p->group_tokens = ceil_div(M, p->groups);
    const int slabs = std::max(1, std::max(1, sms) / p->groups);
    p->R = std::max(1, ceil_div(n_rows, slabs));
    p->grid = ceil_div(n_rows, p->R);
    p->smem = p->group_tokens * K * 4;
}

void gemv_plan_info(int M, int K, const GemvPlan &p, proj_plan_info *i) {
    memset(i, 0, sizeof *i);
    i->bucket = M <= 8 ? 0 : (M <= 32 ? 1 : 2);
    i->compute = hsp::kFmaFp32;
    i->rows_per_cta = p.R;
    i->row_ctas = p.grid;
    i->slices = 1;
    i->k_warps = 16;
    i->row_warps = 1;
    i->row_tiles = 1;
    i->token_tiles = p.groups;  // token groups (grid.y)
    i->ring_stages = 2;  // row blocks in flight
    i->stage_bytes = 0;
    i->smem_bytes = p.smem;
    i->k_per_stage = K;
    i->stages_total = ceil_div(p.R, 2);  // row blocks of two rows
    i->threads = hsp::kGemvThreadsHost;
    i->units_per_slice = ceil_div(K * 4, hsp::kUnitBytes);
    i->engine = 3;
    i->tensor_copies = 0;  // the tokens arrive as one 1-D bulk copy
    (void)M;
}

proj_status launch_gemv_rows(const DeviceInfo &dev, const void *x, const void *w, int n_rows, int M, int K,
                             const hsp::SplitTable &splits, const hsp::PrefetchList &pf, cudaStream_t stream) {
    GemvPlan p;
    make_gemv_plan(M, K, n_rows, dev.sms, &p);
    hsp::GemvLaunchReq r{};
    r.grid = dim3(static_cast<unsigned>(p.grid), static_cast<unsigned>(p.groups), 1);
    r.smem_bytes = p.smem;
    r.pdl = g_opt_pdl.load();
    r.stream = stream;
    StreamArgs &a = r.args;
    a.w = static_cast<const char *>(w);
    a.x = static_cast<const char *>(x);
    a.row_bytes = static_cast<int64_t>(K) * 4;
    a.n_rows = n_rows;
    a.rows_per_cta = p.R;
    a.M = M;
    a.units_total = ceil_div(K * 4, hsp::kUnitBytes);
    a.units_per_slice = a.units_total;
    a.slices = 1;
    a.skip_stage = g_opt_skip_stage_plus1.load() - 1;
    a.trigger_early = g_opt_trigger_early.load();
    const int wus = g_opt_wait_us.load();
    a.wait_limit_ns = wus > 0 ? static_cast<uint64_t>(wus) * 1000ull : kDefaultWaitNs;
    a.err_word = dev.err_word;
    a.splits = splits;
    a.prefetch = pf;
    cudaError_t e = hsp::launch_gemv(r);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch (fp32 register GEMV path)");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PROJ_OK;
}

// One launch over `n_rows` weight rows starting at `w` (already offset to the first row).
proj_status launch_rows(const DeviceInfo &dev, const void *x, const void *w, int n_rows, int M, int K,
                        proj_dtype dt, const hsp::SplitTable &splits, const hsp::PrefetchList &pf,
                        cudaStream_t stream, const hsp::NormArgs *norm = nullptr) {
    if (use_umma(M, dt)) return launch_umma_rows(dev, x, w, n_rows, M, K, dt, splits, pf, stream);
    if (use_reg(M, K, dt)) return launch_reg_rows(dev, x, w, n_rows, M, K, splits, pf, stream, norm);
    if (use_gemv(M, K, dt)) return launch_gemv_rows(dev, x, w, n_rows, M, K, splits, pf, stream);
    Plan p;
    make_plan(M, K, n_rows, dt, dev.cluster_ctas, &p);
    if (p.ring_stages < 1 || p.smem > kSmemLimit)
        return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "no shared-memory plan for M=%d K=%d rows=%d", M, K, n_rows);
    LaunchReq r{};
    if (p.tensor) {
        // weights as [units][rows][128 bytes] (row stride row_bytes, unit stride 128
        // bytes), one box [stage units][R][128 bytes] per stage; tokens likewise
        const uint64_t ke = 128u / static_cast<uint64_t>(elem_size(dt));
        const uint64_t row_bytes = static_cast<uint64_t>(K) * elem_size(dt);
        const uint64_t wdims[3] = {ke, static_cast<uint64_t>(n_rows), static_cast<uint64_t>(p.units_total)};
        const uint64_t xdims[3] = {ke, static_cast<uint64_t>(M), static_cast<uint64_t>(p.units_total)};
        const uint64_t strides[2] = {row_bytes, 128u};
        // (chunk layout: one weight box per unit, token boxes 8 * MT rows high)
        const uint32_t wbox[3] = {static_cast<uint32_t>(ke), static_cast<uint32_t>(p.R),
                                  static_cast<uint32_t>(p.chunk ? 1 : p.stage_units)};
        const uint32_t xbox[3] = {static_cast<uint32_t>(ke), static_cast<uint32_t>(p.chunk ? 8 * p.MT : M),
                                  static_cast<uint32_t>(p.stage_units)};
        proj_status st = encode_map(w, 3, wdims, strides, wbox, dt, &r.tmap_w);
        if (st != PROJ_OK) return st;
        st = encode_map(x, 3, xdims, strides, xbox, dt, &r.tmap_x);
        if (st != PROJ_OK) return st;
    }
    r.tensor = p.tensor;
    r.compute = p.compute;
    r.bucket = p.bucket;
    r.MT = p.MT;
    r.RT = p.RT;
    r.grid = dim3(static_cast<unsigned>(p.grid_x), static_cast<unsigned>(p.S), 1);
    r.smem_bytes = p.smem;
    r.pdl = g_opt_pdl.load();
    r.stream = stream;
    StreamArgs &a = r.args;
    a.w = static_cast<const char *>(w);
    a.x = static_cast<const char *>(x);
    a.row_bytes = static_cast<int64_t>(K) * elem_size(dt);
    a.n_rows = n_rows;
    a.rows_per_cta = p.R;
    a.M = M;
    a.units_total = p.units_total;
    a.units_per_slice = p.units_per_slice;
    a.stage_units = p.stage_units;
    a.stages_per_slice = p.stages_per_slice;
    a.ring_stages = p.ring_stages;
    a.slices = p.S;
    a.pitch = static_cast<uint32_t>(p.pitch);
    a.stage_bytes = static_cast<uint32_t>(p.stage_bytes);
    a.ring_bytes = static_cast<uint32_t>(p.ring_bytes);
    a.x_off = static_cast<uint32_t>(p.x_off);
    a.skip_stage = g_opt_skip_stage_plus1.load() - 1;
    a.trigger_early = g_opt_trigger_early.load();
    const int wus = g_opt_wait_us.load();
    a.wait_limit_ns = wus > 0 ? static_cast<uint64_t>(wus) * 1000ull : kDefaultWaitNs;
    a.err_word = dev.err_word;
    a.splits = splits;
    a.prefetch = pf;
    if (norm) a.norm = *norm;
    cudaError_t e = cudaSuccess;
    switch (p.compute) {
        case hsp::kMmaBf16:
        case hsp::kFmaBf16: e = hsp::launch_bf16(r); break;
        case hsp::kMmaTf32: e = hsp::launch_tf32(r); break;
        default: e = hsp::launch_fp32(r); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PROJ_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

proj_status validate(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                     void *const *outs, int32_t M, int32_t K, proj_dtype dtype, int64_t *n_total) {
    if (!dtype_valid(dtype)) return fail(PROJ_ERR_UNSUPPORTED_DTYPE, "dtype %d is not PROJ_BF16/FP32/TF32", (int)dtype);
    if (!n_splits || !outs) return fail(PROJ_ERR_INVALID_ARG, "n_splits and outs must not be NULL");
    if (num_splits < 1) return fail(PROJ_ERR_INVALID_ARG, "num_splits=%d (need at least 1)", num_splits);
    if (num_splits > PROJ_MAX_SPLITS)
        return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "num_splits=%d exceeds %d", num_splits, PROJ_MAX_SPLITS);
    int64_t n = 0;
    for (int i = 0; i < num_splits; ++i) {
        if (n_splits[i] < 1) return fail(PROJ_ERR_INVALID_ARG, "n_splits[%d]=%d (need at least 1)", i, n_splits[i]);
        n += n_splits[i];
    }
    proj_status st = check_shape(M, K, n, dtype);
    if (st != PROJ_OK) return st;
    *n_total = n;
    if (M == 0) return PROJ_OK;  // nothing to read or write
    if (!x || !w_cat) return fail(PROJ_ERR_INVALID_ARG, "x and w_cat must not be NULL");
    if (!aligned16(x) || !aligned16(w_cat)) return fail(PROJ_ERR_MISALIGNED, "x and w_cat must be 16-byte aligned");
    const uintptr_t ea = static_cast<uintptr_t>(elem_size(dtype)) - 1;
    for (int i = 0; i < num_splits; ++i) {
        if (!outs[i]) return fail(PROJ_ERR_INVALID_ARG, "outs[%d] is NULL", i);
        if (reinterpret_cast<uintptr_t>(outs[i]) & ea)
            return fail(PROJ_ERR_MISALIGNED, "outs[%d] is not aligned to its element size", i);
    }
    return PROJ_OK;
}

proj_status fused_impl(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                       void *const *outs, int32_t M, int32_t K, proj_dtype dtype, const hsp::PrefetchList &pf,
                       proj_stream_t stream) {
    int64_t n_total = 0;
    proj_status st = validate(x, w_cat, n_splits, num_splits, outs, M, K, dtype, &n_total);
    if (st != PROJ_OK) return st;
    if (M == 0) return ok();
    DeviceInfo dev;
    if ((st = device_info(&dev)) != PROJ_OK) return st;
    hsp::SplitTable t;
    memset(&t, 0, sizeof t);
    t.count = num_splits;
    int off = 0;
    for (int i = 0; i < num_splits; ++i) {
        t.off[i] = off;
        t.rows[i] = n_splits[i];
        t.out[i] = outs[i];
        off += n_splits[i];
    }
    st = launch_rows(dev, x, w_cat, static_cast<int>(n_total), M, K, dtype, t, pf,
                     reinterpret_cast<cudaStream_t>(stream));
    return st == PROJ_OK ? ok() : st;
}

// Co-resident CTAs per cluster size of the current device, for plans made on the
// host only.  Without a usable device the plan assumes a GB300: 152 SMs, 152 / 152 /
// 144 / 120 / 112 CTAs co-resident in clusters of 1 / 2 / 4 / 8 / 16.  Leaves the
// last error string as it was.
void plan_ctas(int (&ctas)[17], int (&pairs)[17], int (&trios)[17]) {
    // GB300 (152 SMs) as measured by the occupancy query, for hosts without the device
    static const int kGb300[17] = {0, 152, 152, 0, 144, 0, 0, 0, 120, 0, 0, 0, 0, 0, 0, 0, 112};
    static const int kGb300Pairs[17] = {0, 304, 304, 0, 296, 0, 0, 0, 288, 0, 0, 0, 0, 0, 0, 0, 224};
    static const int kGb300Trios[17] = {0, 456, 456, 0, 448, 0, 0, 0, 432, 0, 0, 0, 0, 0, 0, 0, 336};
    for (int k = 0; k < 17; ++k) {
        ctas[k] = kGb300[k];
        pairs[k] = kGb300Pairs[k];
        trios[k] = kGb300Trios[k];
    }
    char saved[sizeof g_last_error];
    memcpy(saved, g_last_error, sizeof saved);
    DeviceInfo d;
    if (device_info(&d) == PROJ_OK)
        for (int k = 1; k < 17; ++k) {
            ctas[k] = d.cluster_ctas[k];
            pairs[k] = d.pair_ctas[k];
            trios[k] = d.trio_ctas[k];
        }
    else
        (void)cudaGetLastError();
    memcpy(g_last_error, saved, sizeof saved);
}

// ---- RMSNorm epilogue: workspace layout ----------------------------------------

// Workspace of one call, in this order: the split counters (one 256-byte block),
// the parked fp32 values of the normalized columns ([M][cols] per split), the
// per-CTA sums of squares ([CTAs][M] per split).  A pure function of the shape.
struct NormLayout {
    hsp::NormArgs args;     // offsets and CTA ranges (pointers filled in per call)
    size_t vals_at, part_at, bytes;
};

proj_status norm_layout(int32_t M, int32_t K, const int32_t *n_splits, int32_t num_splits, const int32_t *norm_cols,
                        proj_dtype dtype, const int *cluster_ctas, NormLayout *L) {
    memset(L, 0, sizeof *L);
    if (!n_splits || !norm_cols) return fail(PROJ_ERR_INVALID_ARG, "n_splits and norm_cols must not be NULL");
    if (num_splits < 1 || num_splits > PROJ_MAX_SPLITS)
        return fail(PROJ_ERR_INVALID_ARG, "num_splits=%d (1..%d)", num_splits, PROJ_MAX_SPLITS);
    if (dtype != PROJ_BF16) return fail(PROJ_ERR_UNSUPPORTED_DTYPE, "the RMSNorm epilogue runs for PROJ_BF16 only");
    if (M < 1 || M > 8) return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "the RMSNorm epilogue runs for 1 <= M <= 8 (M=%d)", M);
    int64_t n_total = 0;
    for (int i = 0; i < num_splits; ++i) {
        if (n_splits[i] < 1) return fail(PROJ_ERR_INVALID_ARG, "n_splits[%d]=%d (need at least 1)", i, n_splits[i]);
        if (norm_cols[i] < 0 || norm_cols[i] > n_splits[i])
            return fail(PROJ_ERR_INVALID_ARG, "norm_cols[%d]=%d outside [0, %d]", i, norm_cols[i], n_splits[i]);
        n_total += n_splits[i];
    }
    proj_status st = check_shape(M, K, n_total, dtype);
    if (st != PROJ_OK) return st;
    // rows per CTA of the kernel that will run (the CTA ranges below depend on it)
    int R = 0;
    if (use_reg(M, K, dtype)) {
        RegPlan rp;
        make_reg_plan(M, K, static_cast<int>(n_total), cluster_ctas[1], &rp);
        R = rp.R;
    } else {
        Plan p;
        make_plan(M, K, static_cast<int>(n_total), dtype, cluster_ctas, &p);
        if (p.S != 1) return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "the RMSNorm epilogue needs a single-slice plan");
        R = p.R;
    }
    hsp::NormArgs &a = L->args;
    int64_t vals = 0, part = 0;
    int off = 0;
    for (int i = 0; i < num_splits; ++i) {
        a.cols[i] = norm_cols[i];
        if (norm_cols[i] > 0) {
            a.active = 1;
            a.cta_first[i] = off / R;
            a.cta_count[i] = (off + norm_cols[i] - 1) / R - a.cta_first[i] + 1;
            a.vals_off[i] = vals;
            a.part_off[i] = static_cast<int32_t>(part);
            vals += static_cast<int64_t>(M) * norm_cols[i];
            part += static_cast<int64_t>(M) * a.cta_count[i];
        }
        off += n_splits[i];
    }
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    L->vals_at = 256;
    L->part_at = L->vals_at + up(static_cast<size_t>(vals) * 4);
    L->bytes = L->part_at + up(static_cast<size_t>(part) * 4);
    return PROJ_OK;
}

}  // namespace

// A recorded host step (proj_host_plan_create): the graph and its executable.
struct proj_host_plan {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

extern "C" {

size_t proj_rmsnorm_workspace_bytes(int32_t M, int32_t K, const int32_t *n_splits, int32_t num_splits,
                                    const int32_t *norm_cols, proj_dtype dtype) {
    int ctas[17], pairs[17], trios[17];
    plan_ctas(ctas, pairs, trios);
    NormLayout L;
    if (norm_layout(M, K, n_splits, num_splits, norm_cols, dtype, ctas, &L) != PROJ_OK) return 0;
    return L.bytes;
}

proj_status proj_fused_gemm_rmsnorm(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                                    const int32_t *norm_cols, const void *const *gammas, float eps,
                                    void *const *outs, int32_t M, int32_t K, proj_dtype dtype, void *workspace,
                                    size_t workspace_bytes, proj_stream_t stream) {
    int64_t n_total = 0;
    proj_status st = validate(x, w_cat, n_splits, num_splits, outs, M, K, dtype, &n_total);
    if (st != PROJ_OK) return st;
    if (M == 0) return ok();
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(PROJ_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (!gammas) return fail(PROJ_ERR_INVALID_ARG, "gammas must not be NULL");
    DeviceInfo dev;
    if ((st = device_info(&dev)) != PROJ_OK) return st;
    NormLayout L;
    if ((st = norm_layout(M, K, n_splits, num_splits, norm_cols, dtype, dev.cluster_ctas, &L)) != PROJ_OK) return st;
    if (!workspace) return fail(PROJ_ERR_INVALID_ARG, "workspace must not be NULL");
    if (!aligned16(workspace)) return fail(PROJ_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    if (workspace_bytes < L.bytes)
        return fail(PROJ_ERR_INVALID_ARG, "workspace of %zu bytes, this call needs %zu", workspace_bytes, L.bytes);
    hsp::NormArgs a = L.args;
    for (int i = 0; i < num_splits; ++i) {
        if (a.cols[i] == 0) continue;
        if (!gammas[i]) return fail(PROJ_ERR_INVALID_ARG, "gammas[%d] is NULL", i);
        if (reinterpret_cast<uintptr_t>(gammas[i]) & 1u) return fail(PROJ_ERR_MISALIGNED, "gammas[%d] is not 2-byte aligned", i);
        a.gamma[i] = gammas[i];
    }
    a.eps = eps;
    char *ws = static_cast<char *>(workspace);
    a.counter = reinterpret_cast<unsigned *>(ws);
    a.vals = reinterpret_cast<float *>(ws + L.vals_at);
    a.partial = reinterpret_cast<float *>(ws + L.part_at);
    hsp::SplitTable t;
    memset(&t, 0, sizeof t);
    t.count = num_splits;
    int off = 0;
    for (int i = 0; i < num_splits; ++i) {
        t.off[i] = off;
        t.rows[i] = n_splits[i];
        t.out[i] = outs[i];
        off += n_splits[i];
    }
    hsp::PrefetchList none;
    memset(&none, 0, sizeof none);
    st = launch_rows(dev, x, w_cat, static_cast<int>(n_total), M, K, dtype, t, none,
                     reinterpret_cast<cudaStream_t>(stream), a.active ? &a : nullptr);
    return st == PROJ_OK ? ok() : st;
}


proj_status proj_fused_gemm(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                            void *const *outs, int32_t M, int32_t K, proj_dtype dtype, proj_stream_t stream) {
    hsp::PrefetchList none;
    memset(&none, 0, sizeof none);
    return fused_impl(x, w_cat, n_splits, num_splits, outs, M, K, dtype, none, stream);
}

proj_status proj_fused_gemm_prefetch(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                                     void *const *outs, int32_t M, int32_t K, proj_dtype dtype,
                                     const proj_prefetch_range *ranges, int32_t num_ranges, proj_stream_t stream) {
    if (num_ranges < 0 || num_ranges > PROJ_MAX_PREFETCH || (num_ranges > 0 && !ranges))
        return fail(PROJ_ERR_INVALID_ARG, "num_ranges=%d (0..%d) or ranges NULL", num_ranges, PROJ_MAX_PREFETCH);
    hsp::PrefetchList pf;
    memset(&pf, 0, sizeof pf);
    for (int i = 0; i < num_ranges; ++i) {
        if (!ranges[i].ptr || ranges[i].bytes == 0) return fail(PROJ_ERR_INVALID_ARG, "prefetch range %d is empty", i);
        if (!aligned16(ranges[i].ptr) || ranges[i].bytes % 16 != 0)
            return fail(PROJ_ERR_MISALIGNED, "prefetch range %d: pointer and size must be multiples of 16 bytes", i);
        pf.ptr[pf.count] = static_cast<const char *>(ranges[i].ptr);
        pf.bytes[pf.count] = ranges[i].bytes;
        ++pf.count;
    }
    return fused_impl(x, w_cat, n_splits, num_splits, outs, M, K, dtype, pf, stream);
}

proj_status proj_fused_gemm_host(const void *x_host, const void *w_cat, const int32_t *n_splits,
                                 int32_t num_splits, void *const *outs_host, int32_t M, int32_t K, proj_dtype dtype,
                                 void *x_dev, void *const *outs_dev, proj_stream_t stream) {
    int64_t n_total = 0;
    proj_status st = validate(x_dev, w_cat, n_splits, num_splits, outs_dev, M, K, dtype, &n_total);
    if (st != PROJ_OK) return st;
    if (M == 0) return ok();
    if (!x_host || !outs_host) return fail(PROJ_ERR_INVALID_ARG, "x_host and outs_host must not be NULL");
    for (int i = 0; i < num_splits; ++i)
        if (!outs_host[i]) return fail(PROJ_ERR_INVALID_ARG, "outs_host[%d] is NULL", i);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t esz = static_cast<size_t>(elem_size(dtype));
    const size_t x_bytes = static_cast<size_t>(M) * K * esz;  // a multiple of 16 (validated row size)
    // Tokens in page-locked host memory that the device can address are copied by the
    // staging kernel, chained to the projection by programmatic dependent launch; any
    // other host buffer (pageable memory) goes through a copy-engine copy.
    const void *x_src = nullptr;
    {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, x_host) == cudaSuccess) {
            if (pa.type == cudaMemoryTypeHost && pa.devicePointer &&
                (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15u) == 0 &&
                (reinterpret_cast<uintptr_t>(x_dev) & 15u) == 0)
                x_src = pa.devicePointer;
        } else {
            (void)cudaGetLastError();  // pageable memory: not an error, copy it
        }
    }
    cudaError_t e;
    if (x_src) {
        DeviceInfo dev;
        if ((st = device_info(&dev)) != PROJ_OK) return st;
        e = hsp::launch_stage(x_src, x_dev, static_cast<int64_t>(x_bytes / 16), dev.sms, g_opt_pdl.load(), s);
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch (token staging)");
        g_launches.fetch_add(1, std::memory_order_relaxed);
    } else {
        e = cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (tokens to the device)");
    }
    // An output in page-locked host memory that the device can address (mapped, as
    // cudaHostAlloc memory is under unified addressing) is written by the kernel itself,
    // over the host link, instead of through a staging buffer and a copy; the stream's
    // completion makes those stores visible to the host like a copy's.
    void *direct[PROJ_MAX_SPLITS];
    for (int i = 0; i < num_splits; ++i) {
        direct[i] = nullptr;
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, outs_host[i]) == cudaSuccess) {
            if (pa.type == cudaMemoryTypeHost && pa.devicePointer &&
                (reinterpret_cast<uintptr_t>(pa.devicePointer) & (esz - 1)) == 0)
                direct[i] = pa.devicePointer;
        } else {
            (void)cudaGetLastError();  // pageable memory: not an error, copy it
        }
    }
    void *kout[PROJ_MAX_SPLITS];
    for (int i = 0; i < num_splits; ++i) kout[i] = direct[i] ? direct[i] : outs_dev[i];
    hsp::PrefetchList none;
    memset(&none, 0, sizeof none);
    st = fused_impl(x_dev, w_cat, n_splits, num_splits, kout, M, K, dtype, none, stream);
    if (st != PROJ_OK) return st;
    for (int i = 0; i < num_splits; ++i) {
        if (direct[i]) continue;
        e = cudaMemcpyAsync(outs_host[i], outs_dev[i], static_cast<size_t>(M) * n_splits[i] * esz,
                            cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (outputs to the host)");
    }
    return ok();
}

proj_status proj_host_plan_create(const void *x_host, const void *w_cat, const int32_t *n_splits,
                                  int32_t num_splits, void *const *outs_host, int32_t M, int32_t K, proj_dtype dtype,
                                  void *x_dev, void *const *outs_dev, proj_host_plan **plan) {
    if (!plan) return fail(PROJ_ERR_INVALID_ARG, "plan must not be NULL");
    *plan = nullptr;
    int64_t n_total = 0;
    proj_status st = validate(x_dev, w_cat, n_splits, num_splits, outs_dev, M, K, dtype, &n_total);
    if (st != PROJ_OK) return st;
    if (M == 0) return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "a host plan needs M >= 1");
    DeviceInfo dev;
    if ((st = device_info(&dev)) != PROJ_OK) return st;
    cudaStream_t cs = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags (recording stream)");
    proj_host_plan *p = new proj_host_plan;
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        st = proj_fused_gemm_host(x_host, w_cat, n_splits, num_splits, outs_host, M, K, dtype, x_dev, outs_dev,
                                  reinterpret_cast<proj_stream_t>(cs));
        cudaGraph_t g = nullptr;
        const cudaError_t ee = cudaStreamEndCapture(cs, &g);
        p->graph = g;
        if (st == PROJ_OK && ee != cudaSuccess) st = cuda_fail(ee, "cudaStreamEndCapture");
        if (st == PROJ_OK) {
            e = cudaGraphInstantiate(&p->exec, p->graph, 0);
            if (e != cudaSuccess) st = cuda_fail(e, "cudaGraphInstantiate");
        }
    } else {
        st = cuda_fail(e, "cudaStreamBeginCapture");
    }
    (void)cudaStreamDestroy(cs);
    if (st != PROJ_OK) {
        char saved[sizeof g_last_error];
        memcpy(saved, g_last_error, sizeof saved);
        if (p->exec) (void)cudaGraphExecDestroy(p->exec);
        if (p->graph) (void)cudaGraphDestroy(p->graph);
        delete p;
        (void)cudaGetLastError();
        memcpy(g_last_error, saved, sizeof saved);
        return st;
    }
    *plan = p;
    return ok();
}

proj_status proj_host_plan_launch(proj_host_plan *plan, proj_stream_t stream) {
    if (!plan || !plan->exec) return fail(PROJ_ERR_INVALID_ARG, "plan is NULL or not created");
    const cudaError_t e = cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch (host plan)");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ok();
}

proj_status proj_host_plan_destroy(proj_host_plan *plan) {
    if (!plan) return ok();
    cudaError_t e1 = plan->exec ? cudaGraphExecDestroy(plan->exec) : cudaSuccess;
    cudaError_t e2 = plan->graph ? cudaGraphDestroy(plan->graph) : cudaSuccess;
    delete plan;
    if (e1 != cudaSuccess) return cuda_fail(e1, "cudaGraphExecDestroy");
    if (e2 != cudaSuccess) return cuda_fail(e2, "cudaGraphDestroy");
    return ok();
}

proj_status proj_separate_gemm(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                               void *const *outs, int32_t M, int32_t K, proj_dtype dtype, proj_stream_t stream) {
    int64_t n_total = 0;
    proj_status st = validate(x, w_cat, n_splits, num_splits, outs, M, K, dtype, &n_total);
    if (st != PROJ_OK) return st;
    if (M == 0) return ok();
    DeviceInfo dev;
    if ((st = device_info(&dev)) != PROJ_OK) return st;
    const size_t pitch = static_cast<size_t>(K) * elem_size(dtype);
    size_t off = 0;
    for (int i = 0; i < num_splits; ++i) {
        hsp::SplitTable t;
        memset(&t, 0, sizeof t);
        t.count = 1;
        t.rows[0] = n_splits[i];
        t.out[0] = outs[i];
        const void *wi = static_cast<const char *>(w_cat) + off * pitch;
        hsp::PrefetchList none;
        memset(&none, 0, sizeof none);
        st = launch_rows(dev, x, wi, n_splits[i], M, K, dtype, t, none, reinterpret_cast<cudaStream_t>(stream));
        if (st != PROJ_OK) return st;
        off += static_cast<size_t>(n_splits[i]);
    }
    return ok();
}

proj_status proj_pack_weights(const void *const *ws, const int32_t *n_rows, int32_t num, int32_t K,
                              proj_dtype dtype, void *w_cat, proj_stream_t stream) {
    if (!dtype_valid(dtype)) return fail(PROJ_ERR_UNSUPPORTED_DTYPE, "dtype %d is not PROJ_BF16/FP32/TF32", (int)dtype);
    if (!ws || !n_rows || !w_cat) return fail(PROJ_ERR_INVALID_ARG, "ws, n_rows and w_cat must not be NULL");
    if (num < 1 || num > PROJ_MAX_SPLITS)
        return fail(PROJ_ERR_INVALID_ARG, "num=%d (1..%d weights per pack)", num, PROJ_MAX_SPLITS);
    if (K < 1) return fail(PROJ_ERR_INVALID_ARG, "K=%d (need at least 1)", K);
    const size_t pitch = static_cast<size_t>(K) * elem_size(dtype);
    if (pitch % 16 != 0)
        return fail(PROJ_ERR_MISALIGNED, "rows of K=%d elements are %zu bytes, not a multiple of 16", K, pitch);
    if (!aligned16(w_cat)) return fail(PROJ_ERR_MISALIGNED, "w_cat must be 16-byte aligned");
    size_t total_rows = 0;
    for (int i = 0; i < num; ++i) {
        if (n_rows[i] < 0) return fail(PROJ_ERR_INVALID_ARG, "n_rows[%d]=%d is negative", i, n_rows[i]);
        if (n_rows[i] == 0) continue;  // nothing to read: any pointer, NULL included
        if (!ws[i]) return fail(PROJ_ERR_INVALID_ARG, "ws[%d] is NULL", i);
        if (!aligned16(ws[i])) return fail(PROJ_ERR_MISALIGNED, "ws[%d] must be 16-byte aligned", i);
        total_rows += static_cast<size_t>(n_rows[i]);
    }
    // W_cat occupies [lo, hi).  A source inside that range is either exactly its own
    // rows (already packed: nothing to copy) or refused: the copy would read rows that
    // this or an earlier part overwrites.
    const uintptr_t lo = reinterpret_cast<uintptr_t>(w_cat), hi = lo + total_rows * pitch;
    hsp::PackArgs a;
    memset(&a, 0, sizeof a);
    size_t off = 0;
    for (int i = 0; i < num; ++i) {
        const size_t bytes = static_cast<size_t>(n_rows[i]) * pitch;
        const uintptr_t src = reinterpret_cast<uintptr_t>(ws[i]), dst = lo + off * pitch;
        off += static_cast<size_t>(n_rows[i]);
        if (bytes == 0 || src == dst) continue;
        if (src < hi && src + bytes > lo)
            return fail(PROJ_ERR_INVALID_ARG, "ws[%d] overlaps w_cat without being its own rows [%zu, %zu)", i,
                        off - n_rows[i], off);
        a.src[a.count] = reinterpret_cast<const uint4 *>(ws[i]);
        a.dst16[a.count] = static_cast<int64_t>((dst - lo) / 16);
        a.first16[a.count + 1] = a.first16[a.count] + static_cast<int64_t>(bytes / 16);
        ++a.count;
    }
    if (a.count == 0) return ok();  // every part already is its own rows
    DeviceInfo dev;
    proj_status st = device_info(&dev);
    if (st != PROJ_OK) return st;
    cudaError_t e = hsp::launch_pack(w_cat, a, dev.sms * 4, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pack kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ok();
}

int proj_pack_check(const void *w, const void *w_cat, int64_t row_off, int32_t n_rows, int32_t n_total, int32_t K,
                    proj_dtype dtype) {
    if (!w || !w_cat || !dtype_valid(dtype) || row_off < 0 || n_rows < 0 || K < 1) return 0;
    if (row_off + n_rows > n_total) return 0;
    const uintptr_t want = reinterpret_cast<uintptr_t>(w_cat) +
                           static_cast<uintptr_t>(row_off) * static_cast<uintptr_t>(K) * elem_size(dtype);
    return reinterpret_cast<uintptr_t>(w) == want ? 1 : 0;
}

int proj_supported(int32_t M, int32_t K, int32_t n_total, proj_dtype dtype) {
    char saved[sizeof g_last_error];
    memcpy(saved, g_last_error, sizeof saved);
    const bool good = M >= 1 && n_total >= 1 && check_shape(M, K, n_total, dtype) == PROJ_OK;
    memcpy(g_last_error, saved, sizeof saved);
    return good ? 1 : 0;
}

proj_status proj_describe_plan(int32_t M, int32_t K, int32_t n_rows, proj_dtype dtype, proj_plan_info *info) {
    if (!info) return fail(PROJ_ERR_INVALID_ARG, "info must not be NULL");
    proj_status st = check_shape(M, K, n_rows, dtype);
    if (st != PROJ_OK) return st;
    if (M < 1 || n_rows < 1) return fail(PROJ_ERR_UNSUPPORTED_SHAPE, "M and n_rows must be at least 1");
    int ctas[17], pairs[17], trios[17];
    plan_ctas(ctas, pairs, trios);
    if (use_umma(M, dtype)) {
        UPlan u;
        make_umma_plan(M, K, n_rows, dtype, pairs, trios, &u);
        *info = u.info;
        return ok();
    }
    if (use_reg(M, K, dtype)) {
        RegPlan rp;
        make_reg_plan(M, K, n_rows, ctas[1], &rp);
        reg_plan_info(M, K, rp, info);
        return ok();
    }
    if (use_gemv(M, K, dtype)) {
        GemvPlan gp;
        make_gemv_plan(M, K, n_rows, ctas[1], &gp);
        gemv_plan_info(M, K, gp, info);
        return ok();
    }
    Plan p;
    make_plan(M, K, n_rows, dtype, ctas, &p);
    *info = p.info;
    return ok();
}

proj_status proj_set_options(const proj_options *opt) {
    if (!opt) return fail(PROJ_ERR_INVALID_ARG, "opt must not be NULL");
    if (opt->pdl < -1 || opt->pdl > 1) return fail(PROJ_ERR_INVALID_ARG, "pdl must be -1, 0 or 1");
    if (opt->wait_limit_us < 0 || opt->skip_stage_plus1 < 0)
        return fail(PROJ_ERR_INVALID_ARG, "wait_limit_us and skip_stage_plus1 must be >= 0");
    if (opt->large_m_path < 0 || opt->large_m_path > 2 || opt->l2_prefetch < 0 || opt->l2_prefetch > 1 ||
        opt->trigger_early < 0 || opt->trigger_early > 1 || opt->small_m_path < 0 || opt->small_m_path > 1 ||
        opt->reg_path < 0 || opt->reg_path > 2)
        return fail(PROJ_ERR_INVALID_ARG,
                    "large_m_path and reg_path must be 0, 1 or 2; small_m_path, l2_prefetch and trigger_early 0 or 1");
    if (opt->pdl >= 0) g_opt_pdl.store(opt->pdl);
    g_opt_wait_us.store(opt->wait_limit_us);
    g_opt_skip_stage_plus1.store(opt->skip_stage_plus1);
    g_opt_large_m_path.store(opt->large_m_path);
    g_opt_l2_prefetch.store(opt->l2_prefetch);
    g_opt_trigger_early.store(opt->trigger_early);
    g_opt_small_m_path.store(opt->small_m_path);
    g_opt_reg_path.store(opt->reg_path);
    return ok();
}

proj_status proj_get_options(proj_options *opt) {
    if (!opt) return fail(PROJ_ERR_INVALID_ARG, "opt must not be NULL");
    memset(opt, 0, sizeof *opt);
    opt->pdl = g_opt_pdl.load();
    opt->wait_limit_us = g_opt_wait_us.load();
    opt->skip_stage_plus1 = g_opt_skip_stage_plus1.load();
    opt->large_m_path = g_opt_large_m_path.load();
    opt->l2_prefetch = g_opt_l2_prefetch.load();
    opt->trigger_early = g_opt_trigger_early.load();
    opt->small_m_path = g_opt_small_m_path.load();
    opt->reg_path = g_opt_reg_path.load();
    return ok();
}

proj_status proj_check_device_error(proj_stream_t stream) {
    DeviceInfo dev;
    proj_status st = device_info(&dev);
    if (st != PROJ_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpy(&v, dev.err_word, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(dev.err_word, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        if (v == PROJ_ERR_TIMEOUT) return fail(PROJ_ERR_TIMEOUT, "a kernel gave up a bounded wait (timeout)");
        return fail(PROJ_ERR_CUDA, "device error word %d", v);
    }
    return ok();
}

uint64_t proj_launch_count(void) { return g_launches.load(); }

const char *proj_last_error_string(void) { return g_last_error; }

const char *proj_version(void) { return "hsp_proj 0.1 (sm_103a)"; }

}  // extern "C"
