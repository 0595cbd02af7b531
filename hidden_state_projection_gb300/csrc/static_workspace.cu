// static_workspace.cu -- proj_fused_gemm_rmsnorm_static: the RMSNorm-epilogue call for
// callers that cannot allocate device memory.
//
// proj_fused_gemm_rmsnorm needs a caller-owned workspace.  Some callers have no way
// to provide one: code running under an inference runtime that owns every byte of
// device memory through its own pool and forbids side allocations, plugins handed
// only the tensors of one operation, and latency-critical paths where cudaMalloc's
// implicit device-wide synchronisation is not acceptable.  This entry point uses a
// fixed array compiled into the library instead and allocates nothing.
//
// The array lives in device memory of every GPU that loads this library, for the
// life of the process.  Host code cannot use its name as a device address: the
// address is looked up (cudaGetSymbolAddress, with the device current) on the first
// call made in a context, and again whenever the current context is not the one the
// address was looked up in (a device reset with cudaDeviceReset, or another context
// on the same device, gives the array a new address).
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "proj.h"

namespace hsp {
proj_status set_last_error(proj_status st, const char *msg);  // proj_api.cu
uint64_t current_context_id();                                // proj_api.cu
}  // namespace hsp

namespace {

// Large enough for M = 8 tokens and about 28,000 normalized columns in total
// (parked fp32 values M * sum(norm_cols) * 4 bytes, plus the per-CTA sums and the
// split counters).
constexpr size_t kStaticWorkspaceBytes = size_t(1) << 20;  // 1 MiB

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {nullptr};
uint64_t g_addr_ctx[kMaxDevices] = {0};  // context each address was looked up in

// Device address of g_static_workspace in the current context.
cudaError_t workspace_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t ctx = hsp::current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev] || ctx == 0 || ctx != g_addr_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
        g_addr_ctx[dev] = hsp::current_context_id();  // the lookup made a context current if none was
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" proj_status proj_fused_gemm_rmsnorm_static(const void *x, const void *w_cat, const int32_t *n_splits,
                                                      int32_t num_splits, const int32_t *norm_cols,
                                                      const void *const *gammas, float eps, void *const *outs,
                                                      int32_t M, int32_t K, proj_dtype dtype, proj_stream_t stream) {
    if (M == 0) return proj_fused_gemm_rmsnorm(x, w_cat, n_splits, num_splits, norm_cols, gammas, eps, outs, M, K,
                                               dtype, nullptr, 0, stream);
    const size_t need = proj_rmsnorm_workspace_bytes(M, K, n_splits, num_splits, norm_cols, dtype);
    if (need == 0) return PROJ_ERR_UNSUPPORTED_SHAPE;  // the reason is in proj_last_error_string
    char msg[256];
    if (need > kStaticWorkspaceBytes) {
        // Shapes past the fixed array take the allocating-caller entry point instead.
        std::snprintf(msg, sizeof msg,
                      "proj_fused_gemm_rmsnorm_static: this call needs %zu bytes of workspace, the built-in array "
                      "holds %zu (pass a workspace of your own to proj_fused_gemm_rmsnorm)", need, kStaticWorkspaceBytes);
        return hsp::set_last_error(PROJ_ERR_UNSUPPORTED_SHAPE, msg);
    }
    void *ws = nullptr;
    cudaError_t e = workspace_address(&ws);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof msg, "proj_fused_gemm_rmsnorm_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return hsp::set_last_error(PROJ_ERR_CUDA, msg);
    }
    // Every call shares the array and finds the previous call's contents there.  Only
    // the arrival counters and abort flags (the first 256 bytes) must start at zero: a
    // __device__ array is zero when the library is loaded, and every call, one that gave
    // up a wait included, leaves them at zero again.  So nothing is cleared per call.
    return proj_fused_gemm_rmsnorm(x, w_cat, n_splits, num_splits, norm_cols, gammas, eps, outs, M, K, dtype, ws,
                                   kStaticWorkspaceBytes, stream);
}
