/*
 * abi_consumer.c -- the library used from plain C (C99), through include/proj.h only:
 * no C++, no Python, no torch.  Links against libhsp_proj.so (and, for the device run,
 * the CUDA runtime's C API).
 *
 *   abi_consumer host    queries and argument checks that need no GPU (exit 0 on success)
 *   abi_consumer reset   calls before and after cudaDeviceReset (this process's context only):
 *                        the library's per-device caches follow the new context
 *   abi_consumer device  W_cat packed from three weights (proj_pack_weights), then one
 *                        fused and one separate call on small-integer bf16 data,
 *                        checked element by element against a double loop written here
 *                        (entries in {-1, 0, 1} and K = 192: every partial sum is an
 *                        integer of magnitude at most 192, exact in fp32 and in bf16)
 *
 * Exit status: 0 = all checks passed, 1 = a check failed, 2 = usage or setup error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "proj.h"

#ifdef ABI_CONSUMER_DEVICE
#include <cuda_runtime_api.h>
#endif

static int failures = 0;

static void check(int ok, const char *what) {
    if (!ok) {
        fprintf(stderr, "FAILED: %s (last error: %s)\n", what, proj_last_error_string());
        ++failures;
    }
}

static int host_checks(void) {
    const int32_t splits[2] = {16, 8};
    void *outs[2] = {(void *)0x30000, (void *)0x31000};
    proj_plan_info info;

    check(strlen(proj_version()) > 0, "proj_version");
    check(proj_supported(8, 5120, 1792, PROJ_BF16) == 1, "proj_supported(8, 5120, 1792, bf16)");
    check(proj_supported(65, 5120, 1792, PROJ_BF16) == 0, "proj_supported refuses M = 65");
    check(proj_describe_plan(8, 5120, 1792, PROJ_BF16, &info) == PROJ_OK && info.rows_per_cta >= 1 &&
              info.row_ctas * info.rows_per_cta >= 1792,
          "proj_describe_plan");
    /* argument checks return a status before anything touches a device */
    check(proj_fused_gemm((void *)0x10000, (void *)0x20000, splits, 2, outs, 1, 64, (proj_dtype)9, NULL) ==
              PROJ_ERR_UNSUPPORTED_DTYPE,
          "unknown dtype refused");
    check(proj_fused_gemm((void *)0x10000, (void *)0x20000, splits, 2, outs, 65, 64, PROJ_BF16, NULL) ==
              PROJ_ERR_UNSUPPORTED_SHAPE,
          "M = 65 refused");
    check(proj_fused_gemm((void *)0x10008, (void *)0x20000, splits, 2, outs, 1, 64, PROJ_BF16, NULL) ==
              PROJ_ERR_MISALIGNED,
          "misaligned x refused");
    check(proj_fused_gemm(NULL, (void *)0x20000, splits, 2, outs, 1, 64, PROJ_BF16, NULL) == PROJ_ERR_INVALID_ARG,
          "NULL x refused");
    check(strlen(proj_last_error_string()) > 0, "the last refusal has a message");
    {
        /* the packer's refusals happen on the host, before anything is enqueued */
        const void *parts[2] = {(const void *)0x50000, (const void *)0x60000};
        const void *inside[2] = {(const void *)(0x20000 + 8 * 128), (const void *)0x60000};
        const int32_t rows[2] = {16, 8};
        check(proj_pack_weights(parts, rows, 2, 60, PROJ_BF16, (void *)0x20000, NULL) == PROJ_ERR_MISALIGNED,
              "pack: 120-byte rows refused");
        check(proj_pack_weights(inside, rows, 2, 64, PROJ_BF16, (void *)0x20000, NULL) == PROJ_ERR_INVALID_ARG,
              "pack: a source inside w_cat that is not its own rows refused");
        check(proj_pack_weights(parts, rows, 9, 64, PROJ_BF16, (void *)0x20000, NULL) == PROJ_ERR_INVALID_ARG,
              "pack: more parts than PROJ_MAX_SPLITS refused");
    }
    return failures == 0 ? 0 : 1;
}

#ifdef ABI_CONSUMER_DEVICE
/* bf16 bits of a small integer (exact: |v| < 256 needs at most 8 significant bits) */
static uint16_t bf16_of_int(int v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static double double_of_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int device_checks(void) {
    enum { M = 5, K = 192, NS = 3 };
    const int32_t splits[NS] = {17, 1, 40};
    const int N = 17 + 1 + 40;
    uint16_t *x = malloc(sizeof(uint16_t) * M * K), *w = malloc(sizeof(uint16_t) * N * K);
    uint16_t *got = malloc(sizeof(uint16_t) * M * N);
    void *dx = NULL, *dw = NULL, *douts[NS] = {NULL, NULL, NULL};
    int i, s, m, n, k, off, path;
    if (!x || !w || !got) return 2;
    srand(12345);
    for (i = 0; i < M * K; ++i) x[i] = bf16_of_int(rand() % 3 - 1);  /* {-1, 0, 1} */
    for (i = 0; i < N * K; ++i) w[i] = bf16_of_int(rand() % 3 - 1);
    if (cudaMalloc(&dx, sizeof(uint16_t) * M * K) != cudaSuccess ||
        cudaMalloc(&dw, sizeof(uint16_t) * N * K) != cudaSuccess)
        return 2;
    for (s = 0; s < NS; ++s)
        if (cudaMalloc(&douts[s], sizeof(uint16_t) * M * splits[s]) != cudaSuccess) return 2;
    cudaMemcpy(dx, x, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice);
    /* W_cat is packed by the library from three separately allocated weights */
    {
        void *dparts[NS] = {NULL, NULL, NULL};
        const void *cparts[NS];
        uint16_t *back = malloc(sizeof(uint16_t) * N * K);
        if (!back) return 2;
        off = 0;
        for (s = 0; s < NS; ++s) {
            if (cudaMalloc(&dparts[s], sizeof(uint16_t) * splits[s] * K) != cudaSuccess) return 2;
            cudaMemcpy(dparts[s], w + (size_t)off * K, sizeof(uint16_t) * splits[s] * K, cudaMemcpyHostToDevice);
            cparts[s] = dparts[s];
            off += splits[s];
        }
        check(proj_pack_weights(cparts, splits, NS, K, PROJ_BF16, dw, NULL) == PROJ_OK, "proj_pack_weights");
        check(cudaDeviceSynchronize() == cudaSuccess, "device synchronise after the pack");
        cudaMemcpy(back, dw, sizeof(uint16_t) * N * K, cudaMemcpyDeviceToHost);
        check(memcmp(back, w, sizeof(uint16_t) * N * K) == 0, "packed w_cat is the row concatenation");
        for (s = 0; s < NS; ++s) cudaFree(dparts[s]);
        free(back);
    }
    for (path = 0; path < 2; ++path) {
        const proj_status st = path == 0 ? proj_fused_gemm(dx, dw, splits, NS, douts, M, K, PROJ_BF16, NULL)
                                         : proj_separate_gemm(dx, dw, splits, NS, douts, M, K, PROJ_BF16, NULL);
        check(st == PROJ_OK, path == 0 ? "proj_fused_gemm" : "proj_separate_gemm");
        check(cudaDeviceSynchronize() == cudaSuccess, "device synchronise");
        check(proj_check_device_error(NULL) == PROJ_OK, "no device-side error");
        off = 0;
        for (s = 0; s < NS; ++s) {
            cudaMemcpy(got, douts[s], sizeof(uint16_t) * M * splits[s], cudaMemcpyDeviceToHost);
            for (m = 0; m < M; ++m)
                for (n = 0; n < splits[s]; ++n) {
                    double want = 0.0;
                    for (k = 0; k < K; ++k) want += double_of_bf16(x[m * K + k]) * double_of_bf16(w[(off + n) * K + k]);
                    if (double_of_bf16(got[m * splits[s] + n]) != want) {
                        fprintf(stderr, "path %d split %d [%d, %d]: %g, want %g\n", path, s, m, n,
                                double_of_bf16(got[m * splits[s] + n]), want);
                        ++failures;
                        goto next_split;
                    }
                }
        next_split:
            off += splits[s];
        }
    }
    for (s = 0; s < NS; ++s) cudaFree(douts[s]);
    cudaFree(dx);
    cudaFree(dw);
    free(x);
    free(w);
    free(got);
    return failures == 0 ? 0 : 1;
}

/* One round of calls on freshly allocated buffers: an exact fused call (small integers,
 * checked against a double loop) and the no-allocation RMSNorm call (status and finite
 * outputs), then the device error word. */
static void reset_round(const char *when) {
    enum { M = 4, K = 192, NS = 2 };
    const int32_t splits[NS] = {16, 8}, norm_cols[NS] = {16, 8};
    const int N = 24;
    uint16_t x[M * K], w[N * K], got[M * 16], gam[16];
    void *dx = NULL, *dw = NULL, *douts[NS] = {NULL, NULL}, *dg[NS] = {NULL, NULL};
    const void *gammas[NS];
    char what[160];
    int i, m, n, k, s;
    for (i = 0; i < M * K; ++i) x[i] = bf16_of_int((i * 7) % 3 - 1);
    for (i = 0; i < N * K; ++i) w[i] = bf16_of_int((i * 5) % 3 - 1);
    for (i = 0; i < 16; ++i) gam[i] = bf16_of_int(1);
    if (cudaMalloc(&dx, sizeof x) != cudaSuccess || cudaMalloc(&dw, sizeof w) != cudaSuccess) {
        ++failures;
        return;
    }
    for (s = 0; s < NS; ++s)
        if (cudaMalloc(&douts[s], sizeof(uint16_t) * M * splits[s]) != cudaSuccess ||
            cudaMalloc(&dg[s], sizeof(uint16_t) * 16) != cudaSuccess) {
            ++failures;
            return;
        }
    cudaMemcpy(dx, x, sizeof x, cudaMemcpyHostToDevice);
    cudaMemcpy(dw, w, sizeof w, cudaMemcpyHostToDevice);
    for (s = 0; s < NS; ++s) {
        cudaMemcpy(dg[s], gam, sizeof(uint16_t) * 16, cudaMemcpyHostToDevice);
        gammas[s] = dg[s];
    }
    snprintf(what, sizeof what, "proj_fused_gemm (%s)", when);
    check(proj_fused_gemm(dx, dw, splits, NS, douts, M, K, PROJ_BF16, NULL) == PROJ_OK, what);
    check(cudaDeviceSynchronize() == cudaSuccess, "device synchronise");
    cudaMemcpy(got, douts[0], sizeof(uint16_t) * M * 16, cudaMemcpyDeviceToHost);
    for (m = 0; m < M; ++m)
        for (n = 0; n < 16; ++n) {
            double want = 0.0;
            for (k = 0; k < K; ++k) want += double_of_bf16(x[m * K + k]) * double_of_bf16(w[n * K + k]);
            if (double_of_bf16(got[m * 16 + n]) != want) {
                snprintf(what, sizeof what, "fused output [%d, %d] exact (%s)", m, n, when);
                check(0, what);
                m = M;
                break;
            }
        }
    for (s = 0; s < NS; ++s) cudaMemset(douts[s], 0xFF, sizeof(uint16_t) * M * splits[s]); /* NaN poison */
    snprintf(what, sizeof what, "proj_fused_gemm_rmsnorm_static (%s)", when);
    check(proj_fused_gemm_rmsnorm_static(dx, dw, splits, NS, norm_cols, gammas, 1e-6f, douts, M, K, PROJ_BF16,
                                         NULL) == PROJ_OK,
          what);
    check(cudaDeviceSynchronize() == cudaSuccess, "device synchronise after the static call");
    cudaMemcpy(got, douts[0], sizeof(uint16_t) * M * 16, cudaMemcpyDeviceToHost);
    for (i = 0; i < M * 16; ++i)
        if ((got[i] & 0x7F80) == 0x7F80) {
            snprintf(what, sizeof what, "static call output %d finite (%s)", i, when);
            check(0, what);
            break;
        }
    snprintf(what, sizeof what, "no device-side error (%s)", when);
    check(proj_check_device_error(NULL) == PROJ_OK, what);
    for (s = 0; s < NS; ++s) {
        cudaFree(douts[s]);
        cudaFree(dg[s]);
    }
    cudaFree(dx);
    cudaFree(dw);
}

/* The library caches per-device facts: the device error word's address, the
 * no-allocation entry point's array address, kernels' attribute set-up.  A device reset
 * gives the next context new addresses; every cache is keyed by the context, so calls
 * after cudaDeviceReset (in this process only) must work as before it. */
static int reset_checks(void) {
    reset_round("before the reset");
    check(cudaDeviceReset() == cudaSuccess, "cudaDeviceReset");
    reset_round("after the reset");
    check(cudaDeviceReset() == cudaSuccess, "second cudaDeviceReset");
    reset_round("after a second reset");
    return failures == 0 ? 0 : 1;
}
#endif

int main(int argc, char **argv) {
    if (argc < 2) return 2;
    if (strcmp(argv[1], "host") == 0) return host_checks();
#ifdef ABI_CONSUMER_DEVICE
    if (strcmp(argv[1], "device") == 0) return device_checks();
    if (strcmp(argv[1], "reset") == 0) return reset_checks();
#endif
    return 2;
}
