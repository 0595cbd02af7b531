/*
 * oracle.c -- reference CPU implementation of the fused hidden-state projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   y[m][n]  = sum_{k=0..K-1} double(x[m][k]) * double(w_cat[n][k])
 *              accumulated in fp64 in increasing k;
 *   out_i[m][n - off_i] = round_out(y[m][n])   for off_i <= n < off_i + N_i,
 *              off_i = N_0 + ... + N_{i-1}.
 *
 * Passages followed:
 *   - TensorRT-LLM PR #20636 (DeepSeek-V4.1 wq_a/wkv via tinygemm2), Description:
 *     wq_a (5120 -> 1280) and wkv (5120 -> 512) are plain Linear projections of the
 *     same hidden state; their weights are copied into one row-concatenated
 *     [1792, 5120] tensor, one GEMM runs over it and the two halves come back as
 *     dense [M, N_i] outputs; closeness is judged against an FP32 F.linear.
 *   - TensorRT-LLM PR #12055 (indexer wk + weights_proj in one TF32 GEMM),
 *     Description: the two indexer projections become one FP32 GEMM.
 *   - TensorRT-LLM PR #8771 (QK down_proj + indexer K + weights_proj), Walkthrough:
 *     kv_a_proj_with_mqa widened with the indexer rows, output split per projection.
 *   - TensorRT-LLM PR #20502 (GLM-5.2 decode target), glmFusedAGemm commit
 *     message: FP32 sums rounded to BF16 once.
 *
 * Rounding (round_out):
 *   - BF16 outputs: fp64 -> bf16 round-to-nearest, ties to even, written here
 *     from the IEEE 754 definition of the bfloat16 format (1 sign bit,
 *     8 exponent bits with bias 127, 7 fraction bits, gradual underflow),
 *     directly from the fp64 value, never through fp32.
 *   - FP32 outputs: the C conversion double -> float, which rounds to nearest
 *     even under the default floating-point environment.
 *
 * Products of two bf16 values (8+8 significant bits) and of two fp32 values
 * (24+24 bits) are exact in fp64 (53 bits), so the only rounding before
 * round_out is that of the fp64 additions.
 *
 * Threads split the output rows n; each y[m][n] is computed by one thread with
 * the same loop, so the result does not depend on the thread count.
 *
 * RMSNorm epilogue (oracle_fused_rmsnorm): the consumers of the q_a / kv_a
 * projections are RMSNorms (TensorRT-LLM PR #20636, Description: q_norm reads wq_a's
 * output and kv_norm reads wkv's; PR #20502, glm_mla_kv_half_append commit message:
 * the kv_a_proj output's 512 latent columns, not its RoPE part, are normalised).  For a split i with
 * c_i = norm_cols[i] > 0 and every token m, from the fp64 sums above:
 *
 *   ms[m]  = (1 / c_i) * sum_{r < c_i} y[m][off_i + r]^2          (fp64, increasing r)
 *   out_i[m][r] = round_out( y[m][off_i + r] / sqrt(ms[m] + eps) * gamma_i[r] )  r < c_i
 *   out_i[m][r] = round_out( y[m][off_i + r] )                                   r >= c_i
 *
 * with gamma_i in the data type; one rounding per output, as for the projection.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_BF16 = 0, ORACLE_FP32 = 1 };

/* ---- element decode ---------------------------------------------------- */

/* A bf16 value is the top 16 bits of the fp32 with the same sign, exponent and
 * leading fraction bits; widening is therefore a 16-bit left shift (exact). */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int64_t idx, int dtype) {
    if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    return (double)((const float *)base)[idx];
}

/* ---- fp64 -> bf16, round to nearest, ties to even ------------------------ */

uint16_t oracle_double_to_bf16(double v) {
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;

    /* Quantum (spacing of representable values) at the magnitude of a:
     * normal numbers in [2^e, 2^(e+1)) carry 7 fraction bits -> 2^(e-7);
     * below 2^-126 the spacing is fixed at 2^-133 (subnormals). */
    int ex;
    (void)frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) -> e = ex - 1 */
    int e = ex - 1;
    if (e < -126) e = -126;
    int qexp = e - 7;

    double r = ldexp(a, -qexp);   /* exact: scaling by a power of two */
    double n = floor(r);
    double frac = r - n;          /* exact: r and n share the binade */
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;

    /* n is the significand in units of the quantum: [128, 256] for normals,
     * [0, 128] for subnormals.  n == 256 carries into the next binade. */
    uint32_t exp_field, mant;
    if (n >= 256.0) { e += 1; n = 128.0; }
    if (n < 128.0) {               /* subnormal (only reachable when e == -126) */
        exp_field = 0;
        mant = (uint32_t)n;
    } else {
        exp_field = (uint32_t)(e + 127);
        mant = (uint32_t)(n - 128.0);
    }
    if (exp_field >= 255u) return (uint16_t)(sign | 0x7F80u);   /* overflow -> inf */
    return (uint16_t)(sign | (exp_field << 7) | mant);
}

/* ---- the projection ------------------------------------------------------ */

/* y_acc[m*ld + n] for n in [n0, n1): fp64 sums, no rounding. */
static void accumulate_rows(const void *x, const void *w, int64_t M, int64_t K, int dtype,
                            int64_t n0, int64_t n1, double *y_acc, int64_t ld) {
    for (int64_t n = n0; n < n1; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += load_elem(x, m * K + k, dtype) * load_elem(w, n * K + k, dtype);
            y_acc[m * ld + n] = s;
        }
    }
}

/* Sums only: y_acc is [M, N] row-major fp64.  Used by the tests to pin the
 * accumulation separately from the rounding. */
void oracle_accumulate(const void *x, const void *w, int64_t M, int64_t N, int64_t K,
                       int dtype, double *y_acc) {
    accumulate_rows(x, w, M, K, dtype, 0, N, y_acc, N);
}

void oracle_round(const double *y, int64_t count, int dtype, void *out) {
    for (int64_t i = 0; i < count; ++i) {
        if (dtype == ORACLE_BF16) ((uint16_t *)out)[i] = oracle_double_to_bf16(y[i]);
        else ((float *)out)[i] = (float)y[i];
    }
}

typedef struct {
    const void *x, *w;
    int64_t M, K, n0, n1, ld;
    int dtype;
    double *y;
} job_t;

static void *run_job(void *arg) {
    job_t *j = (job_t *)arg;
    accumulate_rows(j->x, j->w, j->M, j->K, j->dtype, j->n0, j->n1, j->y, j->ld);
    return NULL;
}

/* The fused projection: one pass over all rows of w_cat, then every row is
 * rounded once and written to the output of the projection it belongs to.
 * outs[i] is a dense [M, n_splits[i]] array of the output dtype.
 * Returns 0 on success, -1 on bad arguments or allocation failure. */
int oracle_fused(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                 void *const *outs, int64_t M, int64_t K, int dtype, int threads) {
    if (M < 0 || K < 0 || num_splits < 1 || !n_splits || !outs) return -1;
    int64_t N = 0;
    for (int32_t i = 0; i < num_splits; ++i) {
        if (n_splits[i] < 0) return -1;
        N += n_splits[i];
    }
    if (M == 0 || N == 0) return 0;
    double *y = (double *)malloc(sizeof(double) * (size_t)(M * N));
    if (!y) return -1;

    if (threads < 1) threads = 1;
    if (threads > N) threads = (int)N;
    if (threads == 1) {
        accumulate_rows(x, w_cat, M, K, dtype, 0, N, y, N);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
        job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)threads);
        char *live = (char *)calloc((size_t)threads, 1);
        if (!tid || !jobs || !live) { free(tid); free(jobs); free(live); free(y); return -1; }
        for (int t = 0; t < threads; ++t) {
            jobs[t] = (job_t){x, w_cat, M, K, N * t / threads, N * (t + 1) / threads, N, dtype, y};
            if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) == 0) live[t] = 1;
            else run_job(&jobs[t]);          /* no thread: do the rows here */
        }
        for (int t = 0; t < threads; ++t)
            if (live[t]) pthread_join(tid[t], NULL);
        free(tid);
        free(jobs);
        free(live);
    }

    int64_t off = 0;
    for (int32_t i = 0; i < num_splits; ++i) {
        int64_t ni = n_splits[i];
        for (int64_t m = 0; m < M; ++m)
            for (int64_t r = 0; r < ni; ++r) {
                double v = y[m * N + off + r];
                if (dtype == ORACLE_BF16) ((uint16_t *)outs[i])[m * ni + r] = oracle_double_to_bf16(v);
                else ((float *)outs[i])[m * ni + r] = (float)v;
            }
        off += ni;
    }
    free(y);
    return 0;
}

/* The separate-call form: one projection per split over its row range of
 * w_cat.  Each call is the fused definition restricted to one range. */
int oracle_separate(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                    void *const *outs, int64_t M, int64_t K, int dtype, int threads) {
    if (num_splits < 1 || !n_splits || !outs) return -1;
    size_t esz = (dtype == ORACLE_BF16) ? 2 : 4;
    int64_t off = 0;
    for (int32_t i = 0; i < num_splits; ++i) {
        const char *wi = (const char *)w_cat + (size_t)(off * K) * esz;
        int rc = oracle_fused(x, wi, &n_splits[i], 1, &outs[i], M, K, dtype, threads);
        if (rc) return rc;
        off += n_splits[i];
    }
    return 0;
}

/* The fused projection followed by the RMSNorm epilogue described at the top.
 * norm_cols[i] in [0, n_splits[i]] (0: split i is not normalized); gammas[i]
 * points to norm_cols[i] elements of the data type (unused when norm_cols[i] is 0).
 * Returns 0 on success, -1 on bad arguments or allocation failure. */
int oracle_fused_rmsnorm(const void *x, const void *w_cat, const int32_t *n_splits, int32_t num_splits,
                         const int32_t *norm_cols, const void *const *gammas, double eps,
                         void *const *outs, int64_t M, int64_t K, int dtype) {
    if (M < 0 || K < 0 || num_splits < 1 || !n_splits || !outs || !norm_cols || !gammas) return -1;
    int64_t N = 0;
    for (int32_t i = 0; i < num_splits; ++i) {
        if (n_splits[i] < 0 || norm_cols[i] < 0 || norm_cols[i] > n_splits[i]) return -1;
        if (norm_cols[i] > 0 && !gammas[i]) return -1;
        N += n_splits[i];
    }
    if (M == 0 || N == 0) return 0;
    double *y = (double *)malloc(sizeof(double) * (size_t)(M * N));
    if (!y) return -1;
    accumulate_rows(x, w_cat, M, K, dtype, 0, N, y, N);
    int64_t off = 0;
    for (int32_t i = 0; i < num_splits; ++i) {
        const int64_t ni = n_splits[i], ci = norm_cols[i];
        for (int64_t m = 0; m < M; ++m) {
            double inv = 1.0;
            if (ci > 0) {
                double ss = 0.0;
                for (int64_t r = 0; r < ci; ++r) {
                    const double v = y[m * N + off + r];
                    ss += v * v;
                }
                inv = 1.0 / sqrt(ss / (double)ci + eps);
            }
            for (int64_t r = 0; r < ni; ++r) {
                double v = y[m * N + off + r];
                if (r < ci) v = v * inv * load_elem(gammas[i], r, dtype);
                if (dtype == ORACLE_BF16) ((uint16_t *)outs[i])[m * ni + r] = oracle_double_to_bf16(v);
                else ((float *)outs[i])[m * ni + r] = (float)v;
            }
        }
        off += ni;
    }
    free(y);
    return 0;
}
