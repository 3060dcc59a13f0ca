/*
 * convrot_oracle.c -- plain, slow CPU oracle for the INT8ConvRot linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it follows.  The page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal,
 * MPSMatrix, and MLX" (lilting.ch), section "What changed in the computation":
 *   - H: Kronecker products of 4x4 Hadamard matrices stacked to 256x256 and
 *     divided by sqrt(256) = 16; applied to the last dimension in groups of 256.
 *   - weight prep (once):  W_rot = W H^T,  s_W[n] = max_k |W_rot[n,k]| / 127,
 *                          Q_W = round(W_rot / s_W)
 *   - per call:            X_rot = X H,    s_X[m] = max_k |X_rot[m,k]| / 127,
 *                          Q_X = round(X_rot / s_X)
 *   - A = Q_X Q_W^T accumulated in int32,  Y = A (.) s_X s_W^T
 *   - rounded values are clamped to [-128, 127].
 * The unmerged LoRA term follows the page "[PR #249] Add an mps backend:
 * weight-only INT8 and W4A8/W6A8 linears for Apple GPUs", section "What"
 * (lora_down [R,K], lora_up [N,R], lora_scale), applied to the unrotated X.
 *
 * Arithmetic: fp64 everywhere except the integer GEMM (exact, int64 sums that
 * are checked to fit int32) and the one step the reading fixes in fp32 (the
 * scale restore, oracle_epilogue_f32).  Nothing is blocked, fused or
 * reordered: each function is the textbook loop of the formula it names.
 * OpenMP (when compiled in) only splits independent rows across threads.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off [-fopenmp]
 * (-ffp-contract=off so that x86 and Arm hosts compute the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define G 256 /* Hadamard group size */

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the OpenMP runtime will use (1 when built without it). */
int oracle_max_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * H = (B (x) B (x) B (x) B) / 16 for a 4x4 base B (row-major), written out as
 * the Kronecker product: with i = 64 i3 + 16 i2 + 4 i1 + i0 (base-4 digits,
 * most significant digit on the first factor) and likewise j,
 *     H[i][j] = B[i3][j3] B[i2][j2] B[i1][j1] B[i0][j0] / 16.
 * Output: H as a dense 256x256 row-major fp64 array.
 */
void oracle_hadamard256(const double base4[16], double *H) {
    for (int i = 0; i < G; ++i) {
        for (int j = 0; j < G; ++j) {
            double v = 1.0;
            int ii = i, jj = j;
            for (int d = 0; d < 4; ++d) { /* least significant digit first */
                v *= base4[(ii % 4) * 4 + (jj % 4)];
                ii /= 4;
                jj /= 4;
            }
            H[i * G + j] = v / 16.0;
        }
    }
}

/*
 * Group-wise rotation of the last dimension (dense 256x256 matvec per group):
 *   transpose_h == 0:  out[r, 256g + j] = sum_i in[r, 256g + i] * H[i][j]   (X H)
 *   transpose_h == 1:  out[r, 256g + j] = sum_i in[r, 256g + i] * H[j][i]   (W H^T)
 * K must be a multiple of 256.
 */
void oracle_rotate_groups(const double *in, int64_t rows, int64_t K,
                          const double *H, int transpose_h, double *out,
                          int nthreads) {
    set_threads(nthreads);
    const int64_t groups = K / G;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            const double *x = in + r * K + g * G;
            double *y = out + r * K + g * G;
            for (int j = 0; j < G; ++j) {
                double acc = 0.0;
                for (int i = 0; i < G; ++i) {
                    double h = transpose_h ? H[j * G + i] : H[i * G + j];
                    acc += x[i] * h;
                }
                y[j] = acc;
            }
        }
    }
}

/*
 * Row-wise symmetric int8 quantization of v [rows, K]:
 *   s[r]   = max_k |v[r,k]| / 127
 *   pre    = v[r,k] / s[r]                      (the value that is rounded)
 *   q[r,k] = clamp(round_half_even(pre), -128, 127)
 * An all-zero row has no scale to divide by: s = 0 and q = 0 (a reading; the
 * pages do not discuss it).  `pre` may be NULL.
 */
void oracle_quantize_rows(const double *v, int64_t rows, int64_t K, int8_t *q,
                          double *s, double *pre, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double *x = v + r * K;
        double amax = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = fabs(x[k]);
            if (a > amax) amax = a;
        }
        double scale = amax / 127.0;
        s[r] = scale;
        for (int64_t k = 0; k < K; ++k) {
            double p = (scale > 0.0) ? x[k] / scale : 0.0;
            double rq = nearbyint(p); /* default FE_TONEAREST: ties to even */
            if (rq > 127.0) rq = 127.0;
            if (rq < -128.0) rq = -128.0;
            q[r * K + k] = (int8_t)rq;
            if (pre) pre[r * K + k] = p;
        }
    }
}

/*
 * A[m][n] = sum_k Q_X[m][k] * Q_W[n][k], the naive triple loop.  Sums are kept
 * in int64; the return value counts entries that do not fit int32 (such an
 * entry is stored wrapped, and a caller must treat a non-zero return as a
 * failure).
 */
int64_t oracle_int_gemm(const int8_t *QX, const int8_t *QW, int64_t M,
                        int64_t N, int64_t K, int32_t *A, int nthreads) {
    set_threads(nthreads);
    int64_t overflow = 0;
#pragma omp parallel for schedule(static) reduction(+ : overflow)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k)
                acc += (int64_t)QX[m * K + k] * (int64_t)QW[n * K + k];
            if (acc > INT32_MAX || acc < INT32_MIN) ++overflow;
            A[m * N + n] = (int32_t)(uint32_t)(uint64_t)acc;
        }
    }
    return overflow;
}

/*
 * Scale restore Y = A (.) s_X s_W^T in fp32, in the order ((float)A * s_X) * s_W
 * (the reading of an order the pages leave open).  Each product is one IEEE
 * fp32 multiply.
 */
void oracle_epilogue_f32(const int32_t *A, const float *sX, const float *sW,
                         int64_t M, int64_t N, float *Y) {
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float t = (float)A[m * N + n] * sX[m];
            Y[m * N + n] = t * sW[n];
        }
    }
}

/*
 * Optional bias, added after the scale restore as its own fp32 add (eager's
 * order on the page "[PR #249] Add an mps backend: weight-only INT8 and
 * W4A8/W6A8 linears for Apple GPUs", section "Design": the epilogue "adds
 * bias ... in eager's order"): Y[m][n] = Y[m][n] + bias[n], one IEEE fp32
 * addition per element (this file is compiled without FMA contraction).
 */
void oracle_add_bias_f32(float *Y, const float *bias, int64_t M, int64_t N) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) Y[m * N + n] = Y[m * N + n] + bias[n];
}

/*
 * fp32 -> bf16 with round-to-nearest-even (the same page, section "Design":
 * the output is written "bf16 bit-exactly with torch's cast").  From the
 * IEEE 754 definition: bf16 keeps the sign, the 8-bit exponent and the top
 * 7 fraction bits of the fp32 pattern.  The dropped 16 bits are rounded to
 * nearest, ties to the even kept pattern; a carry out of the fraction
 * increments the exponent (up to infinity).  Infinities pass through; a NaN
 * stays a NaN (quiet bit set).
 */
void oracle_round_bf16(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &in[i], 4);
        const uint32_t exp = (u >> 23) & 0xffu;
        const uint32_t frac = u & 0x7fffffu;
        if (exp == 0xffu) {  /* inf or NaN */
            out[i] = (uint16_t)((u >> 16) | (frac ? 0x0040u : 0u));
            continue;
        }
        const uint32_t kept = u >> 16;          /* sign, exponent, 7 fraction bits */
        const uint32_t dropped = u & 0xffffu;
        uint32_t r = kept;
        if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) r += 1u;
        out[i] = (uint16_t)r;
    }
}

/*
 * Unmerged LoRA term in fp64:
 *   T[m][r]  = sum_k X[m][k] * down[r][k]              (X is the unrotated input)
 *   L[m][n]  = scale * sum_r T[m][r] * up[n][r]
 */
void oracle_lora(const double *X, int64_t M, int64_t K, const double *down,
                 int64_t R, const double *up, int64_t N, double scale,
                 double *L, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double *T = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
        for (int64_t r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += X[m * K + k] * down[r * K + k];
            T[r] = acc;
        }
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t r = 0; r < R; ++r) acc += T[r] * up[n * R + r];
            L[m * N + n] = scale * acc;
        }
        free(T);
    }
}

/* Plain fp64 Y = X W^T (the unquantized layer), for error reports and the
 * rotation-invariance check. */
void oracle_matmul_nt(const double *X, const double *W, int64_t M, int64_t N,
                      int64_t K, double *Y, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += X[m * K + k] * W[n * K + k];
            Y[m * N + n] = acc;
        }
    }
}
