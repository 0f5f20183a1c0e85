/*
 * CPU oracle for the tiled fp32 matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may
 * include, link, load or call this file; only the tests, the smoke check and
 * the benchmark's CPU-baseline leg use it.  It shares no code, header or
 * constant with the CUDA kernels.
 *
 * What it computes is the plain definition of the product the pages' tiled
 * kernels compute ("My Triton From Scratch, Part 14: Shared Memory Tiles",
 * section "Shared buffers are physical storage": dot(block<BMxBK>,
 * block<BKxBN>) -> block<BMxBN>, accumulated over the runtime K loop of
 * section "Staging inside a runtime K loop").  Masked, zero-filled edge
 * tiles contribute nothing (section "Matching the safety mask": the masked
 * load gives elements outside the matrix no weight), so the tiled result
 * is, up to rounding order, the untiled textbook product:
 *
 *     C[i][j] = fp32( sum_{k=0}^{K-1} (double)A[i][k] * (double)B[k][j] )
 *
 * with A row-major M x K (row stride K), B row-major K x N (row stride N)
 * and C row-major M x N (row stride N), as in the canonical A and B loads of
 * section "The canonical source pattern" (a + rows*K + cols, b + rows*N +
 * cols).  The sum runs in increasing k in double precision and is rounded
 * once to fp32 (round to nearest even, the C cast).  Each product of two
 * floats is exact in double.  The accumulator starts at zero
 * (tl.zeros in "Staging inside a runtime K loop"), so K == 0 gives C = 0.
 *
 * Alongside C it can return W[i][j] = sum_k |A[i][k]| * |B[k][j]| in double,
 * the scale the elementwise tolerance of the parity tests is measured in.
 *
 * No blocking, no reordering of the k sum: the loops are i, then k, then j,
 * which keeps each C[i][j]'s sum in increasing k while streaming rows of B.
 * Rows are independent and split over OpenMP threads.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -fPIC -shared
 */
#include <stdint.h>
#include <stdlib.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row i: acc[j] = sum_k A[i][k]*B[k][j] (and wacc for W). */
static void oracle_row(const float *A, const float *B, int64_t N, int64_t K,
                       int64_t i, double *acc, double *wacc,
                       float *c_row, double *w_row)
{
    for (int64_t j = 0; j < N; ++j) {
        acc[j] = 0.0;
        if (wacc) wacc[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)A[i * K + k];
        const float *b_row = B + k * N;
        for (int64_t j = 0; j < N; ++j)
            acc[j] += a * (double)b_row[j];
        if (wacc) {
            const double aa = fabs(a);
            for (int64_t j = 0; j < N; ++j)
                wacc[j] += aa * fabs((double)b_row[j]);
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        c_row[j] = (float)acc[j];
        if (w_row) w_row[j] = wacc[j];
    }
}

/* Every row listed in rows[0..nrows): C_out[r][*] is row rows[r] of A*B.
 * rows == NULL means rows 0..nrows-1 (the full product when nrows == M).
 * W_out may be NULL.  nthreads <= 0 uses the OpenMP default.
 * Returns 0, or -1 on a bad argument or allocation failure. */
int oracle_sgemm_rows(const float *A, const float *B, float *C_out,
                      double *W_out, int64_t M, int64_t N, int64_t K,
                      const int64_t *rows, int64_t nrows, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (nrows == 0 || N == 0) return 0;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(|:failed)
#endif
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        double *wacc = W_out ? (double *)malloc((size_t)N * sizeof(double)) : NULL;
        if (!acc || (W_out && !wacc)) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t i = rows ? rows[r] : r;
                if (i < 0 || i >= M) { failed = 1; continue; }
                oracle_row(A, B, N, K, i, acc, wacc, C_out + r * N,
                           W_out ? W_out + r * N : NULL);
            }
        }
        free(acc);
        free(wacc);
    }
    return failed ? -1 : 0;
}

/* The full product: C (M x N) and optionally W (M x N). */
int oracle_sgemm(const float *A, const float *B, float *C, double *W,
                 int64_t M, int64_t N, int64_t K, int nthreads)
{
    return oracle_sgemm_rows(A, B, C, W, M, N, K, NULL, M, nthreads);
}

/* Single elements: out[t] = C[ii[t]][jj[t]], wout[t] = W[ii[t]][jj[t]]
 * (wout may be NULL).  Same per-element sum as oracle_sgemm. */
int oracle_sgemm_elements(const float *A, const float *B, float *out,
                          double *wout, int64_t M, int64_t N, int64_t K,
                          const int64_t *ii, const int64_t *jj, int64_t count)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = ii[t], j = jj[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return -1;
        double acc = 0.0, w = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * K + k];
            const double b = (double)B[k * N + j];
            acc += a * b;
            w += fabs(a) * fabs(b);
        }
        out[t] = (float)acc;
        if (wout) wout[t] = w;
    }
    return 0;
}

/* The general form (BLAS-style), with an optional bias row:
 *
 *     C[i][j] = fp32( alpha * sum_k a(i,k) * b(k,j)  +  beta * C[i][j]  +  bias[j] )
 *
 * summed in increasing k in double, rounded once, with
 *   a(i,k) = trans_a ? A[k*lda + i] : A[i*lda + k]
 *   b(k,j) = trans_b ? B[j*ldb + k] : B[k*ldb + j]
 * and C[i][j] at C[i*ldc + j].  beta == 0 means C is not read (a NaN in C
 * is overwritten); alpha == 0 means A and B are not read.  With alpha = 1,
 * beta = 0, no transposes and packed leading dimensions this is exactly
 * oracle_sgemm (same sum, same rounding).  W (optional, M x N packed)
 * receives |alpha| * sum_k |a(i,k)| |b(k,j)| + |beta| * |C[i][j]|, the
 * scale of the general form's tolerance, plus |bias[j]|.  bias (N floats)
 * may be NULL: no bias.  The pages stop at the plain product; the bias is
 * read as a linear layer's, one value per output column added to every
 * row, inside the same fp64 sum before the single rounding.  Returns 0, or
 * -1 on a bad argument or allocation failure. */
int oracle_sgemm_general_bias(const float *A, int64_t lda, const float *B, int64_t ldb,
                              const float *bias, float *C, int64_t ldc, double *W,
                              int64_t M, int64_t N, int64_t K, double alpha, double beta,
                              int trans_a, int trans_b, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || ldc < N) return -1;
    if (!trans_a && lda < K) return -1;
    if (trans_a && lda < M) return -1;
    if (!trans_b && ldb < N) return -1;
    if (trans_b && ldb < K) return -1;
    if (M == 0 || N == 0) return 0;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(|:failed)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, w = 0.0;
            if (alpha != 0.0) {
                for (int64_t k = 0; k < K; ++k) {
                    const double a = (double)(trans_a ? A[k * lda + i] : A[i * lda + k]);
                    const double b = (double)(trans_b ? B[j * ldb + k] : B[k * ldb + j]);
                    acc += a * b;
                    w += fabs(a) * fabs(b);
                }
            }
            double c = alpha * acc;
            double wc = fabs(alpha) * w;
            if (beta != 0.0) {
                const double c0 = (double)C[i * ldc + j];
                c += beta * c0;
                wc += fabs(beta) * fabs(c0);
            }
            if (bias) {
                c += (double)bias[j];
                wc += fabs((double)bias[j]);
            }
            C[i * ldc + j] = (float)c;
            if (W) W[i * N + j] = wc;
        }
    }
    return failed ? -1 : 0;
}

/* The general form without a bias. */
int oracle_sgemm_general(const float *A, int64_t lda, const float *B, int64_t ldb,
                         float *C, int64_t ldc, double *W, int64_t M, int64_t N,
                         int64_t K, double alpha, double beta, int trans_a, int trans_b,
                         int nthreads)
{
    return oracle_sgemm_general_bias(A, lda, B, ldb, NULL, C, ldc, W, M, N, K, alpha, beta,
                                     trans_a, trans_b, nthreads);
}

/* ------------------------------------------------------------------------
 * 16-bit inputs, fp32 products and sums ("My Triton From Scratch, Part 18",
 * section "Next" announces Part 19, mixed-precision types; the plainest
 * reading, and the one tl.dot takes for 16-bit operands, is inputs stored in
 * 16 bits and accumulation in fp32).  The result is the same definition as
 * above on the values the 16-bit patterns encode:
 *
 *     C[i][j] = fp32( alpha * sum_k a(i,k) * b(k,j)  +  beta * C[i][j] )
 *
 * summed in increasing k in double and rounded once.  A product of two
 * 16-bit values is exact in double (at most 22 significant bits).
 *
 * The patterns are decoded from the formats' definitions:
 *   binary16 (IEEE 754): sign bit 15, exponent bits 14..10 (bias 15),
 *     fraction bits 9..0; exponent 0 is zero or subnormal (f * 2^-24),
 *     exponent 31 is infinity (f == 0) or NaN.
 *   bfloat16: the upper half of a binary32 — sign bit 15, exponent bits
 *     14..7 (bias 127), fraction bits 6..0; exponent 0 is zero or subnormal
 *     (f * 2^-133), exponent 255 is infinity or NaN.
 */
enum { ORACLE_F16 = 1, ORACLE_BF16 = 2 };

double oracle_f16_value(uint16_t h)
{
    const int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

double oracle_bf16_value(uint16_t h)
{
    const int s = (h >> 15) & 1, e = (h >> 7) & 0xFF, f = h & 0x7F;
    double v;
    if (e == 0) v = ldexp((double)f, -133);
    else if (e == 255) v = f ? NAN : INFINITY;
    else v = ldexp((double)(128 + f), e - 134);
    return s ? -v : v;
}

/* The general form on 16-bit A and B (both of type `dtype`, ORACLE_F16 or
 * ORACLE_BF16), fp32 C; layouts, W, the alpha/beta rules and the optional
 * bias row (NULL: none) as in oracle_sgemm_general_bias.  Returns 0, or -1
 * on a bad argument. */
int oracle_gemm_mixed_general_bias(int dtype, const uint16_t *A, int64_t lda,
                                   const uint16_t *B, int64_t ldb, const float *bias, float *C,
                                   int64_t ldc, double *W, int64_t M, int64_t N, int64_t K,
                                   double alpha, double beta, int trans_a, int trans_b,
                                   int nthreads)
{
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    if (M < 0 || N < 0 || K < 0 || ldc < N) return -1;
    if (!trans_a && lda < K) return -1;
    if (trans_a && lda < M) return -1;
    if (!trans_b && ldb < N) return -1;
    if (trans_b && ldb < K) return -1;
    if (M == 0 || N == 0) return 0;
    double (*value)(uint16_t) = dtype == ORACLE_F16 ? oracle_f16_value : oracle_bf16_value;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, w = 0.0;
            if (alpha != 0.0) {
                for (int64_t k = 0; k < K; ++k) {
                    const double a = value(trans_a ? A[k * lda + i] : A[i * lda + k]);
                    const double b = value(trans_b ? B[j * ldb + k] : B[k * ldb + j]);
                    acc += a * b;
                    w += fabs(a) * fabs(b);
                }
            }
            double c = alpha * acc;
            double wc = fabs(alpha) * w;
            if (beta != 0.0) {
                const double c0 = (double)C[i * ldc + j];
                c += beta * c0;
                wc += fabs(beta) * fabs(c0);
            }
            if (bias) {
                c += (double)bias[j];
                wc += fabs((double)bias[j]);
            }
            C[i * ldc + j] = (float)c;
            if (W) W[i * N + j] = wc;
        }
    }
    return 0;
}

/* The 16-bit general form without a bias. */
int oracle_gemm_mixed_general(int dtype, const uint16_t *A, int64_t lda, const uint16_t *B,
                              int64_t ldb, float *C, int64_t ldc, double *W, int64_t M,
                              int64_t N, int64_t K, double alpha, double beta, int trans_a,
                              int trans_b, int nthreads)
{
    return oracle_gemm_mixed_general_bias(dtype, A, lda, B, ldb, NULL, C, ldc, W, M, N, K,
                                          alpha, beta, trans_a, trans_b, nthreads);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
