/*
 * oracle_sgemm.c -- CPU oracle for single-precision GEMM, C = alpha*A*B + beta*C.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load this library. The product path (the
 * CUDA library) never calls it and shares no code, header or constant with it.
 *
 * What it computes is the plain definition of the operation that every kernel
 * on the pages implements:
 *   - "Shared Memory Tiling", kernel listing: each output is
 *     alpha * (sum over k of A[row][k] * B[k][col]) + beta * C[row][col];
 *   - "Warp Tiling: A Third Level of Tiling", section "The Kernel", epilogue:
 *     the same alpha * result + beta * old-C update on row-major matrices;
 *   - "Vectorized Memory Access: 128-bit Loads and Stores", section "The
 *     Kernel", epilogue: identical update, read-modify-write of C.
 * The tiling on those pages only changes the order in which the k-terms are
 * summed, never which terms are summed.
 *
 * Layout: row-major. A(i,k) = A[i*lda + k], B(k,j) = B[k*ldb + j],
 * C(i,j) = C[i*ldc + j] (the pages' pointer offsets with a general leading
 * dimension instead of the implicit lda = K, ldb = ldc = N).
 *
 * Precision: every float operand is widened to double; a product of two floats
 * is exact in double (24 + 24 < 53 significant bits); the sum over k runs in
 * ascending k in double. On integer inputs whose partial sums stay far below
 * 2^53 the result is therefore exact.
 *
 * Readings where the pages are silent:
 *   - beta == 0: C is not read at all (so NaN or garbage in C cannot leak in);
 *   - alpha == 0 or K == 0: A and B are not read; the result is beta * C.
 *
 * Besides the reference value the oracle returns, per element, the magnitude
 * |alpha| * sum_k |A(i,k) B(k,j)| + |beta| * |C(i,j)| that the error bound of
 * the FP32 result is stated against.
 */
#include <math.h>

/* One output element: reference value and magnitude, by the definition. */
static void oracle_one(long i, long j, long K, float alpha, const float *A, long lda,
                       const float *B, long ldb, float beta, const float *C, long ldc,
                       double *value, double *magnitude)
{
    double sum = 0.0;      /* sum_k A(i,k) * B(k,j)     */
    double abs_sum = 0.0;  /* sum_k |A(i,k) * B(k,j)|   */
    if (alpha != 0.0f) {
        for (long k = 0; k < K; ++k) {
            double product = (double)A[i * lda + k] * (double)B[k * ldb + j];
            sum += product;
            abs_sum += fabs(product);
        }
    }
    double v = (double)alpha * sum;
    double m = fabs((double)alpha) * abs_sum;
    if (beta != 0.0f) {
        double c = (double)C[i * ldc + j];
        v += (double)beta * c;
        m += fabs((double)beta) * fabs(c);
    }
    *value = v;
    *magnitude = m;
}

/*
 * Rows [row_begin, row_end) of the reference result.
 * ref[(i-row_begin)*ldr + j] receives the value, mag[...] (same indexing) the
 * magnitude; mag may be NULL. Returns 0, or -1 on an invalid argument.
 */
int oracle_sgemm_rows(long M, long N, long K, float alpha, const float *A, long lda,
                      const float *B, long ldb, float beta, const float *C, long ldc,
                      long row_begin, long row_end, double *ref, double *mag, long ldr)
{
    if (M < 0 || N < 0 || K < 0 || row_begin < 0 || row_end > M || row_begin > row_end)
        return -1;
    if (ldr < N)
        return -1;
    for (long i = row_begin; i < row_end; ++i) {
        for (long j = 0; j < N; ++j) {
            double v, m;
            oracle_one(i, j, K, alpha, A, lda, B, ldb, beta, C, ldc, &v, &m);
            ref[(i - row_begin) * ldr + j] = v;
            if (mag)
                mag[(i - row_begin) * ldr + j] = m;
        }
    }
    return 0;
}

/*
 * Selected elements (rows[t], cols[t]) for t < count, for spot checks of
 * results too large to recompute whole. Returns 0, or -1 on an index outside
 * the M x N result.
 */
int oracle_sgemm_elements(long M, long N, long K, float alpha, const float *A, long lda,
                          const float *B, long ldb, float beta, const float *C, long ldc,
                          long count, const long *rows, const long *cols,
                          double *ref, double *mag)
{
    for (long t = 0; t < count; ++t) {
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N)
            return -1;
        double v, m;
        oracle_one(rows[t], cols[t], K, alpha, A, lda, B, ldb, beta, C, ldc, &v, &m);
        ref[t] = v;
        if (mag)
            mag[t] = m;
    }
    return 0;
}
