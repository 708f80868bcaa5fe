/*
 * CPU oracle for dense row-major GEMM  C[M x N] = A[M x K] . B[K x N].
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or table with the
 * CUDA library.
 *
 * What it computes (the plain definition, accumulated in IEEE double):
 *
 *   C[i][j] = sum_{k=0..K-1} A[i][k] * B[k][j]        (k increasing)
 *   S[i][j] = sum_{k=0..K-1} |A[i][k] * B[k][j]|
 *
 * Sources:
 *   - "GEMM：从朴素实现到 shared memory tiling 与寄存器分块" (quant67.com),
 *     opening statement of the computation target: row-major
 *     C_{MxN} = A_{MxK} x B_{KxN}, 2MNK floating-point operations, and its
 *     section 1 naive kernel (one output per thread, K-loop over
 *     A[row*K+k] * B[k*N+col]).
 *   - "[CUDA 优化实战] sgemm - 超越 cuBLAS" (wingedge777.com), section 1,
 *     sgemm_naive: one C element per thread, accumulate along k.
 *   - m.lqnn.cn SGEMM article, section 1.1: 2*M*N*K operations per GEMM.
 *   - GB300 GEMM roadmap (m.nxbn.cn), section 6.2: correctness is judged
 *     against a high-precision reference, not against another fast GEMM;
 *     S[i][j] is the scale for the normalised error |dC| / sum|a*b|.
 *   - The scaled form alpha * A.B + beta * C (oracle_gemm_scaled_rows) is
 *     documented beside its function.
 *   - Transposed storage of an operand (op = 1, oracle_gemm_op_rows) is
 *     documented beside its function.
 *
 * The only deviation from those kernels is the accumulator type: double
 * instead of float/half, so the oracle is exact up to one double rounding per
 * add.  Half (IEEE binary16) and bfloat16 inputs are decoded to double from
 * their bit layouts by the functions below; no CUDA header is used.
 *
 * Element (i,k) of A is A[i*lda + k]; element (k,j) of B is B[k*ldb + j]
 * (or, for an operand stored transposed, see a_index / b_index); element
 * (r,j) of the output is C[r*ldc + j].  Every pointer is host memory owned
 * by the caller.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal:    (-1)^s * (1024 + f) * 2^(e - 15 - 10),  1 <= e <= 30
 * Subnormal: (-1)^s * f * 2^(-14 - 10),               e == 0
 * e == 31 encodes infinity (f == 0) or NaN. */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Normal:    (-1)^s * (128 + f) * 2^(e - 127 - 7),   1 <= e <= 254
 * Subnormal: (-1)^s * f * 2^(-126 - 7),               e == 0 */
double oracle_bf16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);
    return s ? -v : v;
}

/* Round a double to a binary floating-point format with `p` significant bits,
 * exponent bias `bias` and `ebits` exponent bits, round-to-nearest, ties to
 * even, in one rounding step from the double value.  Returns the bit pattern.
 * Used to state what a correctly rounded FP16/BF16 output of an exact
 * accumulator looks like (the reading that output conversion rounds to
 * nearest-even). */
static uint16_t round_to_bits(double x, int p, int ebits, int bias)
{
    uint16_t sign = signbit(x) ? (uint16_t)(1u << (p - 1 + ebits)) : 0;
    int emax_field = (1 << ebits) - 1;
    double ax = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | (emax_field << (p - 1)) | (1u << (p - 2)));
    if (isinf(x))
        return (uint16_t)(sign | (emax_field << (p - 1)));
    if (ax == 0.0)
        return sign;
    int e2;
    frexp(ax, &e2);          /* ax = m * 2^e2, m in [0.5, 1) => unbiased exponent e2-1 */
    int unb = e2 - 1;
    int emin = 1 - bias;     /* smallest normal exponent */
    int qexp = (unb < emin ? emin : unb) - (p - 1); /* quantum 2^qexp */
    double r = nearbyint(ldexp(ax, -qexp));        /* ties to even (default mode) */
    /* r is the integer significand at quantum 2^qexp. */
    uint32_t field_e, frac;
    if (unb < emin) {
        /* subnormal range: value = r * 2^(emin - p + 1); r <= 2^(p-1) */
        if (r >= ldexp(1.0, p - 1)) { field_e = 1; frac = 0; }
        else { field_e = 0; frac = (uint32_t)r; }
    } else {
        if (r >= ldexp(1.0, p)) { r = ldexp(r, -1); unb += 1; }
        field_e = (uint32_t)(unb + bias);
        frac = (uint32_t)r - (1u << (p - 1));
        if ((int)field_e >= emax_field)
            return (uint16_t)(sign | (emax_field << (p - 1)));
    }
    return (uint16_t)(sign | (field_e << (p - 1)) | frac);
}

uint16_t oracle_f64_to_f16_rn(double x)  { return round_to_bits(x, 11, 5, 15); }
uint16_t oracle_f64_to_bf16_rn(double x) { return round_to_bits(x, 8, 8, 127); }

static double load_elem(int dtype, const void *p, int64_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)p)[idx];
    if (dtype == ORACLE_F16)
        return oracle_f16_to_f64(((const uint16_t *)p)[idx]);
    return oracle_bf16_to_f64(((const uint16_t *)p)[idx]);
}

/* Operand storage.  op(A) is the M x K matrix the product uses and op(B)
 * the K x N one:
 *   op_a == 0: element (i,k) of op(A) is A[i*lda + k]  (A stored M x K)
 *   op_a == 1: element (i,k) of op(A) is A[k*lda + i]  (A stored K x M)
 *   op_b == 0: element (k,j) of op(B) is B[k*ldb + j]  (B stored K x N)
 *   op_b == 1: element (k,j) of op(B) is B[j*ldb + k]  (B stored N x K)
 * op_b == 1 with ldb == K is the column-major B of the m.lqnn.cn SGEMM
 * article, section 3.1 (its baseline kernel indexes B[k + col*K]); op_a == 1
 * is the same storage for A. */
static int64_t a_index(int op_a, int64_t i, int64_t k, int64_t lda)
{
    return op_a ? k * lda + i : i * lda + k;
}

static int64_t b_index(int op_b, int64_t k, int64_t j, int64_t ldb)
{
    return op_b ? j * ldb + k : k * ldb + j;
}

/* Computes rows rows[0..nrows-1] of C = op(A) . op(B) and of S (all M rows
 * in order when rows is NULL; then nrows must equal M).  Output row r (the
 * r-th requested row) is written to C[r*ldc ...] and S[r*ldc ...]; S may be
 * NULL.  Returns 0, or -1 on invalid arguments.  K == 0 yields C = S = 0. */
int oracle_gemm_op_rows(int dtype, int op_a, int op_b, int M, int N, int K,
                        const void *A, int64_t lda, const void *B, int64_t ldb,
                        int nrows, const int64_t *rows,
                        double *C, double *S, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || dtype < 0 || dtype > 2)
        return -1;
    if ((op_a != 0 && op_a != 1) || (op_b != 0 && op_b != 1))
        return -1;
    if (rows == NULL && nrows != M)
        return -1;
    if (K > 0 && (lda < (op_a ? M : K) || ldb < (op_b ? K : N)))
        return -1;
    if (ldc < N)
        return -1;
    for (int r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M)
            return -1;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        double *c = C + (int64_t)r * ldc;
        double *s = S ? S + (int64_t)r * ldc : NULL;
        for (int j = 0; j < N; ++j) {
            c[j] = 0.0;
            if (s) s[j] = 0.0;
        }
        for (int k = 0; k < K; ++k) {
            double a = load_elem(dtype, A, a_index(op_a, i, k, lda));
            for (int j = 0; j < N; ++j) {
                double prod = a * load_elem(dtype, B, b_index(op_b, k, j, ldb));
                c[j] += prod;
                if (s) s[j] += fabs(prod);
            }
        }
    }
    return 0;
}

/* Both operands as stored (op_a = op_b = 0). */
int oracle_gemm_rows(int dtype, int M, int N, int K,
                     const void *A, int64_t lda, const void *B, int64_t ldb,
                     int nrows, const int64_t *rows,
                     double *C, double *S, int64_t ldc)
{
    return oracle_gemm_op_rows(dtype, 0, 0, M, N, K, A, lda, B, ldb, nrows, rows, C, S, ldc);
}

/* The scaled update C_out = alpha * (op(A) . op(B)) + beta * C_in.  The m.lqnn.cn
 * SGEMM article's tiled kernel sgemm_tile_v2 takes alpha and beta arguments
 * (its listing leaves the beta term out), and the GB300 roadmap (m.nxbn.cn,
 * section 7.1) argues for fusing such epilogue work into the GEMM.  Read as
 * the usual BLAS convention: with beta == 0 the old C is not read (any
 * value, NaN included, is ignored).  Everything in double:
 *   C_out[r][j] = alpha * sum_k A[i][k] B[k][j] + beta * C_in[i][j]
 *   S_out[r][j] = |alpha| * sum_k |A[i][k] B[k][j]| + |beta| * |C_in[i][j]|
 * (S is the scale of the normalised error).  C_in has the element type
 * `dtype` and leading dimension ldc_in; output row r is requested row i.
 * Returns 0, or -1 on invalid arguments. */
int oracle_gemm_scaled_op_rows(int dtype, int op_a, int op_b, int M, int N, int K,
                               double alpha, const void *A, int64_t lda,
                               const void *B, int64_t ldb,
                               double beta, const void *C_in, int64_t ldc_in,
                               int nrows, const int64_t *rows,
                               double *C_out, double *S_out, int64_t ldc)
{
    if (beta != 0.0 && (C_in == NULL || ldc_in < N))
        return -1;
    int rc = oracle_gemm_op_rows(dtype, op_a, op_b, M, N, K, A, lda, B, ldb, nrows, rows,
                                 C_out, S_out, ldc);
    if (rc != 0)
        return rc;
    for (int r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int j = 0; j < N; ++j) {
            double ab = C_out[(int64_t)r * ldc + j];
            double c = beta != 0.0 ? load_elem(dtype, C_in, i * ldc_in + j) : 0.0;
            C_out[(int64_t)r * ldc + j] = alpha * ab + beta * c;
            if (S_out)
                S_out[(int64_t)r * ldc + j] = fabs(alpha) * S_out[(int64_t)r * ldc + j] + fabs(beta) * fabs(c);
        }
    }
    return 0;
}

/* Both operands as stored (op_a = op_b = 0). */
int oracle_gemm_scaled_rows(int dtype, int M, int N, int K, double alpha,
                            const void *A, int64_t lda, const void *B, int64_t ldb,
                            double beta, const void *C_in, int64_t ldc_in,
                            int nrows, const int64_t *rows,
                            double *C_out, double *S_out, int64_t ldc)
{
    return oracle_gemm_scaled_op_rows(dtype, 0, 0, M, N, K, alpha, A, lda, B, ldb, beta,
                                      C_in, ldc_in, nrows, rows, C_out, S_out, ldc);
}

/* Number of threads the parallel loop above uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
