/*
 * CPU oracle for C = alpha * op(A) @ op(B) + beta * C  (test infrastructure).
 *
 * This file is test infrastructure, not part of the product: only the tests,
 * the smoke check and the benchmark's CPU-baseline leg load it.  It shares no
 * code with the CUDA library.
 *
 * What it computes (the plain definition, nothing faster):
 *   - tensorcore gemm.md, "Surface": BLAS row-major layout,
 *     C[M,N] = alpha * A[M,K] @ B[K,N] + beta * C[M,N]; a leading dimension
 *     of 0 means "row-major contiguous".
 *   - Foundry metal.md, "GEMM / GEMV (via MPS)": the same formula in fp32.
 *   - phobos matmul page, "matmul" and "matmul_t": acc accumulates the
 *     products of A's rows with B's columns over k; matmul_t reads B stored
 *     [N,K] (a linear layer's weight), i.e. the transpose_b case.
 *   - phobos matmul page, "sgemm": the epilogue alpha*acc + beta*c_old.
 *
 * Every stored element is decoded exactly to a double (the IEEE-754 binary16
 * and bfloat16 encodings are decoded here from their definitions; binary32
 * widens exactly).  The k-sum runs in fp64, in ascending k.  Beside each
 * result R_ij the oracle returns T_ij = sum_k |A_ik * B_kj|, the scale that
 * the tolerance of a finite-precision GEMM is measured against.
 *
 * Reading where the pages are silent: beta == 0 means C_old is not read at
 * all (NaN in C does not propagate), and alpha == 0 is not special-cased.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fused
 * multiply-add contraction, so x86 and aarch64 give the same doubles).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element encodings understood by the oracle (ORACLE_I8: two's-complement
 * int8, the operand type of the tessl architecture.md "Integer GEMM"; its
 * products and their sums for K <= 131072 are integers below 2^53, so the
 * fp64 k-sum is exact) */
enum { ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_F32 = 3, ORACLE_I8 = 4 };

typedef struct {
    int64_t M, N, K;
    int32_t a_dtype, b_dtype, c_dtype;
    int32_t transpose_a, transpose_b;
    double alpha, beta;
    int64_t lda, ldb, ldc;        /* in elements; 0 = contiguous */
    const void *A, *B, *C;        /* stored bits; C may be NULL when beta == 0 */
} oracle_problem;

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = frac * 2^-24; exponent 31: inf / NaN. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * exponent 0: subnormal, value = frac * 2^-133; exponent 255: inf / NaN. */
double oracle_decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

static double load(const void *p, int32_t dtype, int64_t idx)
{
    switch (dtype) {
    case ORACLE_F16: return oracle_decode_f16(((const uint16_t *)p)[idx]);
    case ORACLE_BF16: return oracle_decode_bf16(((const uint16_t *)p)[idx]);
    case ORACLE_I8: return (double)((const int8_t *)p)[idx];
    default: return (double)((const float *)p)[idx];
    }
}

/* The leading-dimension default: 0 means the stored rows are contiguous. */
static void normalize(const oracle_problem *p, int64_t *lda, int64_t *ldb, int64_t *ldc)
{
    *lda = p->lda ? p->lda : (p->transpose_a ? p->M : p->K);
    *ldb = p->ldb ? p->ldb : (p->transpose_b ? p->K : p->N);
    *ldc = p->ldc ? p->ldc : p->N;
}

/* op(A)[i,k]: A stored [M,K], or [K,M] when transpose_a */
static int64_t a_index(const oracle_problem *p, int64_t lda, int64_t i, int64_t k)
{
    return p->transpose_a ? k * lda + i : i * lda + k;
}

/* op(B)[k,j]: B stored [K,N], or [N,K] when transpose_b */
static int64_t b_index(const oracle_problem *p, int64_t ldb, int64_t k, int64_t j)
{
    return p->transpose_b ? j * ldb + k : k * ldb + j;
}

/*
 * Full rows [row0, row1) of the result.  R and T are (row1-row0) x N,
 * row-major.  The loop is the i-k-j ordering of the definition: for each
 * output row, each k adds A[i,k] * B[k,:] into the row's running sums.
 */
int oracle_gemm_rows(const oracle_problem *p, int64_t row0, int64_t row1,
                     double *R, double *T)
{
    if (!p || row0 < 0 || row1 > p->M || row0 > row1) return 1;
    int64_t lda, ldb, ldc;
    normalize(p, &lda, &ldb, &ldc);
    const int64_t N = p->N, K = p->K;

    /* decode op(B) once into a K x N double matrix */
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!Bd) return 2;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j)
            Bd[k * N + j] = load(p->B, p->b_dtype, b_index(p, ldb, k, j));

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = row0; i < row1; ++i) {
        double *S = R + (i - row0) * N;
        double *Ta = T + (i - row0) * N;
        for (int64_t j = 0; j < N; ++j) { S[j] = 0.0; Ta[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double a = load(p->A, p->a_dtype, a_index(p, lda, i, k));
            const double *b = Bd + k * N;
            for (int64_t j = 0; j < N; ++j) {
                const double prod = a * b[j];
                S[j] += prod;
                Ta[j] += fabs(prod);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            double r = p->alpha * S[j];
            if (p->beta != 0.0)
                r += p->beta * load(p->C, p->c_dtype, i * ldc + j);
            S[j] = r;
        }
    }
    free(Bd);
    return 0;
}

/*
 * Single output elements (rows[t], cols[t]) for t < n: the same definition,
 * one dot product each, for spot checks of results too large to recompute.
 */
int oracle_gemm_points(const oracle_problem *p, int64_t n, const int64_t *rows,
                       const int64_t *cols, double *R, double *T)
{
    if (!p) return 1;
    int64_t lda, ldb, ldc;
    normalize(p, &lda, &ldb, &ldc);
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= p->M || cols[t] < 0 || cols[t] >= p->N) return 1;

#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double s = 0.0, ta = 0.0;
        for (int64_t k = 0; k < p->K; ++k) {
            const double prod = load(p->A, p->a_dtype, a_index(p, lda, i, k)) *
                                load(p->B, p->b_dtype, b_index(p, ldb, k, j));
            s += prod;
            ta += fabs(prod);
        }
        double r = p->alpha * s;
        if (p->beta != 0.0)
            r += p->beta * load(p->C, p->c_dtype, i * ldc + j);
        R[t] = r;
        T[t] = ta;
    }
    return 0;
}

/* decode n stored elements of the given encoding into doubles */
int oracle_decode_array(int32_t dtype, int64_t n, const void *src, double *dst)
{
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16 && dtype != ORACLE_F32 && dtype != ORACLE_I8) return 1;
    for (int64_t t = 0; t < n; ++t) dst[t] = load(src, dtype, t);
    return 0;
}

/* number of threads the OpenMP runtime will use (reported by the baseline) */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
