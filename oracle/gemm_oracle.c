/*
 * gemm_oracle.c -- CPU oracle for the row-major FP32 matrix multiply C = A x B.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this library. The CUDA library never links, calls or
 * includes it, and the two share no code, header, table or helper.
 *
 * What it computes (the plain definition, written out):
 *
 *   for every row i < M and column j < N:
 *       acc = +0.0f                                   (an FP32 accumulator)
 *       for k = 0, 1, ..., K-1, in ascending order:
 *           acc = acc + A[i*K + k] * B[k*N + j]
 *       C[i*N + j] = acc
 *
 * Sources:
 *   - page "GEMM 커널 테스트 코드 작성 및 최적화 (1024^3 크기 실험)":
 *       section "메모리 레이아웃" fixes the row-major layout and the three index
 *       formulas A[row*K+k], B[k*N+col], C[row*N+col];
 *       section "Naive GEMM 커널 동작 방식" (and its "연산 흐름" paragraph) fixes
 *       one accumulator per C element, started at zero and updated once per k in
 *       ascending k, then stored;
 *       the settings list under "실험 목적" fixes the element type as FP32.
 *   - page "[AutoMine++] #2. 행렬 곱셈 구현 시행착오", section "직관적 구현 (by CPU)":
 *       the same i / j / k triple loop on the CPU with a `float` running sum.
 *
 * The pages leave one step open: whether `acc + a*b` rounds the product before
 * the add (a separate multiply and add) or not (a fused multiply-add). The CUDA
 * statement on the first page is contracted to a fused multiply-add by nvcc's
 * default settings; the C++ statement on the third page is not contracted by a
 * default MSVC or GCC -ffp-contract=off build. Both readings are provided:
 *
 *   T2S_ORACLE_MUL_ADD (0):  acc = fl(acc + fl(a*b))     -- two roundings
 *   T2S_ORACLE_FMA     (1):  acc = fl(acc + a*b)         -- one rounding (fmaf)
 *
 * This file must be compiled with -ffp-contract=off and without -ffast-math so
 * that mode 0 really rounds twice and no loop is re-associated or vectorised
 * across k. The only parallelism is over independent output elements (OpenMP
 * over rows, or over sampled elements), which cannot change any result.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define T2S_ORACLE_MUL_ADD 0
#define T2S_ORACLE_FMA 1

/* One output element, exactly as the definition above states it. */
static float dot_row_col(int64_t N, int64_t K, const float *A, const float *B,
                         int64_t i, int64_t j, int mode)
{
    float acc = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        const float a = A[i * K + k];
        const float b = B[k * N + j];
        if (mode == T2S_ORACLE_FMA) {
            acc = fmaf(a, b, acc);
        } else {
            const float p = a * b; /* rounded to FP32 here */
            acc = acc + p;         /* and rounded again here */
        }
    }
    return acc;
}

/* Number of host threads the oracle runs on. */
int t2s_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of host threads (<= 0 leaves the OpenMP default). */
void t2s_oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Full product: C (M x N) = A (M x K) x B (K x N), all row-major FP32.
 * Returns 0, or -1 if a dimension is negative or mode is unknown.
 */
int t2s_oracle_sgemm(int64_t M, int64_t N, int64_t K, const float *A,
                     const float *B, float *C, int mode)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (mode != T2S_ORACLE_MUL_ADD && mode != T2S_ORACLE_FMA) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            C[i * N + j] = dot_row_col(N, K, A, B, i, j, mode);
        }
    }
    return 0;
}

/*
 * Sampled product: out[s] = C[rows[s], cols[s]] for s < n_samples, each element
 * computed by the same definition as the full product. For checking a large
 * product element by element without computing all of it.
 * Returns 0, or -1 on a bad argument (negative sizes, an index out of range,
 * unknown mode).
 */
int t2s_oracle_sgemm_at(int64_t M, int64_t N, int64_t K, const float *A,
                        const float *B, int64_t n_samples, const int64_t *rows,
                        const int64_t *cols, float *out, int mode)
{
    if (M < 0 || N < 0 || K < 0 || n_samples < 0) return -1;
    if (mode != T2S_ORACLE_MUL_ADD && mode != T2S_ORACLE_FMA) return -1;
    for (int64_t s = 0; s < n_samples; ++s) {
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < n_samples; ++s) {
        out[s] = dot_row_col(N, K, A, B, rows[s], cols[s], mode);
    }
    return 0;
}

/*
 * Row block: C[r0:r1, :] of the full product into out ((r1-r0) x N, row-major).
 * The CPU-baseline timing runs the oracle on a bounded row block of a large
 * workload through this entry. Returns 0 or -1 on a bad argument.
 */
int t2s_oracle_sgemm_rows(int64_t M, int64_t N, int64_t K, const float *A,
                          const float *B, int64_t r0, int64_t r1, float *out,
                          int mode)
{
    if (M < 0 || N < 0 || K < 0 || r0 < 0 || r1 < r0 || r1 > M) return -1;
    if (mode != T2S_ORACLE_MUL_ADD && mode != T2S_ORACLE_FMA) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = r0; i < r1; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            out[(i - r0) * N + j] = dot_row_col(N, K, A, B, i, j, mode);
        }
    }
    return 0;
}

/*
 * Vector add z = x + y, the memory-bound example of page "4주차: Roofline과 Tiling",
 * section "1. Arithmetic Intensity", example "Vector Add": one FP32 add per element,
 * reading x and y and writing z (12 bytes per element, AI = 1/12 FLOP/B).
 * Returns 0, or -1 if n is negative.
 */
int t2s_oracle_vector_add(int64_t n, const float *x, const float *y, float *z)
{
    if (n < 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        z[i] = x[i] + y[i];
    }
    return 0;
}

/*
 * Element types other than FP32. The pages write both kernels for a template element
 * type T (page "GEMM 커널 테스트 코드 작성 및 최적화 (1024^3 크기 실험)", sections
 * "Naive GEMM 커널 동작 방식" and "Shared Memory Tiled GEMM 연산 방식"); the oracle
 * gives the same definition for two more types.
 *
 * bfloat16 operands. A bfloat16 number is stored as the upper 16 bits of the IEEE
 * binary32 encoding of the same number: 1 sign bit, the 8 binary32 exponent bits and the
 * top 7 fraction bits (the format of Google's TPUs and of Intel's "BFLOAT16 - Hardware
 * Numerics Definition", 2018). Widening to binary32 is therefore exact: the 16 bits become
 * the high half of the binary32 encoding and the low half is zero. The product of two
 * bfloat16 numbers has at most 16 significant bits and fits binary32 exactly, so the
 * definition with bfloat16 inputs and an FP32 accumulator is the FP32 definition above
 * applied to the widened inputs (and MUL_ADD and FMA agree on it).
 * Returns 0, or -1 if n is negative.
 */
int t2s_oracle_bf16_to_f32(int64_t n, const uint16_t *x, float *y)
{
    if (n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t bits = (uint32_t)x[i] << 16;
        memcpy(&y[i], &bits, sizeof(float));
    }
    return 0;
}

/*
 * IEEE 754 binary16 operands: 1 sign bit, 5 exponent bits (bias 15) and 10 fraction bits.
 * Exponent field e = 0 encodes zero and the subnormal numbers f * 2^-24; 1 <= e <= 30 the
 * normal numbers (1 + f / 1024) * 2^(e - 15); e = 31 infinity (f = 0) or NaN (f != 0).
 * Every binary16 value, subnormals included, is exact in binary32, and so is the product of
 * two of them (at most 22 significant bits, magnitudes between 2^-48 and 2^32), so the FP16
 * definition with an FP32 accumulator is again the FP32 definition on the widened inputs.
 * The value is built here from the fields with ldexp (exact); a NaN keeps its sign.
 * Returns 0, or -1 if n is negative.
 */
int t2s_oracle_f16_to_f32(int64_t n, const uint16_t *x, float *y)
{
    if (n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const unsigned sign = (x[i] >> 15) & 1u;
        const int e = (x[i] >> 10) & 0x1f;
        const unsigned f = x[i] & 0x3ffu;
        double v;
        if (e == 0) {
            v = ldexp((double)f, -24);
        } else if (e == 31) {
            v = f == 0 ? INFINITY : NAN;
        } else {
            v = ldexp(1.0 + (double)f / 1024.0, e - 15);
        }
        y[i] = (float)(sign ? -v : v);
    }
    return 0;
}

/* One FP64 output element: the definition at the top with T = double. */
static double dot_row_col_f64(int64_t N, int64_t K, const double *A, const double *B,
                              int64_t i, int64_t j, int mode)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = A[i * K + k];
        const double b = B[k * N + j];
        if (mode == T2S_ORACLE_FMA) {
            acc = fma(a, b, acc);
        } else {
            const double p = a * b; /* rounded to FP64 here */
            acc = acc + p;          /* and rounded again here */
        }
    }
    return acc;
}

/*
 * FP64 full product: C (M x N) = A (M x K) x B (K x N), row-major binary64, one FP64
 * accumulator per element in ascending k (the FP32 definition with T = double).
 * Returns 0, or -1 if a dimension is negative or mode is unknown.
 */
int t2s_oracle_dgemm(int64_t M, int64_t N, int64_t K, const double *A, const double *B,
                     double *C, int mode)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (mode != T2S_ORACLE_MUL_ADD && mode != T2S_ORACLE_FMA) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            C[i * N + j] = dot_row_col_f64(N, K, A, B, i, j, mode);
        }
    }
    return 0;
}

/*
 * FP64 sampled product: out[s] = C[rows[s], cols[s]], each by the FP64 definition.
 * Returns 0, or -1 on a bad argument (negative sizes, an index out of range, unknown mode).
 */
int t2s_oracle_dgemm_at(int64_t M, int64_t N, int64_t K, const double *A, const double *B,
                        int64_t n_samples, const int64_t *rows, const int64_t *cols,
                        double *out, int mode)
{
    if (M < 0 || N < 0 || K < 0 || n_samples < 0) return -1;
    if (mode != T2S_ORACLE_MUL_ADD && mode != T2S_ORACLE_FMA) return -1;
    for (int64_t s = 0; s < n_samples; ++s) {
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < n_samples; ++s) {
        out[s] = dot_row_col_f64(N, K, A, B, rows[s], cols[s], mode);
    }
    return 0;
}
