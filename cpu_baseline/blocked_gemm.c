/*
 * blocked_gemm.c -- a cache-blocked, multi-core CPU implementation of the row-major FP32
 * product C = A x B: the stronger CPU baseline that the bench reports beside the plain
 * oracle. It is a baseline only; nothing checks results against it.
 *
 * Why (page "[AutoMine++] #2. 행렬 곱셈 구현 시행착오", section "직관적 구현 (by CPU)"):
 * after timing the literal triple loop at about 16-17 s for 1024^3, the page notes that
 * raising the cache hit rate and putting every core to work would make it far faster. This
 * file does both. Its blocking is the CPU form of the tiling on page "4주차: Roofline과
 * Tiling", section "3. Tiling": tiles staged in fast memory and reused there.
 *
 *   - C is cut into MC x NC tiles, shared out over the OpenMP threads (every core in the
 *     process's affinity mask);
 *   - K is walked in KC-long chunks, ascending; for each chunk the thread copies the MC x KC
 *     block of A and the KC x NC block of B into contiguous panels (MR-row strips of A,
 *     NR-column strips of B, zero-padded at the edges of M and N) that stay in its L2;
 *   - an MR x NR register block of C is updated by one fused multiply-add per element and k,
 *     k ascending, and stored back after each chunk (an FP32 value stored and reloaded is the
 *     same value).
 *
 * Every element of C is therefore the chain acc = fmaf(A[i][k], B[k][j], acc) for k = 0, 1,
 * ..., K-1 starting from +0.0f: the fused-multiply-add reading of the definition, bit for bit.
 * Padding rows and columns are computed on zeros and never stored. Compile with
 * -ffp-contract=off and without -ffast-math, so that nothing is re-associated; the compiler
 * may vectorise the j loop (independent elements), which changes no result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define MR 6
#define NR 16
#define MC 96  /* a multiple of MR */
#define NC 256 /* a multiple of NR */
#define KC 256

int t2s_cpu_blocked_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void t2s_cpu_blocked_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Copies rows [i0, i0 + mc) x k in [p0, p0 + kc) of A into strips of MR rows:
 * ap[s][k][r] = A[i0 + s*MR + r][p0 + k], zero for rows at or past M. */
static void pack_a(int64_t M, int64_t K, const float *A, int64_t i0, int64_t mc, int64_t p0,
                   int64_t kc, float *ap)
{
    for (int64_t s = 0; s < mc; s += MR) {
        for (int64_t k = 0; k < kc; ++k) {
            for (int r = 0; r < MR; ++r) {
                const int64_t i = i0 + s + r;
                *ap++ = (i < M) ? A[i * K + p0 + k] : 0.0f;
            }
        }
    }
}

/* Copies k in [p0, p0 + kc) x columns [j0, j0 + nc) of B into strips of NR columns:
 * bp[s][k][c] = B[p0 + k][j0 + s*NR + c], zero for columns at or past N. */
static void pack_b(int64_t N, const float *B, int64_t p0, int64_t kc, int64_t j0, int64_t nc,
                   float *bp)
{
    for (int64_t s = 0; s < nc; s += NR) {
        for (int64_t k = 0; k < kc; ++k) {
            const float *row = B + (p0 + k) * N + j0 + s;
            const int64_t valid = N - (j0 + s);
            if (valid >= NR) {
                memcpy(bp, row, NR * sizeof(float));
            } else {
                for (int c = 0; c < NR; ++c) bp[c] = (c < valid) ? row[c] : 0.0f;
            }
            bp += NR;
        }
    }
}

/* acc[r][c] = fmaf(ap[k][r], bp[k][c], acc[r][c]) for k = 0 .. kc-1 in order. */
static void micro_kernel(int64_t kc, const float *restrict ap, const float *restrict bp,
                         float acc[MR][NR])
{
    float c[MR][NR];
    for (int r = 0; r < MR; ++r)
        for (int j = 0; j < NR; ++j) c[r][j] = acc[r][j];
    for (int64_t k = 0; k < kc; ++k) {
        const float *a = ap + k * MR;
        const float *b = bp + k * NR;
        for (int r = 0; r < MR; ++r) {
            const float ar = a[r];
            for (int j = 0; j < NR; ++j) c[r][j] = fmaf(ar, b[j], c[r][j]);
        }
    }
    for (int r = 0; r < MR; ++r)
        for (int j = 0; j < NR; ++j) acc[r][j] = c[r][j];
}

/*
 * C (M x N) = A (M x K) x B (K x N), all row-major FP32, on every OpenMP thread.
 * Returns 0, -1 on a bad argument, -2 if a thread's panel buffers cannot be allocated.
 */
int t2s_cpu_blocked_sgemm(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                          float *C)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (K == 0) {
        for (int64_t i = 0; i < M * N; ++i) C[i] = 0.0f;
        return 0;
    }
    const int64_t tiles_m = (M + MC - 1) / MC, tiles_n = (N + NC - 1) / NC;
    int failed = 0;
#pragma omp parallel
    {
        float *ap = (float *)malloc(sizeof(float) * MC * KC);
        float *bp = (float *)malloc(sizeof(float) * KC * NC);
        if (ap == NULL || bp == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < tiles_m * tiles_n; ++t) {
            if (ap == NULL || bp == NULL) continue;
            /* Neighbouring tiles share their block of B: walk the tiles column-major. */
            const int64_t i0 = (t % tiles_m) * MC, j0 = (t / tiles_m) * NC;
            const int64_t mc = (M - i0 < MC) ? M - i0 : MC;
            const int64_t nc = (N - j0 < NC) ? N - j0 : NC;
            const int64_t mc_pad = (mc + MR - 1) / MR * MR, nc_pad = (nc + NR - 1) / NR * NR;
            for (int64_t p0 = 0; p0 < K; p0 += KC) {
                const int64_t kc = (K - p0 < KC) ? K - p0 : KC;
                pack_a(M, K, A, i0, mc_pad, p0, kc, ap);
                pack_b(N, B, p0, kc, j0, nc_pad, bp);
                for (int64_t jr = 0; jr < nc_pad; jr += NR) {
                    for (int64_t ir = 0; ir < mc_pad; ir += MR) {
                        float acc[MR][NR];
                        /* Resume the sums of the earlier chunks (zero before the first). */
                        for (int r = 0; r < MR; ++r) {
                            const int64_t i = i0 + ir + r;
                            for (int j = 0; j < NR; ++j) {
                                const int64_t col = j0 + jr + j;
                                acc[r][j] = (p0 > 0 && i < M && col < N) ? C[i * N + col] : 0.0f;
                            }
                        }
                        micro_kernel(kc, ap + ir * kc, bp + jr * kc, acc);
                        for (int r = 0; r < MR; ++r) {
                            const int64_t i = i0 + ir + r;
                            if (i >= M) break;
                            for (int j = 0; j < NR; ++j) {
                                const int64_t col = j0 + jr + j;
                                if (col < N) C[i * N + col] = acc[r][j];
                            }
                        }
                    }
                }
            }
        }
        free(ap);
        free(bp);
    }
    return failed ? -2 : 0;
}
