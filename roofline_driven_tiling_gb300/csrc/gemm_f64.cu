// gemm_f64.cu -- C = A x B in binary64 on the CUDA cores (the FP64 instance of the pages'
// template element type).
//
// Tiling as on page "4주차: Roofline과 Tiling", section "3. Tiling": a CTA computes a 32 x 32
// tile of C from 32 x 16 tiles of A and 16 x 32 tiles of B staged in shared memory, and each
// thread keeps a 2 x 2 block of C in registers. The next K tile is loaded into registers while
// the current one is multiplied (two shared-memory buffers, one barrier per K tile).
//
// GB300 executes 2 FP64 fused multiply-adds per SM per clock, 64 times fewer than FP32, so the
// FP64 ridge point is 1.26 TFLOP/s / 6.8 TB/s = 0.19 FLOP per byte: every tiling, even none,
// is far above it, larger tiles buy nothing, and the tile size is chosen for balance instead: 32 x 32 tiles make many small CTAs, so every SM ends the grid with nearly the same
// number of tiles (64 x 64 tiles lost 4% to the last partial wave at 2048^3).
//
// Every C element is summed with one IEEE fused multiply-add per k in ascending k, so the
// result is bit-identical to the FP64 naive and shared-memory kernels and to the definition
// evaluated with fma(). Index arithmetic is 64-bit; ragged edges are zero-filled on load and
// masked on store.
#include <cuda_runtime.h>

#include <cstdint>

#include "t2s_internal.h"

namespace t2s {
namespace {

constexpr int kBM = 32, kBN = 32, kBK = 16, kThreads = 256;
constexpr int kTM = 2, kTN = 2;                // C block per thread
constexpr int kLoadsA = kBM * kBK / kThreads;  // 2
constexpr int kLoadsB = kBK * kBN / kThreads;  // 2
static_assert((kBM / kTM) * (kBN / kTN) == kThreads, "one C block per thread");

__global__ void __launch_bounds__(kThreads) dgemm_kernel(int64_t M, int64_t N, int64_t K,
                                                         const double* __restrict__ A,
                                                         const double* __restrict__ B,
                                                         double* __restrict__ C) {
  // A tiles stored k-major (As[k][m]) so a thread's two rows are contiguous.
  __shared__ double As[2][kBK][kBM];
  __shared__ double Bs[2][kBK][kBN];
  const int t = threadIdx.x;
  const int ty = t / 16, tx = t % 16;  // rows 2*ty, 2*ty+1; columns tx, tx + 16
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;
  const int64_t ktiles = (K + kBK - 1) / kBK;

  for (int64_t mt = blockIdx.y; mt * kBM < M; mt += gridDim.y) {
    const int64_t m0 = mt * kBM;
    double ra[kLoadsA], rb[kLoadsB];
    // Global -> registers for K tile kt (zeros outside the matrices).
    auto fetch = [&](int64_t kt) {
#pragma unroll
      for (int i = 0; i < kLoadsA; ++i) {
        const int idx = t + kThreads * i;
        const int64_t m = m0 + idx / kBK, k = kt * kBK + idx % kBK;
        ra[i] = (m < M && k < K) ? A[m * K + k] : 0.0;
      }
#pragma unroll
      for (int i = 0; i < kLoadsB; ++i) {
        const int idx = t + kThreads * i;
        const int64_t k = kt * kBK + idx / kBN, n = n0 + idx % kBN;
        rb[i] = (k < K && n < N) ? B[k * N + n] : 0.0;
      }
    };
    auto store = [&](int buf) {
#pragma unroll
      for (int i = 0; i < kLoadsA; ++i) {
        const int idx = t + kThreads * i;
        As[buf][idx % kBK][idx / kBK] = ra[i];
      }
#pragma unroll
      for (int i = 0; i < kLoadsB; ++i) {
        const int idx = t + kThreads * i;
        Bs[buf][idx / kBN][idx % kBN] = rb[i];
      }
    };

    double acc[kTM][kTN];
#pragma unroll
    for (int i = 0; i < kTM; ++i)
#pragma unroll
      for (int j = 0; j < kTN; ++j) acc[i][j] = 0.0;

    if (ktiles > 0) {
      fetch(0);
      store(0);
    }
    __syncthreads();
    for (int64_t kt = 0; kt < ktiles; ++kt) {
      const int buf = static_cast<int>(kt & 1);
      if (kt + 1 < ktiles) fetch(kt + 1);
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
        double a[kTM], b[kTN];
#pragma unroll
        for (int i = 0; i < kTM; ++i) a[i] = As[buf][k][kTM * ty + i];
#pragma unroll
        for (int j = 0; j < kTN; ++j) b[j] = Bs[buf][k][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < kTM; ++i)
#pragma unroll
          for (int j = 0; j < kTN; ++j) acc[i][j] = __fma_rn(a[i], b[j], acc[i][j]);
      }
      // The other buffer was last read in iteration kt - 1, which every thread finished
      // before the barrier at the end of that iteration.
      if (kt + 1 < ktiles) store(buf ^ 1);
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kTM; ++i) {
      const int64_t m = m0 + kTM * ty + i;
      if (m >= M) break;
#pragma unroll
      for (int j = 0; j < kTN; ++j) {
        const int64_t n = n0 + tx + 16 * j;
        if (n < N) C[m * N + n] = acc[i][j];
      }
    }
    __syncthreads();  // the next row tile reuses buffer 0
  }
}

}  // namespace

cudaError_t launch_dgemm(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                         double* C, cudaStream_t stream) {
  const int64_t gy = (M + kBM - 1) / kBM;
  const dim3 grid(static_cast<unsigned>((N + kBN - 1) / kBN),
                  static_cast<unsigned>(gy < 65535 ? gy : 65535));
  dgemm_kernel<<<grid, kThreads, 0, stream>>>(M, N, K, A, B, C);
  return cudaGetLastError();
}

}  // namespace t2s
