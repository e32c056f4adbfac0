// gemm_simple.cu -- the two comparison kernels of page "GEMM 커널 테스트 코드 작성
// 및 최적화 (1024^3 크기 실험)".
//
// naive : section "Naive GEMM 커널 동작 방식" and "쓰레드 매핑" -- one thread per
//         C element, 16 x 16 blocks, the k loop reads A and B from global memory.
// smem32: section "Shared Memory Tiled GEMM 연산 방식", "타일 개념", "타일 로딩
//         단계" -- 32 x 32 blocks; per K tile each thread stages one element of
//         A and one of B in shared memory (zeros outside the matrices), a block
//         barrier, 32 multiply-adds from shared memory, a second barrier.
//
// Both are templates over the element type T, as on the page: T = float accumulates with
// fmaf in ascending k (bit-identical to each other and to the FP32 product kernel), T = double
// with fma in ascending k (bit-identical to the FP64 product kernel). Index arithmetic is
// 64-bit.
#include <cuda_runtime.h>

#include "t2s_internal.h"

namespace t2s {
namespace {

// One IEEE fused multiply-add (a single rounding) in the element type.
__device__ __forceinline__ float fma_rn(float a, float b, float c) { return __fmaf_rn(a, b, c); }
__device__ __forceinline__ double fma_rn(double a, double b, double c) { return __fma_rn(a, b, c); }

template <class T>
__global__ void __launch_bounds__(256) naive_kernel(int64_t M, int64_t N, int64_t K,
                                                    const T* __restrict__ A,
                                                    const T* __restrict__ B,
                                                    T* __restrict__ C) {
  const int64_t col = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (col >= N) return;
  // Row blocks beyond the grid's 65535-block y extent are taken in a grid-stride loop.
  for (int64_t row = static_cast<int64_t>(blockIdx.y) * blockDim.y + threadIdx.y; row < M;
       row += static_cast<int64_t>(gridDim.y) * blockDim.y) {
    const T* a = A + row * K;
    const T* b = B + col;
    T acc = T(0);
    for (int64_t k = 0; k < K; ++k) acc = fma_rn(a[k], b[k * N], acc);
    C[row * N + col] = acc;
  }
}

constexpr int kTile = 32;

template <class T>
__global__ void __launch_bounds__(kTile* kTile) smem32_kernel(int64_t M, int64_t N, int64_t K,
                                                              const T* __restrict__ A,
                                                              const T* __restrict__ B,
                                                              T* __restrict__ C) {
  __shared__ T As[kTile][kTile];
  __shared__ T Bs[kTile][kTile];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kTile + tx;
  const int64_t tiles = (K + kTile - 1) / kTile;
  // Row tiles beyond the grid's y extent are taken in a block-uniform grid-stride loop.
  for (int64_t rt = blockIdx.y; rt * kTile < M; rt += gridDim.y) {
    const int64_t row = rt * kTile + ty;
    T acc = T(0);
    for (int64_t t = 0; t < tiles; ++t) {
      const int64_t ka = t * kTile + tx;  // column of A this thread stages
      const int64_t kb = t * kTile + ty;  // row of B this thread stages
      As[ty][tx] = (row < M && ka < K) ? A[row * K + ka] : T(0);
      Bs[ty][tx] = (kb < K && col < N) ? B[kb * N + col] : T(0);
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kTile; ++k) acc = fma_rn(As[ty][k], Bs[k][tx], acc);
      __syncthreads();
    }
    if (row < M && col < N) C[row * N + col] = acc;
  }
}

template <class T>
cudaError_t run_naive(int64_t M, int64_t N, int64_t K, const T* A, const T* B, T* C,
                      cudaStream_t stream) {
  const dim3 block(16, 16);
  const int64_t gy = (M + 15) / 16;
  const dim3 grid(static_cast<unsigned>((N + 15) / 16), static_cast<unsigned>(gy < 65535 ? gy : 65535));
  naive_kernel<T><<<grid, block, 0, stream>>>(M, N, K, A, B, C);
  return cudaGetLastError();
}

template <class T>
cudaError_t run_smem32(int64_t M, int64_t N, int64_t K, const T* A, const T* B, T* C,
                       cudaStream_t stream) {
  const dim3 block(kTile, kTile);
  const int64_t gy = (M + kTile - 1) / kTile;
  const dim3 grid(static_cast<unsigned>((N + kTile - 1) / kTile),
                  static_cast<unsigned>(gy < 65535 ? gy : 65535));
  smem32_kernel<T><<<grid, block, 0, stream>>>(M, N, K, A, B, C);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_naive(const Problem& p) {
  return run_naive<float>(p.M, p.N, p.K, p.A, p.B, p.C, p.stream);
}

cudaError_t launch_smem32(const Problem& p) {
  return run_smem32<float>(p.M, p.N, p.K, p.A, p.B, p.C, p.stream);
}

cudaError_t launch_naive_f64(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                             double* C, cudaStream_t stream) {
  return run_naive<double>(M, N, K, A, B, C, stream);
}

cudaError_t launch_smem32_f64(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                              double* C, cudaStream_t stream) {
  return run_smem32<double>(M, N, K, A, B, C, stream);
}

}  // namespace t2s
