// gemm_16bit.cu -- C (FP32) = A x B with 16-bit floating-point inputs (bfloat16 or IEEE
// binary16) on the tcgen05 tensor cores.
//
// The element type of the operands is a template parameter on the pages' kernels; these are
// the 16-bit cases on the tensor cores of GB300 (kind::f16 with BF16 or FP16 operands, FP32
// accumulation). Products of two BF16 or two FP16 values are exact in FP32, so the result
// differs from the FP32 definition applied to the widened values only by the order of the
// FP32 additions.
//
// 1. Operands. A (M x K, row-major) is K-major for the tensor core and is read in place by TMA
//    when its rows are a multiple of 16 bytes (K % 8 == 0) and it is 16-byte aligned;
//    otherwise it is first copied into an M x Kp plane (Kp = ceil(K / 64) x 64, zeros beyond
//    K). B (K x N, row-major) is MN-major for the tensor core; when N % 8 == 0 and B is
//    16-byte aligned it too is read in place (128-byte-swizzled MN-major atoms), otherwise it
//    is first transposed into an N x Kp K-major plane.
// 2. The persistent tcgen05 kernel of tc_gemm.cuh: 64- or 128-deep k blocks of MMAs with
//    K = 16, K chunks of 2048 accumulated in TMEM and added into FP32 registers with
//    round-to-nearest by the epilogue warps. With B in place and more than one 128-row tile
//    row, pairs of CTAs on two SMs run 256-row tiles with .cta_group::2 MMAs; the widest of
//    them, 256 x 512, sum all of K in TMEM (K <= 16384).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "t2s_device.cuh"
#include "t2s_internal.h"
#include "t2s_tmap.h"
#include "tc_gemm.cuh"

namespace t2s {
namespace {

constexpr int64_t kKPad16 = 64;

int64_t padded_k16(int64_t K) { return (K + kKPad16 - 1) / kKPad16 * kKPad16; }

size_t up256b(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// B (K x N, 16-bit, row-major) -> Bt (N x Kp), zeros for k >= K; 32 x 32 tiles through shared
// memory so that reads (along n) and writes (along k) are coalesced.
__global__ void __launch_bounds__(256) transpose_16bit_kernel(const uint16_t* __restrict__ B,
                                                              uint16_t* __restrict__ Bt,
                                                              int64_t K, int64_t N, int64_t Kp) {
  __shared__ uint16_t tile[32][34];
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 32;
  for (int64_t kt = blockIdx.y; kt * 32 < Kp; kt += gridDim.y) {
    const int64_t k0 = kt * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t k = k0 + ty + 8 * i, n = n0 + tx;
      tile[ty + 8 * i][tx] = (k < K && n < N) ? B[k * N + n] : static_cast<uint16_t>(0);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = n0 + ty + 8 * i, k = k0 + tx;
      if (n < N) Bt[n * Kp + k] = tile[tx][ty + 8 * i];
    }
    __syncthreads();
  }
}

// A (M x K, 16-bit) -> Ap (M x Kp), zeros for k >= K.
__global__ void __launch_bounds__(256) pad_rows_16bit_kernel(const uint16_t* __restrict__ A,
                                                             uint16_t* __restrict__ Ap,
                                                             int64_t M, int64_t K, int64_t Kp) {
  const int64_t total = M * Kp;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / Kp, k = i % Kp;
    Ap[i] = k < K ? A[row * K + k] : static_cast<uint16_t>(0);
  }
}

// K values the tensor core sums from zero before the epilogue adds them into the FP32 sums
// (shorter chunks measured 3-5 % slower; error at K = 4096: 4.0e-4 against a bound of 4.1e-3).
constexpr int kHalfChunkK = 2048;
// Longest K for the 512-wide pair tiles, whose tensor cores sum all of K without the
// round-to-nearest chunk additions (error at K = 8192: 2.0e-3 against a bound of 8.2e-3).
constexpr int64_t kWideMaxK = 16384;

// The configurations of one 16-bit format (tc::kBf16 or tc::kF16). Tile widths BN (M is 128
// per CTA), BK = 64 (128-byte rows) unless stated: wider tiles read A less per FLOP.
template <int KIND>
struct HalfConfigs {
  static constexpr int C = kHalfChunkK;
  // B as a transposed K-major plane.
  using T128 = tc::TcConfig<KIND, 128, 64, 6, C>;  // 6 stages of 32 KB
  using T192 = tc::TcConfig<KIND, 192, 64, 4, C>;  // 4 stages of 40 KB
  using T224 = tc::TcConfig<KIND, 224, 64, 4, C>;  // 4 stages of 44 KB
  using T256 = tc::TcConfig<KIND, 256, 64, 4, C>;  // 4 stages of 48 KB
  // B read in place (MN-major): whole 64-column atoms.
  using M128 = tc::TcConfig<KIND, 128, 64, 6, C, true>;
  using M192 = tc::TcConfig<KIND, 192, 64, 4, C, true>;
  using M256 = tc::TcConfig<KIND, 256, 64, 4, C, true>;
  // Pairs of CTAs on two SMs, 256-row tiles; each CTA stages 128 rows of A and half of B, in
  // 128-deep K blocks: each stage costs a barrier round trip between the producer, the MMA
  // issuer and the peer, and 64-deep blocks with the same bytes in flight ran slower (4096^3:
  // 1171 against 1283 TFLOP/s for the 256-wide pair, 825 against 1060 for the 128-wide one).
  using P128 = tc::TcConfig<KIND, 128, 128, 4, C, true, true>;  // 4 stages of 48 KB
  using P256 = tc::TcConfig<KIND, 256, 128, 3, C, true, true>;
  // 256 x 512 pair tiles: two N = 256 MMAs per k step into one 512-column accumulator, the
  // tensor core summing all of K; 4 stages of 48 KB (64-deep K blocks).
  // 128-deep blocks in 2 stages of 96 KB ran slower (8192^3: 1625 against 1824 TFLOP/s).
  using P512 = tc::TcConfig<KIND, 512, 64, 4, C, true, true, true>;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Index of the width (of `n` candidates) with the fewest balanced persistent rounds, weighted
// for the narrower tiles' extra operand traffic.
int pick_width(int64_t M, int64_t N, int sms, const int* widths, const double* weight, int n) {
  const int64_t tm = (M + 127) / 128;
  int best = 0;
  double best_cost = 0.0;
  for (int i = 0; i < n; ++i) {
    const int64_t tiles = tm * ((N + widths[i] - 1) / widths[i]);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const double cost = static_cast<double>(rounds) * widths[i] * weight[i];
    if (i == 0 || cost < best_cost) {
      best = i;
      best_cost = cost;
    }
  }
  return best;
}

template <int KIND>
cudaError_t launch_half(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                        float* C, void* workspace, cudaStream_t stream, unsigned* status) {
  using Cf = HalfConfigs<KIND>;
  const int64_t Kp = padded_k16(K);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint16_t* bt = reinterpret_cast<uint16_t*>(w);
  uint16_t* ap = reinterpret_cast<uint16_t*>(w + up256b(static_cast<size_t>(N) * Kp * 2));
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool a_in_place = K % 8 == 0 && aligned16(A);
  const uint16_t* a = A;
  int64_t lda = K;
  if (!a_in_place) {
    const int64_t work = M * Kp;
    const int64_t blocks = std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(sms) * 16);
    pad_rows_16bit_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(A, ap, M, K, Kp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    a = ap;
    lda = Kp;
  }
  Problem p{M, N, K, nullptr, nullptr, C, stream, status};
  if (N % 8 == 0 && aligned16(B)) {
    // Weights: measured time of one persistent round per unit of tile area, relative to the
    // 256-wide pair (4096^3: 18.5 us per round of 256 x 128 pair tiles, 26.8 of 128 x 192
    // single-SM tiles, 26.8 of 256 x 256 pair tiles, 45.4 of 256 x 512 pair tiles).
    const int widths[4] = {128, 192, 256, 512};
    const double weight[4] = {1.38, 1.33, 1.0, 0.85};
    // Pairs need two tile rows; 192 columns are three boxes and cannot be split in two.
    const int n_widths = (M > 128 && K <= kWideMaxK) ? 4 : 3;
    const int best = pick_width(M, N, sms, widths, weight, n_widths);
    if (M > 128) {
      switch (best) {
        case 1: return tc::run_tc<typename Cf::M192>(p, a, nullptr, B, nullptr, lda, N, Kp);
        case 2: return tc::run_tc<typename Cf::P256>(p, a, nullptr, B, nullptr, lda, N, Kp);
        case 3: return tc::run_tc<typename Cf::P512>(p, a, nullptr, B, nullptr, lda, N, Kp);
        default: return tc::run_tc<typename Cf::P128>(p, a, nullptr, B, nullptr, lda, N, Kp);
      }
    }
    switch (best) {
      case 1: return tc::run_tc<typename Cf::M192>(p, a, nullptr, B, nullptr, lda, N, Kp);
      case 2: return tc::run_tc<typename Cf::M256>(p, a, nullptr, B, nullptr, lda, N, Kp);
      default: return tc::run_tc<typename Cf::M128>(p, a, nullptr, B, nullptr, lda, N, Kp);
    }
  }
  {
    const int64_t gy = Kp / 32;
    const dim3 grid(static_cast<unsigned>((N + 31) / 32),
                    static_cast<unsigned>(gy < 65535 ? gy : 65535));
    transpose_16bit_kernel<<<grid, dim3(32, 8), 0, stream>>>(B, bt, K, N, Kp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Width by balanced persistent rounds, as for the 3xTF32 kernel.
  const int widths[4] = {128, 192, 224, 256};
  const double weight[4] = {1.15, 1.03, 1.01, 1.0};
  const int best = pick_width(M, N, sms, widths, weight, 4);
  switch (best) {
    case 1: return tc::run_tc<typename Cf::T192>(p, a, nullptr, bt, nullptr, lda, Kp, Kp);
    case 2: return tc::run_tc<typename Cf::T224>(p, a, nullptr, bt, nullptr, lda, Kp, Kp);
    case 3: return tc::run_tc<typename Cf::T256>(p, a, nullptr, bt, nullptr, lda, Kp, Kp);
    default: return tc::run_tc<typename Cf::T128>(p, a, nullptr, bt, nullptr, lda, Kp, Kp);
  }
}

}  // namespace

// Bt plane (N x Kp) and, when A cannot be read in place, an A plane (M x Kp): 2 bytes each,
// both counted so the size does not depend on the pointers.
size_t half_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int64_t Kp = padded_k16(K);
  return up256b(static_cast<size_t>(N) * Kp * 2) + up256b(static_cast<size_t>(M) * Kp * 2);
}

cudaError_t launch_bf16(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                        float* C, void* workspace, cudaStream_t stream, unsigned* status) {
  return launch_half<tc::kBf16>(M, N, K, A, B, C, workspace, stream, status);
}

cudaError_t launch_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                       float* C, void* workspace, cudaStream_t stream, unsigned* status) {
  return launch_half<tc::kF16>(M, N, K, A, B, C, workspace, stream, status);
}

}  // namespace t2s
