// gemm_tf32x3.cu -- C = A x B in FP32 on the tcgen05 tensor cores with 3xTF32 error
// compensation (Ootomo and Yokota, "Recovering single precision accuracy from Tensor Cores
// while surpassing the FP32 theoretical peak performance", 2022). Not on the pages; the
// operation is the same C = A x B as the product kernel.
//
// 1. Split pre-pass (one bandwidth-bound launch). Every x of A and B becomes
//      big = tf32(x), small = tf32(x - big)      (x - big is exact in FP32)
//    with tf32() = round to nearest even at 10 explicit mantissa bits (IEEE 754
//    rounding applied to the TF32 format, written from the definition below). The planes
//    are K-major with a padded row length Kp = ceil(K / 32) * 32 and zeros in the padding:
//      A_big, A_small : M x Kp      (A is already K-major: a row-wise copy)
//      B_big, B_small : N x Kp      (B is K x N row-major: transposed through shared memory)
//    so that every tensor-map stride is a multiple of 128 bytes whatever K and N are.
// 2. Product kernel, persistent: one CTA per SM (64 threads plus 4 epilogue warps per 128
//    columns of the tile: 320 threads at BN = 224) walks 128 x BN tiles of C; for large
//    products, clusters of two CTAs on two SMs walk 256 x BN tiles with cta_group::2 MMAs
//    (M 256, issued by the first CTA), each CTA staging half of the B planes.
//      warp 0     -- TMA producer: per K block, one box of each of the four planes;
//      warp 1     -- allocates TMEM, one lane issues tcgen05.mma kind::tf32 (M=128, N=BN,
//                    K=8), three per k step into one FP32 accumulator in TMEM, in the order
//                    small*big, big*small, big*big; tcgen05.commit frees each ring slot;
//      warps 2..  -- epilogue: tcgen05.ld of their 32 TMEM lanes (rows), stores to C.
//    TMEM holds two accumulators. The tensor core accumulates one K chunk (256 values) from
//    zero; the epilogue warps add each chunk's partial sums into FP32 registers with
//    round-to-nearest while the next chunk's MMAs run. The tensor core's internal FP32
//    accumulation does not round to nearest: summed over all of K in TMEM its error grows
//    faster than K and leaves the 1e-6 K max|a| max|b| bound at K = 8192; chunking keeps
//    that error to 256 values and lets it average out across chunks.
//    Shared-memory operands use the canonical K-major layout with the 128-byte (BK = 32) or
//    64-byte (BK = 16) swizzle the TMA writes, described to the tensor core by matrix
//    descriptors.
// The missing small*small term is below 2^-22 relative; the tensor core's own summation
// order within a chunk makes the result differ from the FP32 definition by rounding only.
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

constexpr int64_t kKPad = 32;

int64_t padded_k(int64_t K) { return (K + kKPad - 1) / kKPad * kKPad; }

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ------------------------------------------------------------------ split pre-pass
// Round a binary32 value to the TF32 format (1 sign, 8 exponent, 10 mantissa bits), round
// to nearest, ties to even, by integer arithmetic on the encoding: add half an ulp of the
// 10-bit mantissa (minus one, plus the lowest kept bit for the tie rule) and clear the 13
// dropped bits. A carry out of the mantissa correctly increments the exponent. NaN and
// infinity are passed through. A finite value within half a TF32 ulp of FLT_MAX
// (|x| >= 0x7F7FF000) would round up to infinity; it keeps its truncated value instead, the
// largest TF32 value of its sign, so that x - tf32(x) stays finite and exact and the
// correction term of the split carries the rest.
__device__ __forceinline__ float tf32_round(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7f800000u) == 0x7f800000u) return x;
  const uint32_t r = (u + 0x00000fffu + ((u >> 13) & 1u)) & 0xffffe000u;
  if ((r & 0x7f800000u) == 0x7f800000u) return __uint_as_float(u & 0xffffe000u);
  return __uint_as_float(r);
}

__device__ __forceinline__ void split(float x, float& big, float& small) {
  // The tensor core reads only the top 19 bits of an FP32 operand: a NaN whose payload lies
  // in the 13 low bits alone would read as an infinity, so NaNs become the quiet NaN.
  big = isnan(x) ? __uint_as_float(0x7fc00000u) : tf32_round(x);
  // x - big is exact; for non-finite x the correction term is dropped.
  small = isfinite(x) ? tf32_round(__fsub_rn(x, big)) : 0.0f;
}

// Both splits in one launch, their blocks interleaved (even blocks A, odd blocks B) so that
// the two run side by side: alone, neither kept HBM busy (about 5.6 and 4.2 TB/s).
//  * A (M x K, row-major) -> big, small (M x Kp), zeros for k >= K: work items of 256 x 4
//    consecutive k of one row, one per thread group of four; 16-byte loads when every row
//    starts on a 16-byte boundary (kVec: K % 4 == 0 and A 16-byte aligned).
//  * B (K x N, row-major) -> big, small (N x Kp): 32 x 32 tiles transposed through shared
//    memory, so that both the reads (along n) and the writes (along k) are coalesced.
template <bool kVec>
__global__ void __launch_bounds__(256) split_kernel(const float* __restrict__ A,
                                                    float* __restrict__ a_big,
                                                    float* __restrict__ a_small,
                                                    const float* __restrict__ B,
                                                    float* __restrict__ b_big,
                                                    float* __restrict__ b_small, int64_t M,
                                                    int64_t N, int64_t K, int64_t Kp) {
  __shared__ float tile[32][33];
  const int64_t part_blocks = gridDim.x / 2;
  const int64_t id = blockIdx.x / 2;
  if ((blockIdx.x & 1) == 0) {
    const int64_t q = Kp / 4;                 // float4 groups per row
    const int64_t per_row = (q + 255) / 256;  // work items per row
    for (int64_t it = id; it < M * per_row; it += part_blocks) {
      const int64_t row = it / per_row;
      const int64_t c = (it - row * per_row) * 256 + threadIdx.x;
      if (c >= q) continue;
      const float* arow = A + row * K;
      const int64_t k = 4 * c;
      float x[4];
      if (kVec && k + 3 < K) {
        const float4 v = *reinterpret_cast<const float4*>(arow + k);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = (k + e < K) ? arow[k + e] : 0.0f;
      }
      float b[4], s[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split(x[e], b[e], s[e]);
      *reinterpret_cast<float4*>(a_big + row * Kp + k) = make_float4(b[0], b[1], b[2], b[3]);
      *reinterpret_cast<float4*>(a_small + row * Kp + k) = make_float4(s[0], s[1], s[2], s[3]);
    }
    return;
  }
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const int64_t tiles_n = (N + 31) / 32;
  for (int64_t t = id; t < tiles_n * (Kp / 32); t += part_blocks) {
    const int64_t n0 = (t % tiles_n) * 32, k0 = (t / tiles_n) * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t k = k0 + ty + 8 * i, n = n0 + tx;
      tile[ty + 8 * i][tx] = (k < K && n < N) ? B[k * N + n] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = n0 + ty + 8 * i, k = k0 + tx;
      if (n < N) {
        float b, s;
        split(tile[tx][ty + 8 * i], b, s);
        b_big[n * Kp + k] = b;
        b_small[n * Kp + k] = s;
      }
    }
    __syncthreads();
  }
}

// Tile widths BN (M is 128): wider tiles read A less often per FLOP; the dispatcher picks
// the width whose tile count spreads evenly over the SMs.
using Tf32N128 = tc::TcConfig<tc::kTf32x3, 128, 32, 3, 256>;  // 3 stages of 64 KB, 4 epilogue warps
using Tf32N192 = tc::TcConfig<tc::kTf32x3, 192, 16, 4, 256>;  // 4 stages of 40 KB, 8 epilogue warps
using Tf32N224 = tc::TcConfig<tc::kTf32x3, 224, 16, 4, 256>;  // 4 stages of 44 KB, 8 epilogue warps
using Tf32N256 = tc::TcConfig<tc::kTf32x3, 256, 16, 4, 256>;  // 4 stages of 48 KB, 8 epilogue warps
// 256-row tiles on CTA pairs (tcgen05 cta_group::2, M 256): each CTA stages its 128 rows of the
// A planes and half of the tile's rows of the B planes, so an SM's shared memory receives and
// feeds a quarter fewer operand bytes per MMA; 6 stages (30 KB at 224 columns, 32 KB at 256).
using Tf32P224 = tc::TcConfig<tc::kTf32x3, 224, 16, 6, 256, false, true>;
using Tf32P256 = tc::TcConfig<tc::kTf32x3, 256, 16, 6, 256, false, true>;

}  // namespace

// Split planes: A_big, A_small (M x Kp) and B_big, B_small (N x Kp), 4 bytes each, each
// plane starting on a 256-byte boundary.
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int64_t Kp = padded_k(K);
  return 2 * up256(static_cast<size_t>(M) * Kp * 4) + 2 * up256(static_cast<size_t>(N) * Kp * 4);
}

cudaError_t launch_tf32x3(const Problem& p, void* workspace) {
  const int64_t Kp = padded_k(p.K);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t a_plane = up256(static_cast<size_t>(p.M) * Kp * 4);
  const size_t b_plane = up256(static_cast<size_t>(p.N) * Kp * 4);
  float* a_big = reinterpret_cast<float*>(w);
  float* a_small = reinterpret_cast<float*>(w + a_plane);
  float* b_big = reinterpret_cast<float*>(w + 2 * a_plane);
  float* b_small = reinterpret_cast<float*>(w + 2 * a_plane + b_plane);

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  {
    const int64_t a_items = p.M * ((Kp / 4 + 255) / 256);
    const int64_t b_items = ((p.N + 31) / 32) * (Kp / 32);
    const int64_t part = std::min<int64_t>(std::max(a_items, b_items), 1 << 20);
    const unsigned blocks = static_cast<unsigned>(2 * part);
    const bool vec = p.K % 4 == 0 && (reinterpret_cast<uintptr_t>(p.A) & 15u) == 0;
    if (vec)
      split_kernel<true><<<blocks, 256, 0, p.stream>>>(p.A, a_big, a_small, p.B, b_big, b_small,
                                                       p.M, p.N, p.K, Kp);
    else
      split_kernel<false><<<blocks, 256, 0, p.stream>>>(p.A, a_big, a_small, p.B, b_big,
                                                        b_small, p.M, p.N, p.K, Kp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Persistent CTAs take tiles in rounds of `sms` (CTA pairs: 256-row tiles in rounds of
  // sms / 2); the cost of a configuration is its number of rounds times its width, weighted by
  // the per-tile efficiency measured on GB300 (narrow tiles re-read A more often: 128-wide tiles
  // run about 15 % slower per FLOP than 256; pairs, fed half of B per SM, about 6-7 % faster
  // than single CTAs of the same width: 4096^3 0.510 against 0.541 ms per call, 8192^3 3.46
  // against 3.75, 2048^3 0.089 against 0.091; with few tiles they leave SMs idle, 1024^3 0.045
  // against 0.038).
  const int widths[6] = {128, 192, 224, 256, 224, 256};
  const bool pair[6] = {false, false, false, false, true, true};
  const double weight[6] = {1.15, 1.03, 1.01, 1.0, 0.94, 0.93};
  const int64_t tm = (p.M + 127) / 128;
  int best = 0;
  double best_cost = 0.0;
  for (int i = 0; i < 6; ++i) {
    if (pair[i] && (p.M <= 128 || p.K < 256)) continue;  // pairs need two tile rows
    const int64_t rows = pair[i] ? (tm + 1) / 2 : tm;
    const int64_t units = rows * ((p.N + widths[i] - 1) / widths[i]);
    const int64_t slots = pair[i] ? sms / 2 : sms;
    const int64_t rounds = (units + slots - 1) / slots;
    const double cost = static_cast<double>(rounds) * widths[i] * weight[i];
    if (i == 0 || cost < best_cost) {
      best = i;
      best_cost = cost;
    }
  }
  if (p.K < 256) best = 0;  // one short chunk: the wide epilogue does not pay
  switch (best) {
    case 1: return tc::run_tc<Tf32N192>(p, a_big, a_small, b_big, b_small, Kp, Kp, Kp);
    case 2: return tc::run_tc<Tf32N224>(p, a_big, a_small, b_big, b_small, Kp, Kp, Kp);
    case 3: return tc::run_tc<Tf32N256>(p, a_big, a_small, b_big, b_small, Kp, Kp, Kp);
    case 4: return tc::run_tc<Tf32P224>(p, a_big, a_small, b_big, b_small, Kp, Kp, Kp);
    case 5: return tc::run_tc<Tf32P256>(p, a_big, a_small, b_big, b_small, Kp, Kp, Kp);
    default: return tc::run_tc<Tf32N128>(p, a_big, a_small, b_big, b_small, Kp, Kp, Kp);
  }
}

}  // namespace t2s
