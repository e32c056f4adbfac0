// probes.cu -- throughput probes that give the roofline its measured ceilings.
//
// Page "4주차: Roofline과 Tiling", section "2. Roofline", places a kernel under
// min(peak FLOP/s, bandwidth x AI); the pages give no GB300 figures, so the peaks are measured
// here with the same instructions the products use, and nothing else:
//  * the FP32 CUDA-core pipe: packed two-wide fused multiply-adds (fma.rn.f32x2) in long
//    independent chains, with no memory traffic, at the product kernels' occupancy of 8 warps
//    per SM (two CTAs of 4 warps);
//  * the TF32 tensor pipe: back-to-back tcgen05.mma kind::tf32 (M = 128, N = 256, K = 8) on
//    operands resident in shared memory, accumulating in TMEM, one CTA per SM, the instruction
//    and shared-memory layout of the 3xTF32 product (K-major, 128-byte swizzle).
//  * the store path out of the SMs: a matrix written with no arithmetic in the short-K product's
//    store pattern (256 x 128 tiles of 8 warps, one CTA per SM, the product's grouped tile
//    order), either through 64 x 32 TMA boxes staged in shared memory (that kernel's epilogue)
//    or with 16-byte stores from registers in the register-tile layout (the other kernels').
// The FMA and MMA probes write one value per thread to `out` so that their work is observable;
// the store probe's work is the matrix it writes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "t2s_device.cuh"
#include "t2s_internal.h"
#include "t2s_tmap.h"
#include "tc_gemm.cuh"

namespace t2s {
namespace {

constexpr int kFmaChains = 16;  // packed accumulators (32 FP32 values) per thread
constexpr int kFmaThreads = 128;
constexpr int kFmaCtasPerSm = 2;

__global__ void __launch_bounds__(kFmaThreads, kFmaCtasPerSm)
    ffma_probe_kernel(int64_t iters, float* __restrict__ out) {
  uint64_t acc[kFmaChains];
#pragma unroll
  for (int j = 0; j < kFmaChains; ++j) {
    const float v = static_cast<float>(threadIdx.x + j);
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc[j]) : "f"(v), "f"(-v));
  }
  // acc = 0.5 acc + 1 converges to 2: no overflow, no subnormals.
  const uint64_t half = pack_dup(0.5f), one = pack_dup(1.0f);
  for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < kFmaChains; ++j)
      asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[j]) : "l"(half), "l"(one));
  }
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < kFmaChains; ++j) {
    const float2 v = unpack2(acc[j]);
    sum += v.x + v.y;
  }
  out[static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x] = sum;
}

// The tcgen05 layout constants of the probe: TF32 operands, N = 256, 32-deep K blocks in
// 128-byte swizzled rows.
using ProbeCfg = tc::TcConfig<tc::kTf32x3, 256, 32, 1, 256>;
constexpr int kMmaThreads = 128;
constexpr uint32_t kProbeA = 128 * 128;   // A: 128 rows x 128 bytes
constexpr uint32_t kProbeB = 256 * 128;   // B: 256 rows x 128 bytes
constexpr int kProbeSmem = kProbeA + kProbeB + 64 + 1024;
constexpr int kMmaPerBlock = ProbeCfg::BK / ProbeCfg::MMA_K;  // 4 MMAs per 32-deep K block
constexpr int64_t kMmaFlops = 2LL * 128 * 256 * 8;

__global__ void __launch_bounds__(kMmaThreads, 1)
    tf32_mma_probe_kernel(int64_t iters, float* __restrict__ out, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base, sB = base + kProbeA;
  const uint32_t bar = sB + kProbeB, slot = bar + 8u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Zero operands, made visible to the tensor core (async proxy).
  for (uint32_t off = threadIdx.x * 16u; off < kProbeA + kProbeB; off += kMmaThreads * 16u)
    st_shared_v4(sA + off, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc<1>(slot, 256);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(slot) : "memory");
  if (threadIdx.x == 0) {
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < kMmaPerBlock; ++k) {
        const uint32_t off = k * ProbeCfg::MMA_K * ProbeCfg::ELEM;  // 32 bytes per K step
        tc::mma_issue<tc::kTf32x3, 1>(tmem, tc::smem_desc<ProbeCfg>(sA + off),
                                      tc::smem_desc<ProbeCfg>(sB + off), ProbeCfg::IDESC,
                                      (it != 0 || k != 0) ? 1u : 0u);
      }
    }
    tc::mma_commit<1>(bar);
  }
  __syncwarp();
  // Every thread waits for the MMAs (bounded); on expiry the status word records it.
  const bool done = mbar_wait_bounded(bar, 0u, status);
  tc::tc_fence_after();
  uint32_t r[16];
  tc::tmem_ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16), r);
  out[static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x] =
      done ? __uint_as_float(r[lane & 15]) : -1.0f;
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<1>(tmem, 256);
}

// Store probe: 256 x 128 tiles, 8 warps of 64 x 64 (4 along M, 2 along N), in the grouped
// order of the short-K product (groups of 8 tile rows, column-major inside a group).
constexpr int kStoreThreads = 256;
constexpr int kStoreBoxBytes = 64 * 128;                     // 64 rows x 32 floats
constexpr int kStoreSmem = 8 * 2 * kStoreBoxBytes + 1024;    // two boxes per warp

__device__ __forceinline__ void store_tile_origin(int tile, int tiles_m, int tiles_n, int& m0,
                                                  int& n0) {
  constexpr int kGroup = 8;
  const int per_group = kGroup * tiles_n;
  const int first_m = (tile / per_group) * kGroup;
  const int gsz = min(tiles_m - first_m, kGroup);
  m0 = (first_m + (tile % per_group) % gsz) * 256;
  n0 = ((tile % per_group) / gsz) * 128;
}

// Each warp stages its 64 x 64 part in its own 16 KB of shared memory (the value is the same
// everywhere, so the swizzle of the boxes does not change what lands in C) and stores it as two
// 64 x 32 boxes; before restaging it waits until its previous stores have read the boxes.
__global__ void __launch_bounds__(kStoreThreads, 1)
    store_probe_tma_kernel(const __grid_constant__ CUtensorMap tmC, int tiles_m, int tiles_n,
                           float value) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm0 = (warp % 4) * 64, wn0 = (warp / 4) * 64;
  const uint32_t stg = base + static_cast<uint32_t>(warp) * 2u * kStoreBoxBytes;
  const uint32_t v = __float_as_uint(value);
  const int tiles = tiles_m * tiles_n;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    int m0, n0;
    store_tile_origin(t, tiles_m, tiles_n, m0, n0);
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 2 * kStoreBoxBytes / (32 * 16); ++i)
      st_shared_v4(stg + static_cast<uint32_t>(i * 32 + lane) * 16u, v, v, v, v);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&tmC, stg, n0 + wn0, m0 + wm0);
      tma_store_2d(&tmC, stg + kStoreBoxBytes, n0 + wn0 + 32, m0 + wm0);
    }
  }
  if (lane == 0) bulk_wait_all();
}

// Lane (g, h) of a warp writes rows g + 8i (i < 8) and the 16-byte chunks at columns
// 4h + 16j (j < 4) of its 64 x 64 part, as the product kernels' epilogue does.
__global__ void __launch_bounds__(kStoreThreads, 1)
    store_probe_plain_kernel(float* __restrict__ C, int64_t N, int tiles_m, int tiles_n,
                             float value) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, h = lane & 3;
  const int wm0 = (warp % 4) * 64, wn0 = (warp / 4) * 64;
  const float4 v = make_float4(value, value, value, value);
  const int tiles = tiles_m * tiles_n;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    int m0, n0;
    store_tile_origin(t, tiles_m, tiles_n, m0, n0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float* row = C + static_cast<int64_t>(m0 + wm0 + g + 8 * i) * N + (n0 + wn0 + 4 * h);
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<float4*>(row + 16 * j) = v;
    }
  }
}

int sm_count_current() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace

cudaError_t launch_ffma_probe(int64_t iters, float* out, cudaStream_t stream, int64_t* flops) {
  const int sms = sm_count_current();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int ctas = kFmaCtasPerSm * sms;
  ffma_probe_kernel<<<ctas, kFmaThreads, 0, stream>>>(iters, out);
  *flops = static_cast<int64_t>(ctas) * kFmaThreads * iters * kFmaChains * 2 * 2;
  return cudaGetLastError();
}

cudaError_t launch_tf32_mma_probe(int64_t iters, float* out, unsigned* status, cudaStream_t stream,
                                  int64_t* flops) {
  const int sms = sm_count_current();
  if (sms <= 0) return cudaErrorInvalidDevice;
  cudaError_t e = cudaFuncSetAttribute(tf32_mma_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return e;
  tf32_mma_probe_kernel<<<sms, kMmaThreads, kProbeSmem, stream>>>(iters, out, status);
  *flops = static_cast<int64_t>(sms) * iters * kMmaPerBlock * kMmaFlops;
  return cudaGetLastError();
}

cudaError_t launch_store_probe(int64_t M, int64_t N, float* C, int mode, float value,
                               cudaStream_t stream, int64_t* bytes) {
  const int sms = sm_count_current();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int tiles_m = static_cast<int>(M / 256), tiles_n = static_cast<int>(N / 128);
  const int tiles = tiles_m * tiles_n;
  const int ctas = tiles < sms ? tiles : sms;
  if (mode == 0) {
    CUtensorMap tm;
    cudaError_t e = encode_tmap_f32_2d(&tm, C, N, M, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(store_probe_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kStoreSmem);
    if (e != cudaSuccess) return e;
    store_probe_tma_kernel<<<ctas, kStoreThreads, kStoreSmem, stream>>>(tm, tiles_m, tiles_n,
                                                                        value);
  } else {
    store_probe_plain_kernel<<<ctas, kStoreThreads, 0, stream>>>(C, N, tiles_m, tiles_n, value);
  }
  *bytes = M * N * 4;
  return cudaGetLastError();
}

}  // namespace t2s
