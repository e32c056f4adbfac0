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
// Each probe writes one value per thread to `out` so that its work is observable.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "t2s_device.cuh"
#include "t2s_internal.h"
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

}  // namespace t2s
