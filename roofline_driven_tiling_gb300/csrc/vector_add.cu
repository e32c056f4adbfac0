// vector_add.cu -- z = x + y in FP32: the memory-bound example of page "4주차: Roofline과
// Tiling" (section "1. Arithmetic Intensity", example "Vector Add": N FLOPs for 12N bytes,
// AI = 1/12 FLOP/B). It measures the bandwidth slope of the roofline on which the GEMM kernels
// are placed: the kernel does nothing but stream two vectors in and one out.
//
// GB300 design: 32-byte (256-bit) global loads and stores when all three pointers are 32-byte
// aligned (16-byte, then 4-byte accesses otherwise), loads marked non-coherent and not
// allocated in L1, stores marked evict-first; a grid-stride loop over a grid of 8 CTAs of 256
// threads per SM, each thread keeping two 32-byte loads of each input in flight.
#include <cuda_runtime.h>

#include <cstdint>

#include "t2s_internal.h"

namespace t2s {
namespace {

struct alignas(32) f8 {
  float v[8];
};

__device__ __forceinline__ f8 ld8(const float* p) {
  f8 r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]),
                 "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st8(float* p, const f8& r) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(r.v[0]),
               "f"(r.v[1]), "f"(r.v[2]), "f"(r.v[3]), "f"(r.v[4]), "f"(r.v[5]), "f"(r.v[6]),
               "f"(r.v[7])
               : "memory");
}

// Width 8: 32-byte vectors; 4: float4; 1: scalars. Elements [0, n8 * W) go through the
// vector path; the tail (< W elements) through the scalar loop of thread 0's block.
template <int W>
__global__ void __launch_bounds__(256) vector_add_kernel(int64_t n, const float* __restrict__ x,
                                                         const float* __restrict__ y,
                                                         float* __restrict__ z) {
  const int64_t nv = n / W;  // whole vectors
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if constexpr (W == 8) {
    for (; i + stride < nv; i += 2 * stride) {
      const f8 a0 = ld8(x + 8 * i), b0 = ld8(y + 8 * i);
      const f8 a1 = ld8(x + 8 * (i + stride)), b1 = ld8(y + 8 * (i + stride));
      f8 c0, c1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c0.v[e] = __fadd_rn(a0.v[e], b0.v[e]);
        c1.v[e] = __fadd_rn(a1.v[e], b1.v[e]);
      }
      st8(z + 8 * i, c0);
      st8(z + 8 * (i + stride), c1);
    }
    for (; i < nv; i += stride) {
      const f8 a = ld8(x + 8 * i), b = ld8(y + 8 * i);
      f8 c;
#pragma unroll
      for (int e = 0; e < 8; ++e) c.v[e] = __fadd_rn(a.v[e], b.v[e]);
      st8(z + 8 * i, c);
    }
  } else if constexpr (W == 4) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* y4 = reinterpret_cast<const float4*>(y);
    float4* z4 = reinterpret_cast<float4*>(z);
    for (; i < nv; i += stride) {
      const float4 a = __ldg(x4 + i), b = __ldg(y4 + i);
      z4[i] = make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z),
                          __fadd_rn(a.w, b.w));
    }
  } else {
    for (; i < nv; i += stride) z[i] = __fadd_rn(x[i], y[i]);
  }
  if (W > 1 && blockIdx.x == 0) {
    for (int64_t t = nv * W + threadIdx.x; t < n; t += blockDim.x) z[t] = __fadd_rn(x[t], y[t]);
  }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace t2s

extern "C" int t2s_vector_add_f32(int64_t n, const float* x, const float* y, float* z,
                                  t2s_stream_t stream) {
  using namespace t2s;
  if (n < 0) return T2S_ERR_INVALID;
  if (n == 0) return T2S_OK;
  if (x == nullptr || y == nullptr || z == nullptr) return T2S_ERR_INVALID;
  if (!aligned(x, 4) || !aligned(y, 4) || !aligned(z, 4)) return T2S_ERR_INVALID;
  if (z == x || z == y) return T2S_ERR_INVALID;  // inputs are read through the read-only path
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return T2S_ERR_CUDA;
  }
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int width = (aligned(x, 32) && aligned(y, 32) && aligned(z, 32)) ? 8
                    : (aligned(x, 16) && aligned(y, 16) && aligned(z, 16)) ? 4
                                                                          : 1;
  const int64_t vectors = n / width;
  const int64_t want = (vectors + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : want < cap ? want : cap);
  if (width == 8) vector_add_kernel<8><<<grid, 256, 0, s>>>(n, x, y, z);
  else if (width == 4) vector_add_kernel<4><<<grid, 256, 0, s>>>(n, x, y, z);
  else vector_add_kernel<1><<<grid, 256, 0, s>>>(n, x, y, z);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return T2S_ERR_CUDA;
  }
  return T2S_OK;
}
