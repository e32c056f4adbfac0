// gemm_tf32x3_noalloc.cu -- the 3xTF32 product for callers that cannot allocate memory.
//
// t2s_gemm_f32_tf32x3 needs a scratch buffer for the split operands, which its caller
// allocates. Some callers cannot: a plugin inside a framework that owns all device memory
// through its own pool and a fixed budget, a latency-critical loop where the implicit
// device synchronisation and unbounded time of cudaMalloc / cudaFree are not acceptable,
// or plain C code that has no device allocator of its own. This entry point serves them:
// its scratch is a file-scope device array that exists, on every GPU that loads this
// library, from the load until the process exits.
//
// In host code the array's name denotes a host-side stand-in, not a device address, so it
// must never be passed to a kernel. Its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) on the first call made on the device,
// and then passed down like a caller-owned workspace.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "t2s_internal.h"

namespace t2s {
namespace {

constexpr size_t kStaticScratchBytes = T2S_TF32X3_NOALLOC_MAX_SCRATCH;
constexpr int kMaxDevices = 64;

// Split planes of the last call made on this device (shared by every call).
static __device__ __align__(256) unsigned char g_tf32x3_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_tf32x3_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace t2s

extern "C" int t2s_gemm_f32_tf32x3_noalloc(int64_t M, int64_t N, int64_t K, const float* A,
                                           const float* B, float* C, t2s_stream_t stream) {
  // Shapes are checked first, so an oversized problem is reported as such even before
  // the device is touched.
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM)
    return T2S_ERR_INVALID;
  if (t2s_gemm_f32_tf32x3_workspace_size(M, N, K) > t2s::kStaticScratchBytes)
    return T2S_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const cudaError_t e = t2s::scratch_address(&scratch);
  if (e != cudaSuccess) {
    t2s::set_last_cuda_error(e);
    return T2S_ERR_CUDA;
  }
  // The split pre-pass writes every scratch byte the product kernel reads (the zero
  // padding beyond K included), so what the previous call left there is never used.
  return t2s_gemm_f32_tf32x3(M, N, K, A, B, C, scratch, t2s::kStaticScratchBytes, stream);
}
