// api.cu -- the C ABI of include/t2s_gemm.h: argument checks, dispatch to the
// kernels, the device status word, and the bounded-wait self-test.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "t2s_device.cuh"
#include "t2s_internal.h"

namespace t2s {
namespace {

// Bounded waits that give up record T2S_ERR_TIMEOUT here (one word per device;
// a static device variable, so nothing is allocated). Host code must not pass
// the symbol itself to a kernel: its device address is looked up per device.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status_ptr[kMaxDevices] = {};
thread_local int g_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return T2S_ERR_CUDA;
}

// Device address of the status word on the current device, looked up once per device.
cudaError_t status_word(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

bool misaligned(const void* p, uintptr_t bytes) {
  return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) != 0;
}

// The checks every GEMM entry point shares, for operands of `ab_bytes`-byte elements (A, B)
// and a C of `c_bytes`-byte elements. Sets `*noop` when there is nothing to compute (M == 0
// or N == 0).
int validate(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
             uintptr_t ab_bytes, bool* noop, uintptr_t c_bytes = 4) {
  if (M < 0 || N < 0 || K < 0) return T2S_ERR_INVALID;
  if (M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return T2S_ERR_INVALID;
  const bool has_a = M > 0 && K > 0, has_b = K > 0 && N > 0, has_c = M > 0 && N > 0;
  if ((has_a && A == nullptr) || (has_b && B == nullptr) || (has_c && C == nullptr))
    return T2S_ERR_INVALID;
  if ((has_a && misaligned(A, ab_bytes)) || (has_b && misaligned(B, ab_bytes)) ||
      (has_c && misaligned(C, c_bytes)))
    return T2S_ERR_INVALID;
  if (has_c && ((has_a && C == A) || (has_b && C == B))) return T2S_ERR_INVALID;
  *noop = !has_c;
  return T2S_OK;
}

// Checks the common contract; on success fills `p` and returns T2S_OK. `*noop` is set
// when there is nothing to compute (M == 0 or N == 0).
int prepare(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
            t2s_stream_t stream, Problem* p, bool* noop) {
  const int rc = validate(M, N, K, A, B, C, 4, noop);
  if (rc != T2S_OK || *noop) return rc;
  p->M = M;
  p->N = N;
  p->K = K;
  p->A = A;
  p->B = B;
  p->C = C;
  p->stream = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = status_word(&p->status);
  if (e != cudaSuccess) return fail_cuda(e);
  return T2S_OK;
}

// K == 0: the empty sum, +0.0f everywhere.
int zero_fill(const Problem& p) {
  const cudaError_t e = cudaMemsetAsync(p.C, 0, static_cast<size_t>(p.M) * p.N * sizeof(float),
                                        p.stream);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

using Launcher = cudaError_t (*)(const Problem&);

int gemm_common(Launcher launch, int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                float* C, t2s_stream_t stream) {
  Problem p{};
  bool noop = false;
  const int rc = prepare(M, N, K, A, B, C, stream, &p, &noop);
  if (rc != T2S_OK || noop) return rc;
  if (K == 0) return zero_fill(p);
  const cudaError_t e = launch(p);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

__global__ void wait_selftest_kernel(unsigned* status, uint64_t limit_ns) {
  __shared__ alignas(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // Nothing ever arrives on this barrier: the wait must give up and record it.
  if (threadIdx.x == 0) mbar_wait_bounded(b, 0, status, limit_ns);
}

}  // namespace

void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

int gemm_f32_block(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                   t2s_stream_t stream, int concurrent) {
  Problem p{};
  bool noop = false;
  const int rc = prepare(M, N, K, A, B, C, stream, &p, &noop);
  if (rc != T2S_OK || noop) return rc;
  if (K == 0) return zero_fill(p);
  const cudaError_t e = launch_ffma_concurrent(p, concurrent);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

int gemm_f32_kchunk(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                    t2s_stream_t stream, int concurrent, int64_t k0, int64_t kc, bool accumulate) {
  Problem p{};
  bool noop = false;
  const int rc = prepare(M, N, K, A, B, C, stream, &p, &noop);
  if (rc != T2S_OK || noop) return rc;
  if (K == 0) return zero_fill(p);
  if (kc <= 0 || k0 < 0 || k0 >= K || k0 % 32 != 0 || kc % 32 != 0) return T2S_ERR_INVALID;
  const cudaError_t e = launch_ffma_range(p, concurrent, k0, kc, accumulate);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace t2s

using namespace t2s;

extern "C" {

int t2s_gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                 t2s_stream_t stream) {
  return gemm_common(launch_ffma, M, N, K, A, B, C, stream);
}

int t2s_gemm_f32_naive(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                       float* C, t2s_stream_t stream) {
  return gemm_common(launch_naive, M, N, K, A, B, C, stream);
}

int t2s_gemm_f32_smem32(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                        float* C, t2s_stream_t stream) {
  return gemm_common(launch_smem32, M, N, K, A, B, C, stream);
}

size_t t2s_gemm_f32_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int splits) {
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return 0;
  if (splits > 64) return 0;
  if (splits <= 0) splits = splitk_auto(M, N, K);
  const int planes = K > 0 ? splitk_planes(K, splits) : 1;
  return planes <= 1 ? 0 : static_cast<size_t>(planes) * M * N * sizeof(float);
}

int t2s_gemm_f32_splitk(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                        int splits, void* workspace, size_t workspace_bytes, t2s_stream_t stream) {
  if (splits > 64) return T2S_ERR_INVALID;
  Problem p{};
  bool noop = false;
  const int rc = prepare(M, N, K, A, B, C, stream, &p, &noop);
  if (rc != T2S_OK || noop) return rc;
  if (K == 0) return zero_fill(p);
  if (splits <= 0) splits = splitk_auto(M, N, K);
  const int planes = splitk_planes(K, splits);
  if (planes > 1) {
    const size_t need = static_cast<size_t>(planes) * M * N * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need) return T2S_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return T2S_ERR_WORKSPACE;
  }
  const cudaError_t e = planes > 1 ? launch_ffma_splitk(p, splits, static_cast<float*>(workspace))
                                   : launch_ffma(p);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

size_t t2s_gemm_f32_streamk_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return 0;
  return streamk_workspace_bytes(M, N, K);
}

int t2s_gemm_f32_streamk(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                         float* C, void* workspace, size_t workspace_bytes, t2s_stream_t stream) {
  Problem p{};
  bool noop = false;
  const int rc = prepare(M, N, K, A, B, C, stream, &p, &noop);
  if (rc != T2S_OK || noop) return rc;
  if (K == 0) return zero_fill(p);
  if (!streamk_supported(p)) {
    const cudaError_t e = launch_ffma(p);
    return e == cudaSuccess ? T2S_OK : fail_cuda(e);
  }
  const size_t need = streamk_workspace_bytes(M, N, K);
  if (workspace == nullptr || workspace_bytes < need) return T2S_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return T2S_ERR_WORKSPACE;
  const cudaError_t e = launch_ffma_streamk(p, static_cast<float*>(workspace));
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

size_t t2s_gemm_f32_tf32x3_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return 0;
  return tf32x3_workspace_bytes(M, N, K);
}

int t2s_gemm_f32_tf32x3(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                        void* workspace, size_t workspace_bytes, t2s_stream_t stream) {
  Problem p{};
  bool noop = false;
  const int rc = prepare(M, N, K, A, B, C, stream, &p, &noop);
  if (rc != T2S_OK || noop) return rc;
  if (K == 0) return zero_fill(p);
  const size_t need = tf32x3_workspace_bytes(M, N, K);
  if (workspace == nullptr || workspace_bytes < need) return T2S_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return T2S_ERR_WORKSPACE;
  const cudaError_t e = launch_tf32x3(p, workspace);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

size_t t2s_gemm_bf16_f32_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return 0;
  return half_workspace_bytes(M, N, K);
}

size_t t2s_gemm_f16_f32_workspace_size(int64_t M, int64_t N, int64_t K) {
  return t2s_gemm_bf16_f32_workspace_size(M, N, K);
}

}  // extern "C"

namespace t2s {
namespace {

using LauncherF64 = cudaError_t (*)(int64_t, int64_t, int64_t, const double*, const double*,
                                    double*, cudaStream_t);
using LauncherHalf = cudaError_t (*)(int64_t, int64_t, int64_t, const uint16_t*, const uint16_t*,
                                     float*, void*, cudaStream_t, unsigned*);

int gemm_half_common(LauncherHalf launch, int64_t M, int64_t N, int64_t K, const uint16_t* A,
                     const uint16_t* B, float* C, void* workspace, size_t workspace_bytes,
                     t2s_stream_t stream) {
  bool noop = false;
  const int rc = validate(M, N, K, A, B, C, 2, &noop);
  if (rc != T2S_OK || noop) return rc;
  Problem p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = C;
  p.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = status_word(&p.status);
  if (e != cudaSuccess) return fail_cuda(e);
  if (K == 0) return zero_fill(p);
  const size_t need = half_workspace_bytes(M, N, K);
  if (workspace == nullptr || workspace_bytes < need) return T2S_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return T2S_ERR_WORKSPACE;
  e = launch(M, N, K, A, B, C, workspace, p.stream, p.status);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

int gemm_f64_common(LauncherF64 launch, int64_t M, int64_t N, int64_t K, const double* A,
                    const double* B, double* C, t2s_stream_t stream) {
  bool noop = false;
  const int rc = validate(M, N, K, A, B, C, 8, &noop, 8);
  if (rc != T2S_OK || noop) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (K == 0) {
    e = cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * sizeof(double), s);
  } else {
    e = launch(M, N, K, A, B, C, s);
  }
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

}  // namespace
}  // namespace t2s

extern "C" {

int t2s_gemm_bf16_f32(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                      float* C, void* workspace, size_t workspace_bytes, t2s_stream_t stream) {
  return t2s::gemm_half_common(t2s::launch_bf16, M, N, K, A, B, C, workspace, workspace_bytes,
                               stream);
}

int t2s_gemm_f16_f32(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                     float* C, void* workspace, size_t workspace_bytes, t2s_stream_t stream) {
  return t2s::gemm_half_common(t2s::launch_f16, M, N, K, A, B, C, workspace, workspace_bytes,
                               stream);
}

int t2s_gemm_f64(int64_t M, int64_t N, int64_t K, const double* A, const double* B, double* C,
                 t2s_stream_t stream) {
  return t2s::gemm_f64_common(t2s::launch_dgemm, M, N, K, A, B, C, stream);
}

int t2s_gemm_f64_naive(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                       double* C, t2s_stream_t stream) {
  return t2s::gemm_f64_common(t2s::launch_naive_f64, M, N, K, A, B, C, stream);
}

int t2s_gemm_f64_smem32(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                        double* C, t2s_stream_t stream) {
  return t2s::gemm_f64_common(t2s::launch_smem32_f64, M, N, K, A, B, C, stream);
}

const char* t2s_status_string(int status) {
  switch (status) {
    case T2S_OK: return "ok";
    case T2S_ERR_INVALID: return "invalid argument";
    case T2S_ERR_CUDA: return "CUDA error (see t2s_last_cuda_error)";
    case T2S_ERR_TIMEOUT: return "a kernel gave up a bounded barrier wait";
    case T2S_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case T2S_ERR_TOO_LARGE: return "problem needs more scratch than the built-in 32 MiB array";
    default: return "unknown status";
  }
}

int t2s_device_status(t2s_stream_t stream) {
  unsigned* word = nullptr;
  cudaError_t e = status_word(&word);
  if (e != cudaSuccess) return fail_cuda(e);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  unsigned value = 0;
  e = cudaMemcpyAsync(&value, word, sizeof(value), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  return value == 0 ? T2S_OK : static_cast<int>(value);
}

int t2s_last_cuda_error(void) { return g_last_cuda_error; }

int t2s_selftest_wait_timeout(int64_t limit_ns, t2s_stream_t stream) {
  unsigned* word = nullptr;
  cudaError_t e = status_word(&word);
  if (e != cudaSuccess) return fail_cuda(e);
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000) limit_ns = 1000000000;
  e = launch_wait_selftest(word, static_cast<uint64_t>(limit_ns),
                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

int t2s_probe_outputs(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return 256 * sms;
}

int t2s_probe_fp32_fma(int64_t iters, float* out, int64_t* flops, t2s_stream_t stream) {
  if (iters < 1 || iters > (1LL << 24) || out == nullptr || flops == nullptr) return T2S_ERR_INVALID;
  const cudaError_t e = launch_ffma_probe(iters, out, reinterpret_cast<cudaStream_t>(stream), flops);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

int t2s_probe_tf32_mma(int64_t iters, float* out, int64_t* flops, t2s_stream_t stream) {
  if (iters < 1 || iters > (1LL << 16) || out == nullptr || flops == nullptr) return T2S_ERR_INVALID;
  unsigned* word = nullptr;
  cudaError_t e = status_word(&word);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_tf32_mma_probe(iters, out, word, reinterpret_cast<cudaStream_t>(stream), flops);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

int t2s_probe_store_f32(int64_t M, int64_t N, float* C, int mode, float value, int64_t* bytes,
                        t2s_stream_t stream) {
  if (M < 256 || N < 128 || M % 256 != 0 || N % 128 != 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM)
    return T2S_ERR_INVALID;
  if ((M / 256) * (N / 128) > 0x7fffffffLL) return T2S_ERR_INVALID;
  if (C == nullptr || (reinterpret_cast<uintptr_t>(C) & 15u) != 0 || bytes == nullptr)
    return T2S_ERR_INVALID;
  if (mode != 0 && mode != 1) return T2S_ERR_INVALID;
  const cudaError_t e =
      launch_store_probe(M, N, C, mode, value, reinterpret_cast<cudaStream_t>(stream), bytes);
  return e == cudaSuccess ? T2S_OK : fail_cuda(e);
}

int t2s_gemm_f32_plan(int64_t M, int64_t N, int64_t K, int sms) {
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return -1;
  if (sms < 1) return -1;
  return ffma_plan(M, N, K, sms);
}

int t2s_gemm_f32_splitk_plan(int64_t M, int64_t N, int64_t K, int sms) {
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM) return -1;
  if (sms < 1) return -1;
  return splitk_choice(M, N, K, sms);
}

int t2s_version(void) { return 100; }

}  // extern "C"
