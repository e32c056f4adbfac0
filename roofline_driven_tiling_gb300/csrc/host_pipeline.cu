// host_pipeline.cu -- C = A x B for matrices in host memory, with the host<->device copies
// overlapped with the product.
//
// The product needs all of B but only a row block of A for a row block of C, so the
// pipeline is: copy B; then for each row block i of A, copy it, multiply it (on one of two
// compute streams, so consecutive blocks can share the GPU), and copy the block of C back
// as soon as it is done. Host->device and device->host copies use separate copy streams,
// so both directions run under the products. Only the copy of B, the first block of A and
// the last block of C remain exposed.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "t2s_internal.h"

namespace t2s {
namespace {

#ifndef T2S_PIPE_MIN_ROWS
#define T2S_PIPE_MIN_ROWS 1024
#endif
#ifndef T2S_PIPE_CONCURRENT
#define T2S_PIPE_CONCURRENT 2
#endif

constexpr int kMaxDevices = 64;
constexpr int kMaxBlocks = 8;

// Streams and events reused by every call on a device (created once, never freed: they
// are driver objects, not device memory). A mutex serialises the enqueue sequences of
// concurrent host threads; a stream wait captures an event's state when it is enqueued,
// so reusing the events in a later call cannot disturb an earlier one.
struct PipelineResources {
  bool ready = false;
  cudaStream_t copy_in = nullptr, copy_out = nullptr, compute2 = nullptr;
  cudaEvent_t start = nullptr, b_ready = nullptr, done_out = nullptr, done_compute2 = nullptr;
  cudaEvent_t a_ready[kMaxBlocks] = {}, c_ready[kMaxBlocks] = {};
};

std::mutex g_pipe_mu;
PipelineResources g_pipe[kMaxDevices];

cudaError_t make_event(cudaEvent_t* e) {
  return cudaEventCreateWithFlags(e, cudaEventDisableTiming);
}

cudaError_t resources(PipelineResources** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  PipelineResources& r = g_pipe[dev];
  if (!r.ready) {
    if ((e = cudaStreamCreateWithFlags(&r.copy_in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&r.copy_out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&r.compute2, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = make_event(&r.start)) != cudaSuccess) return e;
    if ((e = make_event(&r.b_ready)) != cudaSuccess) return e;
    if ((e = make_event(&r.done_out)) != cudaSuccess) return e;
    if ((e = make_event(&r.done_compute2)) != cudaSuccess) return e;
    for (int i = 0; i < kMaxBlocks; ++i) {
      if ((e = make_event(&r.a_ready[i])) != cudaSuccess) return e;
      if ((e = make_event(&r.c_ready[i])) != cudaSuccess) return e;
    }
    r.ready = true;
  }
  *out = &r;
  return cudaSuccess;
}

}  // namespace
}  // namespace t2s

extern "C" int t2s_gemm_f32_host(int64_t M, int64_t N, int64_t K, const float* hA,
                                 const float* hB, float* hC, float* dA, float* dB, float* dC,
                                 t2s_stream_t stream) {
  using namespace t2s;
  if (M < 0 || N < 0 || K < 0 || M > T2S_MAX_DIM || N > T2S_MAX_DIM || K > T2S_MAX_DIM)
    return T2S_ERR_INVALID;
  if (M == 0 || N == 0) return T2S_OK;
  const bool has_ab = K > 0;
  if (hC == nullptr || dC == nullptr || (has_ab && (hA == nullptr || hB == nullptr ||
                                                    dA == nullptr || dB == nullptr)))
    return T2S_ERR_INVALID;
  if (has_ab && (dC == dA || dC == dB)) return T2S_ERR_INVALID;

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  PipelineResources* r = nullptr;
  cudaError_t e = resources(&r);
  auto fail = [](cudaError_t err) {
    set_last_cuda_error(err);
    return T2S_ERR_CUDA;
  };
  if (e != cudaSuccess) return fail(e);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // Row blocks of at least T2S_PIPE_MIN_ROWS rows (1024 measured best at 3072^3 to 4096^3),
  // at most kMaxBlocks of them.
  int nb = static_cast<int>(M / T2S_PIPE_MIN_ROWS);
  nb = nb < 1 ? 1 : nb > kMaxBlocks ? kMaxBlocks : nb;
  const int64_t rows_per = (M + nb - 1) / nb;

  // Everything starts after the work already enqueued on the caller's stream.
  if ((e = cudaEventRecord(r->start, s)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(r->copy_in, r->start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(r->copy_out, r->start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(r->compute2, r->start, 0)) != cudaSuccess) return fail(e);
  if (has_ab) {
    if ((e = cudaMemcpyAsync(dB, hB, static_cast<size_t>(K) * N * sizeof(float),
                             cudaMemcpyHostToDevice, r->copy_in)) != cudaSuccess)
      return fail(e);
    if ((e = cudaEventRecord(r->b_ready, r->copy_in)) != cudaSuccess) return fail(e);
  }
  for (int i = 0; i < nb; ++i) {
    const int64_t r0 = i * rows_per;
    if (r0 >= M) break;
    const int64_t rows = (r0 + rows_per <= M) ? rows_per : M - r0;
    const cudaStream_t cs = (i & 1) ? r->compute2 : s;
    if (has_ab) {
      if ((e = cudaMemcpyAsync(dA + r0 * K, hA + r0 * K, static_cast<size_t>(rows) * K * sizeof(float),
                               cudaMemcpyHostToDevice, r->copy_in)) != cudaSuccess)
        return fail(e);
      if ((e = cudaEventRecord(r->a_ready[i], r->copy_in)) != cudaSuccess) return fail(e);
      if ((e = cudaStreamWaitEvent(cs, r->a_ready[i], 0)) != cudaSuccess) return fail(e);
    }
    // Blocks alternate between two compute streams, so two of them share the GPU.
    const int rc = gemm_f32_block(rows, N, K, has_ab ? dA + r0 * K : nullptr, has_ab ? dB : nullptr,
                                  dC + r0 * N, reinterpret_cast<t2s_stream_t>(cs), nb > 1 ? T2S_PIPE_CONCURRENT : 1);
    if (rc != T2S_OK) return rc;
    if ((e = cudaEventRecord(r->c_ready[i], cs)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(r->copy_out, r->c_ready[i], 0)) != cudaSuccess) return fail(e);
    if ((e = cudaMemcpyAsync(hC + r0 * N, dC + r0 * N, static_cast<size_t>(rows) * N * sizeof(float),
                             cudaMemcpyDeviceToHost, r->copy_out)) != cudaSuccess)
      return fail(e);
  }
  // The caller's stream completes only after every copy back and the second compute stream.
  if ((e = cudaEventRecord(r->done_out, r->copy_out)) != cudaSuccess) return fail(e);
  if ((e = cudaEventRecord(r->done_compute2, r->compute2)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(s, r->done_out, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(s, r->done_compute2, 0)) != cudaSuccess) return fail(e);
  return T2S_OK;
}
