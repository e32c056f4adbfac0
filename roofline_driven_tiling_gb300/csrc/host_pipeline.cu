// host_pipeline.cu -- C = A x B for matrices in host memory, with the host<->device copies
// overlapped with the product.
//
// Two schedules, whichever leaves fewer bytes to copy before the first product can start:
//
// Row blocks. The product needs all of B but only a row block of A for a row block of C:
// copy B; then for each row block i of A, copy it, multiply it (on one of two compute
// streams, so consecutive blocks can share the GPU), and copy the block of C back as soon
// as it is done. The copy of B and of the first block of A are exposed.
//
// K chunks. The product over K chunk j needs only the columns of A and the rows of B in that
// chunk: copy chunk j of A (a strided copy of M rows) and of B while chunk j - 1 is being
// multiplied. Each chunk's product resumes from the accumulators the previous one stored in C
// (an FP32 value stored and reloaded is the same value, so the chain of fused multiply-adds
// and the result are those of one pass over K). Once the operands have arrived (estimated
// from the copy and FLOP rates), the rest of K runs as row blocks on two streams, each block
// of C copied back as soon as it is done, so that the copy back overlaps the products. Only
// the first chunk of A and B is exposed before the products start.
//
// Host->device and device->host copies use separate copy streams, so both directions run
// under the products; the last block of C is copied back after the products in both.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "t2s_internal.h"

namespace t2s {
namespace {

// Schedule settings (measured at 2048^3 to 8192^3 on GB300; the alternatives tried are
// within 1.5 % or slower). Row blocks have at least kMinRows rows and run on kConcurrent
// compute streams. K chunks hold about kKChunk values (a multiple of 32); the first and the
// last take 1 / kEdgeDiv of that, so that the products start sooner, and half that from
// kLargeOutputs elements of C on, where even the short first chunk's product covers the copy
// of the next chunk (end to end, 4096^3: 57.8 against 57.1 TFLOP/s; 8192^2 x 4096: 62.9
// against 62.5; at 2048^3 the shorter edge measured 4 % slower). The rest of K after the
// switch runs in row blocks of kTailRows. The switch comes once the operands have arrived,
// estimated from a copy rate of kCopyGBs and a product rate of kTflops.
constexpr int64_t kMinRows = 1024;
constexpr int kConcurrent = 2;
constexpr int64_t kKChunk = 1024;
constexpr int64_t kEdgeDiv = 2;
constexpr int64_t kLargeOutputs = int64_t{1} << 23;
constexpr int64_t kTailRows = 1024;
constexpr double kCopyGBs = 200.0;
constexpr double kTflops = 60.0;

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
  cudaEvent_t chunks_done = nullptr;
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
    if ((e = make_event(&r.chunks_done)) != cudaSuccess) return e;
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

  // Row blocks of at least kMinRows rows (1024 measured best at 3072^3 to 4096^3),
  // at most kMaxBlocks of them.
  int nb = static_cast<int>(M / kMinRows);
  nb = nb < 1 ? 1 : nb > kMaxBlocks ? kMaxBlocks : nb;
  const int64_t rows_per = (M + nb - 1) / nb;

  // K chunk boundaries: an edge chunk, whole chunks of about kKChunk values, an
  // edge chunk; at most kMaxBlocks chunks, every boundary but K a multiple of 32.
  const int64_t kt = kKChunk / 32 * 32;
  const int64_t edge_div = M * N >= kLargeOutputs ? 2 * kEdgeDiv : kEdgeDiv;
  const int64_t edge = (kt / edge_div + 31) / 32 * 32;
  int64_t kb[kMaxBlocks + 1] = {0};
  int nk = 0;
  if (has_ab && K > 2 * edge) {
    const int64_t mid = K - 2 * edge;
    int64_t m = (mid + kt - 1) / kt;
    m = m > kMaxBlocks - 2 ? kMaxBlocks - 2 : m;
    const int64_t step = m > 0 ? ((mid + m - 1) / m + 31) / 32 * 32 : 0;
    kb[++nk] = edge;
    for (int64_t i = 0; i < m && kb[nk] + step < K; ++i, ++nk) kb[nk + 1] = kb[nk] + step;
    kb[++nk] = K;
  }
  // The K-chunk schedule when it has at least two chunks and exposes fewer bytes.
  const bool by_k = nk >= 2 && kb[1] * (M + N) < K * (N + rows_per);
  // The rest of K after the switch runs in row blocks of kTailRows.
  if (by_k) {
    nb = static_cast<int>(M / kTailRows);
    nb = nb < 1 ? 1 : nb > kMaxBlocks ? kMaxBlocks : nb;
  }
  const int64_t rows_blk = (M + nb - 1) / nb;

  // Everything starts after the work already enqueued on the caller's stream.
  if ((e = cudaEventRecord(r->start, s)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(r->copy_in, r->start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(r->copy_out, r->start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(r->compute2, r->start, 0)) != cudaSuccess) return fail(e);
  int64_t last_k0 = 0;
  if (by_k) {
    // Chunk j of A (columns k0 .. k0 + kj - 1 of every row) and of B (rows k0 .. k0 + kj - 1);
    // the products of the first chunks, each resuming from C, on the caller's stream.
    for (int j = 0; j < nk; ++j) {
      const int64_t k0 = kb[j], kj = kb[j + 1] - kb[j];
      if ((e = cudaMemcpy2DAsync(dA + k0, static_cast<size_t>(K) * sizeof(float), hA + k0,
                                 static_cast<size_t>(K) * sizeof(float),
                                 static_cast<size_t>(kj) * sizeof(float), static_cast<size_t>(M),
                                 cudaMemcpyHostToDevice, r->copy_in)) != cudaSuccess)
        return fail(e);
      if ((e = cudaMemcpyAsync(dB + k0 * N, hB + k0 * N, static_cast<size_t>(kj) * N * sizeof(float),
                               cudaMemcpyHostToDevice, r->copy_in)) != cudaSuccess)
        return fail(e);
      if ((e = cudaEventRecord(r->a_ready[j], r->copy_in)) != cudaSuccess) return fail(e);
    }
    // The chunks multiplied over all rows: enough of them to cover the copies, after which
    // the row blocks take the rest of K (their C blocks then go back while later blocks
    // compute). The copy of the operands takes about (M + N) K 4 bytes / copy rate, the
    // product 2 M N K / FLOP rate.
    const double copy_s = 4.0 * static_cast<double>(M + N) * K / (kCopyGBs * 1e9);
    const double per_k_s = 2.0 * static_cast<double>(M) * N / (kTflops * 1e12);
    const double k_cover = copy_s / per_k_s;
    int p = 1;
    while (p < nk - 1 && static_cast<double>(kb[p]) < k_cover) ++p;
    for (int j = 0; j < p; ++j) {
      if ((e = cudaStreamWaitEvent(s, r->a_ready[j], 0)) != cudaSuccess) return fail(e);
      const int rc = gemm_f32_kchunk(M, N, K, dA, dB, dC, stream, 1, kb[j], kb[j + 1] - kb[j],
                                     j > 0);
      if (rc != T2S_OK) return rc;
    }
    if ((e = cudaEventRecord(r->chunks_done, s)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(r->compute2, r->chunks_done, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(s, r->a_ready[nk - 1], 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(r->compute2, r->a_ready[nk - 1], 0)) != cudaSuccess) return fail(e);
    last_k0 = kb[p];
  } else if (has_ab) {
    if ((e = cudaMemcpyAsync(dB, hB, static_cast<size_t>(K) * N * sizeof(float),
                             cudaMemcpyHostToDevice, r->copy_in)) != cudaSuccess)
      return fail(e);
    if ((e = cudaEventRecord(r->b_ready, r->copy_in)) != cudaSuccess) return fail(e);
  }
  // Row blocks: the whole product of each block (row-block schedule) or the rest of its K.
  // Chunk sizes passed on are rounded up to 32; the kernels stop at K.
  const int64_t last_kc = (K - last_k0 + 31) / 32 * 32;
  for (int i = 0; i < nb; ++i) {
    const int64_t r0 = i * rows_blk;
    if (r0 >= M) break;
    const int64_t rows = (r0 + rows_blk <= M) ? rows_blk : M - r0;
    const cudaStream_t cs = (i & 1) ? r->compute2 : s;
    if (has_ab && !by_k) {
      if ((e = cudaMemcpyAsync(dA + r0 * K, hA + r0 * K, static_cast<size_t>(rows) * K * sizeof(float),
                               cudaMemcpyHostToDevice, r->copy_in)) != cudaSuccess)
        return fail(e);
      if ((e = cudaEventRecord(r->a_ready[i], r->copy_in)) != cudaSuccess) return fail(e);
      if ((e = cudaStreamWaitEvent(cs, r->a_ready[i], 0)) != cudaSuccess) return fail(e);
    }
    // Blocks alternate between two compute streams, so two of them share the GPU.
    const int conc = nb > 1 ? kConcurrent : 1;
    const float* a_blk = has_ab ? dA + r0 * K : nullptr;
    const float* b_all = has_ab ? dB : nullptr;
    const t2s_stream_t ts = reinterpret_cast<t2s_stream_t>(cs);
    const int rc = by_k ? gemm_f32_kchunk(rows, N, K, a_blk, b_all, dC + r0 * N, ts, conc, last_k0,
                                          last_kc, true)
                        : gemm_f32_block(rows, N, K, a_blk, b_all, dC + r0 * N, ts, conc);
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
