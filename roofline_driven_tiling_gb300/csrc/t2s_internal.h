// t2s_internal.h -- declarations shared by the library's translation units.
// Not part of the public C ABI (that is include/t2s_gemm.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/t2s_gemm.h"

namespace t2s {

// Bounded barrier waits give up after this long (2 s); a correct kernel never
// waits more than microseconds on one barrier.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// One validated product: sizes, device pointers, stream, and the device status
// word the kernels record bounded-wait failures in.
struct Problem {
  int64_t M, N, K;
  const float* A;
  const float* B;
  float* C;
  cudaStream_t stream;
  unsigned* status;
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_naive(const Problem& p);
cudaError_t launch_smem32(const Problem& p);
cudaError_t launch_ffma(const Problem& p);
// The product when `concurrent` products of the same size run on the GPU at once (the
// configuration is chosen for all their tiles together); the same bits as launch_ffma.
cudaError_t launch_ffma_concurrent(const Problem& p, int concurrent);
// The product over the K values [k0, k0 + kc) only (kc > 0; k0 and kc multiples of 32,
// k0 < K), added onto the values already in p.C when `accumulate` is set: the accumulators
// resume from C, so consecutive chunks give the same bits as one pass over K.
cudaError_t launch_ffma_range(const Problem& p, int concurrent, int64_t k0, int64_t kc,
                              bool accumulate);
// The configuration the product takes (the codes of t2s_gemm_f32_plan).
int ffma_plan(int64_t M, int64_t N, int64_t K, int sms);
// t2s_gemm_f32 for a block of a larger computation that runs beside `concurrent - 1` others.
int gemm_f32_block(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                   t2s_stream_t stream, int concurrent);
// The same for the K values [k0, k0 + kc) of the product, added onto C when `accumulate`
// is set (see launch_ffma_range).
int gemm_f32_kchunk(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                    t2s_stream_t stream, int concurrent, int64_t k0, int64_t kc, bool accumulate);
// Split K: `splits` requested chunks (>= 1); partial products in `workspace`
// (splitk_planes(K, splits) planes of M x N floats), summed into p.C in plane order.
int splitk_auto(int64_t M, int64_t N, int64_t K);
// The automatic chunk count on a GPU with `sms` multiprocessors (1: no split).
int splitk_choice(int64_t M, int64_t N, int64_t K, int sms);
int splitk_planes(int64_t K, int splits);
cudaError_t launch_ffma_splitk(const Problem& p, int splits, float* workspace);
// Stream K: the flattened tile x k-block space shared evenly over two CTAs per SM, partial
// tiles of shared tiles in `workspace` (streamk_workspace_bytes), added by a fixup kernel.
// Needs the TMA path (streamk_supported).
size_t streamk_workspace_bytes(int64_t M, int64_t N, int64_t K);
bool streamk_supported(const Problem& p);
cudaError_t launch_ffma_streamk(const Problem& p, float* workspace);
// The product on a persistent grid (2 CTAs per SM, one TMA ring across tiles); TMA path
// only (K % 4 == 0, N % 4 == 0, 16-byte aligned A and B). The bits of launch_ffma.
cudaError_t launch_ffma_persistent(const Problem& p);
// The persistent product with a TMA-store epilogue (256 x 128 tiles, one CTA per SM) for short
// K; the bits of launch_ffma. Needs the TMA path and a 16-byte aligned C (pstore_ok).
cudaError_t launch_ffma_pstore(const Problem& p);
bool pstore_ok(const Problem& p);
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_tf32x3(const Problem& p, void* workspace);
// BF16 or FP16 operands (uint16_t bit patterns), FP32 C; workspace for the transposed/padded
// planes (the same size for both formats).
size_t half_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_bf16(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                        float* C, void* workspace, cudaStream_t stream, unsigned* status);
cudaError_t launch_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                       float* C, void* workspace, cudaStream_t stream, unsigned* status);
// FP64 (binary64) kernels: product, naive and 32 x 32 shared-memory comparison points.
cudaError_t launch_dgemm(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                         double* C, cudaStream_t stream);
cudaError_t launch_naive_f64(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                             double* C, cudaStream_t stream);
cudaError_t launch_smem32_f64(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                              double* C, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t stream);
// Throughput probes (probes.cu); *flops receives the FLOPs of the launch.
cudaError_t launch_ffma_probe(int64_t iters, float* out, cudaStream_t stream, int64_t* flops);
cudaError_t launch_tf32_mma_probe(int64_t iters, float* out, unsigned* status, cudaStream_t stream,
                                  int64_t* flops);
// Writes `value` to the M x N matrix C (M % 256 == 0, N % 128 == 0, checked by the caller) in
// the short-K product's store pattern: mode 0 TMA boxes, mode 1 16-byte stores from registers.
cudaError_t launch_store_probe(int64_t M, int64_t N, float* C, int mode, float value,
                               cudaStream_t stream, int64_t* bytes);
// Records a CUDA error for t2s_last_cuda_error() on this host thread.
void set_last_cuda_error(cudaError_t e);

}  // namespace t2s
