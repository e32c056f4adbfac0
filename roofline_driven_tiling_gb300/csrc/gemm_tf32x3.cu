// gemm_tf32x3.cu -- 3xTF32 tensor-core product (tcgen05 + TMEM).
#include <cuda_runtime.h>

#include "t2s_internal.h"

namespace t2s {

// Split planes: A_big, A_small (M x K) and B_big, B_small (N x K), 4 bytes each.
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const size_t a = static_cast<size_t>(M) * K * 4, b = static_cast<size_t>(N) * K * 4;
  const auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return 2 * up(a) + 2 * up(b);
}

cudaError_t launch_tf32x3(const Problem&, void*) { return cudaErrorNotSupported; }

}  // namespace t2s
