// t2s_tmap.cu -- TMA tensor-map encoding through the driver entry point.
#include "t2s_tmap.h"

#include <mutex>

namespace t2s {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled g_encode = nullptr;
cudaError_t g_lookup_error = cudaSuccess;
std::once_flag g_once;

void lookup() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  g_lookup_error = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
  if (g_lookup_error == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
    g_lookup_error = cudaErrorSymbolNotFound;
  if (g_lookup_error == cudaSuccess) g_encode = reinterpret_cast<EncodeTiled>(fn);
}

}  // namespace

cudaError_t encode_2d(CUtensorMap* map, CUtensorMapDataType type, uint32_t elem_bytes,
                      const void* base, int64_t cols, int64_t rows, uint32_t box_cols,
                      uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  std::call_once(g_once, lookup);
  if (g_encode == nullptr) return g_lookup_error;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = g_encode(map, type, 2, const_cast<void*>(base), dims, strides, box,
                              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_f32_2d(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, cols, rows, box_cols, box_rows,
                   swizzle);
}

cudaError_t encode_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                                uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, box_cols, box_rows,
                   swizzle);
}

}  // namespace t2s
