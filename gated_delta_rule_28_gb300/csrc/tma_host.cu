// Host side of the TMA loads: 2-D tensor maps over row-major bf16 matrices,
// 64 x 64-element boxes with the 128-byte swizzle, so that a box lands in shared
// memory as one K-block of the K-major operand layout used by the tensor-core
// kernels. The encoder is the driver's cuTensorMapEncodeTiled, reached through the
// runtime's entry-point query (no link-time dependence on the driver library).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"

namespace gdn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

cudaError_t make_tmap_bf16(TmaMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes) {
  static_assert(sizeof(TmaMap) == sizeof(CUtensorMap), "tensor map storage");
  auto fn = encoder();
  if (!fn) return cudaErrorNotSupported;
  if (!base || (reinterpret_cast<uintptr_t>(base) & 15u) || (row_bytes & 15u) || cols < 64 || rows < 1)
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_f32_32x128(TmaMap *map, const void *base, uint64_t rows) {
  auto fn = encoder();
  if (!fn) return cudaErrorNotSupported;
  if (!base || (reinterpret_cast<uintptr_t>(base) & 15u) || rows < 128) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128 * sizeof(float)};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gdn
