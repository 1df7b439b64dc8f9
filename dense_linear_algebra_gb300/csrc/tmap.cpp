// tmap.cpp — tensor-map encoding for the tensor copies (see tmap.h).
#include "tmap.h"

#include <mutex>

#include <cuda_runtime.h>

namespace fxtx {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
    cudaGetLastError();
  });
  return fn;
}

}  // namespace

bool encode_rows_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t rows, int64_t cols,
                     int64_t pitch_bytes, int elem, int box_rows, int box_bytes, int swizzle) {
  EncodeFn fn = encode_fn();
  if (!fn || box_bytes % 16 != 0 || (swizzle != 0 && swizzle != box_bytes) ||
      (swizzle != 0 && swizzle != 32 && swizzle != 64 && swizzle != 128))
    return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(box_bytes / elem), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle == 0    ? CU_TENSOR_MAP_SWIZZLE_NONE
                        : swizzle == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                        : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                        : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fxtx
