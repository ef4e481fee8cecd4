// tmap.h — host-side TMA tensor-map encoding for [batch, rows, heads, D] tensors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace mslk {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (no link-time dependency on libcuda); null if the
// driver does not provide it.
inline EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 (or, with u8, one-byte E4M3) [batch, rows, heads, D] with free strides (elements)
// -> 4-D tiled map with a box_d x box_rows box and no swizzle (rows land densely in shared
// memory, D elements each).  Dimensions of extent 1 get a dummy stride (never stepped over).
inline bool encode_rows_plain(EncodeTiledFn enc, CUtensorMap* map, const void* base, int D,
                              long long rows, long long heads, long long batch, long long s_m,
                              long long s_h, long long s_b, int box_d, int box_rows, bool u8 = false) {
  const long long elt = u8 ? 1 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  long long st_m = s_m * elt;
  long long st_h = heads > 1 ? s_h * elt : st_m * rows;
  long long st_b = batch > 1 ? s_b * elt : st_h * heads;
  if (rows == 1) st_m = 16;
  if (st_m <= 0 || st_m % 16) st_m = 16;
  if (st_h <= 0 || st_h % 16) st_h = 16;
  if (st_b <= 0 || st_b % 16) st_b = 16;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st_m), static_cast<cuuint64_t>(st_h),
                           static_cast<cuuint64_t>(st_b)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mslk
