// tmap.cuh — host-side creation of TMA tensor maps.
//
// cuTensorMapEncodeTiled is a driver API function. The library reaches it
// through cudaGetDriverEntryPointByVersion, so it does not link libcuda and
// still loads on a machine without a GPU driver.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace uly {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once per process (thread-safe static initialisation); null if the
// driver does not provide it.
inline EncodeTiledFn encode_tiled_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// A rank-4 bf16 tensor [d3][d2][d1][d0] (d0 fastest, contiguous), tiled in
// boxes of box0 x 1 x 1 x box3 with 128-byte swizzle (box0 * 2 == 128 bytes).
// Out-of-range elements of a box read as zero.
inline bool make_tmap_bf16_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                              uint32_t box0, uint32_t box3, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  const cuuint32_t box[4] = {box0, 1, 1, box3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The two fp32 row planes of the backward, [2][nrows][pitch] (pitch a
// multiple of 4 floats; only the first `len` floats of a row are in the
// tensor, so reads past them return zero), in boxes of 128 x 1 x 2: the same
// 128 rows of both planes land as [plane][128] floats.
inline bool make_tmap_f32_rows(CUtensorMap* map, const void* base, uint64_t len, uint64_t nrows, uint64_t pitch) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || pitch % 4 != 0) return false;
  const cuuint64_t dims[3] = {len, nrows, 2};
  const cuuint64_t strides[2] = {pitch * 4, nrows * pitch * 4};
  const cuuint32_t box[3] = {128, 1, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace uly
