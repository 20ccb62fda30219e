// tmap.h -- host-side TMA tensor-map encoding (the driver's cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point so that the library needs no libcuda link line).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace k3 {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A row-major byte matrix [rows][row_bytes] seen as a 2-D tensor of uint8; boxes of
// box_rows x box_bytes land in shared memory row by row (128-byte swizzled when swz128).
// Out-of-range rows read as zero.  Returns false when the driver refuses the description.
inline bool make_map_2d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                        uint32_t box_bytes, uint32_t box_rows, bool swz128) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major byte tensor [outer][mid][inner_bytes] (strides mid_stride and outer_stride in
// bytes, multiples of 16) seen as 3-D; boxes of box_outer x 1 x box_bytes land in shared
// memory as box_outer rows of box_bytes (swizzled when swizzle != NONE).  Out-of-range
// coordinates read as zero.
inline bool make_map_3d(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t mid,
                        uint64_t mid_stride, uint64_t outer, uint64_t outer_stride,
                        uint32_t box_bytes, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || outer == 0 || mid == 0) return false;
  const cuuint64_t dims[3] = {inner_bytes, mid, outer};
  const cuuint64_t strides[2] = {mid_stride, outer_stride};
  const cuuint32_t box[3] = {box_bytes, 1, box_outer};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// make_map_2d with a chosen swizzle.
inline bool make_map_2d_sw(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                           uint32_t box_bytes, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace k3
