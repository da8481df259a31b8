// tmap.h -- host-side TMA tensor-map encoding through the driver entry point
// (no link-time dependency on libcuda).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace ca {

inline PFN_cuTensorMapEncodeTiled_v12000 get_encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with a box of
// [box_rows, box_cols] elements and 128-byte swizzle (box_cols * 2 == 128).
// Out-of-range rows read as zero.  Returns false on failure.
inline bool encode_bf16_2d_sw128(CUtensorMap* map, const void* base, uint64_t rows,
                                 uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  auto fn = get_encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over `depth` matrices of [rows, cols] (row stride
// cols elements, matrix stride `mat_stride_elems`), box [1, box_rows,
// box_cols], 128-byte swizzle.  Rows >= `rows` read as zero, which is how a
// caller masks the unused tail of a cache or shard.
inline bool encode_bf16_3d_sw128(CUtensorMap* map, const void* base, uint64_t depth,
                                 uint64_t rows, uint64_t cols, uint64_t mat_stride_elems,
                                 uint32_t box_rows, uint32_t box_cols) {
  auto fn = get_encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, depth};
  cuuint64_t strides[2] = {cols * 2, mat_stride_elems * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor map over a row-major [rows, 128] matrix seen as three
// dimensions -- 64 columns, rows, and the two 64-column halves of a row -- so
// that one box of [2, box_rows, 64] brings both halves of box_rows rows,
// stored half after half: [half][row][64], each 128-byte row swizzled as
// in a [box_rows, 64] box.  Rows >= `rows` read as zero.
inline bool encode_bf16_halves_sw128(CUtensorMap* map, const void* base, uint64_t rows,
                                     uint32_t box_rows) {
  auto fn = get_encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, 2};
  cuuint64_t strides[2] = {256, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ca
