// Tensor maps (cuTensorMapEncodeTiled, through the runtime's driver entry point) for the TMA
// copies of the tensor-core kernels: bf16 tensors with the 128- or 64-byte swizzle, MN-major
// operand pairs as 64-column blocks, and 8-bit (e4m3 code) tensors.  Host only.
#pragma once

#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace moe {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Swizzle of a box whose inner extent is box_w bf16 elements (64 -> 128 bytes, 32 -> 64 bytes).
inline CUtensorMapSwizzle swizzle_for(uint32_t box_w) {
  return box_w == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
}

// 2D bf16 tensor [rows, width] (width contiguous) with a box of box_w x box_r.
inline bool map_2d(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint32_t box_w,
            uint32_t box_r) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {width, rows};
  const cuuint64_t strides[1] = {width * 2};
  const cuuint32_t box[2] = {box_w, box_r};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_w),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand pairs: [rows, width] bf16 (width a multiple of 64) seen as 64-column blocks,
// dims {64, rows, width / 64}, box {64, 64, 2}: one copy fills two 64 x 64 boxes back to back,
// the layout of two 2D boxes of columns c and c + 64.
inline bool map_mn2(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {64, rows, width / 64};
  const cuuint64_t strides[2] = {width * 2, 128};
  const cuuint32_t box[3] = {64, 64, 2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same for [G, rows, width] weights: dims {64, rows, width / 64, G}, box {64, 64, 2, 1}.
inline bool map_mn2_g(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint64_t G) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {64, rows, width / 64, G};
  const cuuint64_t strides[3] = {width * 2, 128, width * rows * 2};
  const cuuint32_t box[4] = {64, 64, 2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 8-bit tensors (e4m3 codes) [rows, width] and [G, rows, width], boxes of 128 x 128 (x 1): 128-byte
// rows with the 128-byte swizzle, the layout of a 64-wide bf16 box.
inline bool map_u8_2d(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {width, rows};
  const cuuint64_t strides[1] = {width};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool map_u8_3d(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint64_t G) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {width, rows, G};
  const cuuint64_t strides[2] = {width, width * rows};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D bf16 tensor [G, rows, width] with a box of box_w x box_r x 1.
inline bool map_3d(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint64_t G,
            uint32_t box_w, uint32_t box_r) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {width, rows, G};
  const cuuint64_t strides[2] = {width * 2, width * rows * 2};
  const cuuint32_t box[3] = {box_w, box_r, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_w),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows gathered by tile::gather4 from [rows, width] bf16 (token order): a box one row high and 64
// columns wide, 128-byte swizzle, so four gathered rows land like four rows of a 64-wide box.
inline bool map_gather_rows(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows) {
  return map_2d(m, base, width, rows, 64, 1);
}

}  // namespace moe
