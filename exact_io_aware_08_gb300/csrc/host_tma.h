// Host side of TMA: build the 3-D tensor maps the kernels load and store through.
//
// Every [B, H, N, d] bf16 tensor is described as a 3-D tensor {d, N, B*H} (innermost first), so
// a 128-row box that runs past the end of one head's sequence reads zeros instead of the next
// head's rows, and a store clips those rows.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      return nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// bf16 tensor {inner, rows, planes} with dense strides; box {box_inner, box_rows, 1};
// 128-byte swizzle (box_inner * 2 must be <= 128).  Out-of-bounds elements read as zero.
inline bool make_map_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint64_t planes, uint32_t box_inner, uint32_t box_rows,
                             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 8-bit tensor {inner, rows, planes} (e4m3 codes) with dense strides; box {box_inner, box_rows, 1}
// in bytes; 128-byte swizzle (box_inner <= 128).
inline bool make_map_u8_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                           uint64_t planes, uint32_t box_inner, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {inner, inner * rows};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Packed token-major bf16 tensor [total, H, d] as {d, H, total}: box {box_inner, 1, box_rows}
// covers box_rows consecutive tokens of one head and lands in shared memory exactly like the
// [B, H, N, d] box above.
inline bool make_map_bf16_tok(CUtensorMap* map, const void* base, uint64_t d, uint64_t heads,
                              uint64_t total, uint32_t box_inner, uint32_t box_rows,
                              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d, heads, total};
  const cuuint64_t strides[2] = {d * 2, d * heads * 2};
  const cuuint32_t box[3] = {box_inner, 1, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 tensor {d0, d1, d2} with byte strides (stride1, stride2) for dims 1 and 2; box
// {b0, b1, b2}; no swizzle (a row-major box in shared memory).
// ``sw128``: the shared-memory box uses the 128-byte swizzle (inner box extent 32 floats).
inline bool make_map_f32_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0,
                            uint32_t b1, uint32_t b2, bool sw128 = false) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa
