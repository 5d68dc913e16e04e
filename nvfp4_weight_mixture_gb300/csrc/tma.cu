// Host-side TMA tensor-map encoding (driver entry point fetched through the
// runtime, so the library links only against cudart).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace moe {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

}  // namespace

// A byte matrix of `rows` rows of `row_bytes` bytes (row_bytes a multiple of
// 16, base 16-byte aligned) seen as 8-byte elements; a box is `box_bytes` x
// `box_rows`.  Rows past the end read as zeros.
cudaError_t make_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                          uint32_t box_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (row_bytes & 15u) || (box_bytes & 15u) ||
      box_bytes / 8 > 256 || box_rows > 256 || box_rows == 0)
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {row_bytes / 8, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes / 8, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// FP16 matrix of `rows` x `cols` (row pitch cols * 2 bytes, a multiple of 16),
// box `box_cols` x `box_rows`, optionally with the 128-byte swizzle (then
// box_cols * 2 must be 128).  Rows and columns past the end read as zeros.
cudaError_t make_fp16_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                          uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || ((cols * 2) & 15u) || box_cols > 256 ||
      box_rows > 256 || box_rows == 0 || ((box_cols * 2) & 15u) ||
      (swizzle128 && box_cols * 2 != 128))
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// FP16 matrix of `rows` x `cols` (cols % 64 == 0) seen as 64-element segments:
// dimensions (64 elements, rows, cols / 64) with strides (2 cols, 128) bytes,
// so that one box of 64 x box_rows x box_segs lands as box_segs consecutive K
// segments, each a tile of box_rows rows of 128 bytes (row r of segment c at
// row c * box_rows + r of the box, 128-byte swizzled).  Rows and segments
// past the end read as zeros.
cudaError_t make_fp16_segments_map(CUtensorMap* map, const void* base, uint64_t cols,
                                   uint64_t rows, uint32_t box_rows, uint32_t box_segs) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (cols % 64) || box_rows > 256 ||
      box_rows == 0 || box_segs == 0 || box_segs > 256)
    return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, box_segs};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_fp16_map_swz(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                              uint32_t box_cols, uint32_t box_rows, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMapSwizzle sw;
  switch (swizzle_bytes) {
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return cudaErrorInvalidValue;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || ((cols * 2) & 15u) || box_cols > 256 ||
      box_rows > 256 || box_rows == 0 || ((box_cols * 2) & 15u) ||
      (swizzle_bytes && box_cols * 2 != (uint32_t)swizzle_bytes))
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace moe
