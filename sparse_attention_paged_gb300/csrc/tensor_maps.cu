// tensor_maps.cu -- TMA tensor-map encoding for the key pool and the queries.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tensor_maps.cuh"

namespace dsa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

// TMA moves a bounded number of elements per clock, so every map describes
// the data in 4-byte units (the bytes and the 128-byte-swizzled shared-memory
// image are the same as with the native element type): a 128-byte row of
// either dtype is 32 units.

// Key pool: dims {row bytes / 4, 64 slots, num_pages}, box = one page's
// 128-byte column block (fp8: the whole row; bf16: half a row, the second
// half at unit coordinate kHalfRowUnits).
bool encode_kcache_map(CUtensorMap* m, const RowsParams& p) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool bf16 = p.kv_dtype == DSA_KV_BF16;
  const cuuint64_t row_bytes = (cuuint64_t)kDim * (bf16 ? 2 : 1);
  cuuint64_t dims[3] = {row_bytes / 4, (cuuint64_t)kPage, (cuuint64_t)p.num_pages};
  cuuint64_t strides[2] = {row_bytes, (cuuint64_t)p.page_stride};
#ifndef DSA_FP8_BOX_ROWS
#define DSA_FP8_BOX_ROWS 64
#endif
  const cuuint32_t rows = bf16 ? (cuuint32_t)kPage : (cuuint32_t)DSA_FP8_BOX_ROWS;
  cuuint32_t box[3] = {32u, rows, 1u};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(p.kcache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Queries viewed as [rows * 64, 64 units] (a bf16 row of 128 values is 256
// bytes = 64 units), box {32 units, box_rows}; the second half-row at unit
// coordinate kHalfRowUnits.
bool encode_q_map(CUtensorMap* m, const RowsParams& p, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim * 2 / 4, (cuuint64_t)p.rows * kHeads};
  cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
  cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint16_t*>(p.q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa
