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

// Tensor map over the key pool: dims {D values, 64 slots, num_pages}, box of
// one page (fp8: 128 B rows; bf16: 64-value half rows), 128-byte swizzle.
bool encode_kcache_map(CUtensorMap* m, const RowsParams& p) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool bf16 = p.kv_dtype == DSA_KV_BF16;
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)kPage, (cuuint64_t)p.num_pages};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * (bf16 ? 2 : 1), (cuuint64_t)p.page_stride};
  cuuint32_t box[3] = {bf16 ? 64u : 128u, (cuuint32_t)kPage, 1u};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                  const_cast<uint8_t*>(p.kcache), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map over q viewed as [rows * 64, 128] bf16, box {64 values, box_rows}.
bool encode_q_map(CUtensorMap* m, const RowsParams& p, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)p.rows * kHeads};
  cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa
