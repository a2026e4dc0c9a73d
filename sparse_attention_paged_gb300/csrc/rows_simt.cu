// rows_simt.cu -- first, plain CUDA-core version of the indexer logits
// (one CTA per (row, page)); used to bring up the ABI before the tensor-core
// kernels land.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {

__global__ void __launch_bounds__(256) rows_simt_kernel(RowsParams p) {
  const int page = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int T = p.W * kPage;
  const int L = p.seqlens[r];
  float* orow = p.out + (long long)r * p.out_stride + (long long)page * kPage;

  if (L > T) {
    if (tid < kPage) orow[tid] = __int_as_float(0x7fc00000);
    if (tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
    return;
  }
  if (page * kPage >= L) {  // whole page past the row's length
    if (tid < kPage) orow[tid] = -INFINITY;
    return;
  }
  const int phys = p.block_table[(long long)r * p.bt_stride + page];
  if (phys < 0 || phys >= p.num_pages) {
    if (tid < kPage)
      orow[tid] = (page * kPage + tid < L) ? __int_as_float(0x7fc00000) : -INFINITY;
    if (tid == 0) raise_status(p.status, DSA_ERR_BAD_PAGE);
    return;
  }

  __shared__ float qs[kHeads][kDim + 1];
  __shared__ float ks[8][kDim];
  __shared__ float ws[kHeads];
  const uint16_t* qrow = p.q + (long long)r * kHeads * kDim;
  for (int i = tid; i < kHeads * kDim; i += blockDim.x) {
    __nv_bfloat16_raw raw;
    raw.x = qrow[i];
    qs[i / kDim][i % kDim] = __bfloat162float(__nv_bfloat16(raw));
  }
  if (tid < kHeads) ws[tid] = p.w[(long long)r * kHeads + tid];
  __syncthreads();

  const uint8_t* pg = p.kcache + (long long)phys * p.page_stride;
  for (int j = warp; j < kPage; j += 8) {
    const int t = page * kPage + j;
    if (t >= L) {
      if (lane == 0) orow[j] = -INFINITY;
      continue;
    }
    for (int i = 0; i < 4; ++i) {
      const int d = lane * 4 + i;
      float v;
      if (p.kv_dtype == DSA_KV_FP8_E4M3) {
        __nv_fp8_e4m3 f;
        f.__x = pg[j * kDim + d];
        v = float(f);
      } else {
        __nv_bfloat16_raw raw;
        raw.x = reinterpret_cast<const uint16_t*>(pg)[j * kDim + d];
        v = __bfloat162float(__nv_bfloat16(raw));
      }
      ks[warp][d] = v;
    }
    __syncwarp();
    float d0 = 0.f, d1 = 0.f;
    for (int d = 0; d < kDim; ++d) {
      const float kv = ks[warp][d];
      d0 = fmaf(qs[lane][d], kv, d0);
      d1 = fmaf(qs[lane + 32][d], kv, d1);
    }
    float v = ws[lane] * fmaxf(d0, 0.f) + ws[lane + 32] * fmaxf(d1, 0.f);
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) {
      float s = 1.f;
      if (p.kscale != nullptr)
        s = reinterpret_cast<const float*>(p.kscale + (long long)phys * p.page_stride)[j];
      orow[j] = s * v;
    }
    __syncwarp();
  }
}

cudaError_t launch_rows_simt(const RowsParams& p, cudaStream_t stream) {
  dim3 grid(p.W, p.rows);
  rows_simt_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
