// store_sm103.cu -- the key-cache producer: new key rows (bf16, D = 128) go
// into their slots of the paged cache, as e4m3 codes plus a per-position
// fp32 scale in the fused 8,448-byte page, or as bf16 (256 bytes per
// position).  The page layouts are those the indexer kernels read ("The
// Dispatch Wire: Connecting a Triton Indexer Kernel to Production
// Inference", section "The Reasoning and Decision-Making"; "The Dispatch
// Decision: Wiring a Triton Kernel into Production", section "The Problem
// That Led Here").  The pages give no quantisation rule; the one used here
// maps the row's largest |k| to e4m3's largest finite value:
//
//   s = max_d |k_d| / 448   (s = 1 for an all-zero row)
//   code_d = e4m3(k_d / s), round to nearest even, saturated to +-448
//
// with every step in fp32, so that k_d ~ code_d * s is what the indexer's
// position scale undoes.
//
// A warp takes four key rows, loading all of them before it converts any (the
// rows' latency overlaps); per row, lane l holds d = 4l .. 4l+3 (8 bytes of
// bf16), a warp max gives s, the lane writes its 4 codes (the warp's 128
// bytes are one coalesced store) and lane 0 the scale.  HBM-bound: 256 bytes
// read and 132 (fp8) or 256 (bf16) written per row.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {

namespace {

constexpr int kStoreWarps = 8;                 // warps per block
constexpr int kRowsPerWarp = 4;
constexpr int kFp8ScaleOffset = kPage * kDim;  // 8,192: the scales follow the codes

struct StoreParams {
  const uint16_t* k;          // bf16 bits [n, 128]
  const int* slots;           // [n]: page * 64 + slot, < 0 = skip
  uint8_t* kcache;
  long long page_stride;
  int num_pages;
  int n;
  int* status;
};

template <int KV>
__global__ void __launch_bounds__(kStoreWarps * 32)
    store_kernel(const StoreParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long i0 = ((long long)blockIdx.x * kStoreWarps + warp) * kRowsPerWarp;
  // the rows and slots may have been written by the previous launch
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  // every row's load first, so that a warp has kRowsPerWarp rows in flight
  uint2 raw[kRowsPerWarp];
  int slot_all[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const long long i = i0 + r;
    slot_all[r] = i < p.n ? __ldg(p.slots + i) : -1;
    raw[r] = i < p.n ? __ldg(reinterpret_cast<const uint2*>(p.k + i * kDim) + lane)
                     : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    if (slot_all[r] < 0) continue;                   // warp-uniform
    const int page = slot_all[r] / kPage, slot = slot_all[r] % kPage;
    if (page >= p.num_pages) {
      if (lane == 0) raise_status(p.status, DSA_ERR_BAD_PAGE);
      continue;
    }
    uint8_t* pg = p.kcache + (long long)page * p.page_stride;
    if (KV == DSA_KV_BF16) {
      *reinterpret_cast<uint2*>(pg + slot * (kDim * 2) + lane * 8) = raw[r];
      continue;
    }
    const float x[4] = {__uint_as_float(raw[r].x << 16), __uint_as_float(raw[r].x & 0xffff0000u),
                        __uint_as_float(raw[r].y << 16), __uint_as_float(raw[r].y & 0xffff0000u)};
    float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
    uint32_t codes = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __nv_fp8_storage_t c =
          __nv_cvt_float_to_fp8(__fdiv_rn(x[u], s), __NV_SATFINITE, __NV_E4M3);
      codes |= (uint32_t)c << (8 * u);
    }
    *reinterpret_cast<uint32_t*>(pg + slot * kDim + lane * 4) = codes;
    if (lane == 0) *reinterpret_cast<float*>(pg + kFp8ScaleOffset + slot * 4) = s;
  }
}

template <int KV>
cudaError_t launch_store_t(const StoreParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.n + kStoreWarps * kRowsPerWarp - 1) / (kStoreWarps * kRowsPerWarp));
  cfg.blockDim = dim3(kStoreWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, store_kernel<KV>, p);
}

}  // namespace

cudaError_t launch_store(const uint16_t* k, const int* slots, int n, uint8_t* kcache,
                         long long page_stride, int num_pages, int kv_dtype, int* status,
                         cudaStream_t stream) {
  const StoreParams p{k, slots, kcache, page_stride, num_pages, n, status};
  if (kv_dtype == DSA_KV_FP8_E4M3) return launch_store_t<DSA_KV_FP8_E4M3>(p, stream);
  return launch_store_t<DSA_KV_BF16>(p, stream);
}

}  // namespace dsa
