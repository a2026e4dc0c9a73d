// decode_sm103.cu -- decode kernel of the DSA indexer paged MQA-logits for
// GB300 (sm_103a): TMA page gathers through the block table, tcgen05 MMA with
// the accumulator in TMEM, and a fused ReLU / head-weight / scale epilogue.
//
// Grid (G, B), G = min(W, a per-dtype cap), fixed by the table width alone, so the
// launch never depends on the lengths and can be captured in a CUDA graph.
// CTA (c, b) owns the pages c, c+G, c+2G, ... of request b: with G = W this is
// one CTA per (request, page) ("The Dispatch Wire: Connecting a Triton
// Indexer Kernel to Production Inference", section "The Reasoning and
// Decision-Making"); a CTA whose first page lies past the request's length
// only writes -inf and exits ("The Moment the Context-Length Tax Vanished:
// Committing the O(actual) Triton Indexer", section "The Commit: Engineering
// as Narrative").  Work is O(actual length): pages past it are never read.
//
// Per valid page pair (a 128-position tile):
//   TMA      page rows -> shared memory (128-byte swizzle), no gathered copy
//            ("The Dispatch Decision: Wiring a Triton Kernel into
//            Production", section "The Problem That Led Here");
//   tcgen05  S[t, h] = sum_d k[t, d] * q[h, d], M = 128 positions, N = 64
//            heads, accumulator in TMEM (double-buffered);
//   epilogue each of 128 threads owns one position: relu, head weights and
//            the position's scale in registers, one coalesced store.
//
// fp8 keys are consumed as stored (e4m3, kind::f8f6f4).  The bf16 query is
// split once per CTA into two e4m3 terms with a power-of-two scale per head:
// q * 2^e_h = hi + lo, hi = e4m3(q * 2^e_h), lo = e4m3(q * 2^e_h - hi), with
// 2^e_h folded into the head weight.  hi + lo reproduces every bf16 value
// whose magnitude is at least ~2^-10 of its head's maximum exactly, and the
// rest to within 2^-18 of the head's maximum.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"
#include "tensor_maps.cuh"

namespace dsa {

using namespace sm100;

namespace {

#ifndef DSA_DEC_FP8_SLOTS
#define DSA_DEC_FP8_SLOTS 16
#endif
#ifndef DSA_DEC_BF16_SLOTS
#define DSA_DEC_BF16_SLOTS 32
#endif
#ifndef DSA_DEC_FP8_STAGES
#define DSA_DEC_FP8_STAGES 3
#endif
#ifndef DSA_DEC_FP8_CTAS
#define DSA_DEC_FP8_CTAS 3
#endif
#ifndef DSA_DEC_BF16_STAGES
#define DSA_DEC_BF16_STAGES 2
#endif
#ifndef DSA_DEC_BF16_CTAS
#define DSA_DEC_BF16_CTAS 2
#endif
constexpr int kDecThreads = 192;          // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr long long kWaitLimit = 2000000000ll;   // ~1 s of SM clock: bound on any wait

template <int KV>
struct DecCfg;

template <>
struct DecCfg<DSA_KV_FP8_E4M3> {
  static constexpr int kStages = DSA_DEC_FP8_STAGES;
  static constexpr int kCtasPerSm = DSA_DEC_FP8_CTAS;
  static constexpr int kMaxSlots = DSA_DEC_FP8_SLOTS;     // G cap: CTAs per request
  static constexpr int kPageBytes = kPage * kDim;         // 8 KB of e4m3 rows
  static constexpr int kTileBytes = 2 * kPageBytes;       // 128 rows x 128 B
  static constexpr int kQBytes = 2 * kHeads * kDim;       // hi + lo: 16 KB
};

template <>
struct DecCfg<DSA_KV_BF16> {
  static constexpr int kStages = DSA_DEC_BF16_STAGES;
  static constexpr int kCtasPerSm = DSA_DEC_BF16_CTAS;
  static constexpr int kMaxSlots = DSA_DEC_BF16_SLOTS;
  static constexpr int kPageBytes = kPage * kDim * 2;     // 16 KB
  static constexpr int kTileBytes = 2 * kPageBytes;       // 2 K-blocks x 128 rows x 128 B
  static constexpr int kQBytes = kHeads * kDim * 2;       // 16 KB
};

// Shared memory: [Q operand][A stages][control: barriers at +0, TMEM slot at
// +256, abort flag at +260, head weights at +512]; kCtasPerSm CTAs fit on an SM.
constexpr int kCtrlBytes = 1024;

template <int KV>
constexpr int dec_smem_bytes() {
  using C = DecCfg<KV>;
  return 1024 /* alignment slack */ + C::kQBytes + C::kStages * C::kTileBytes + kCtrlBytes;
}

__device__ __forceinline__ float nanf_() { return __int_as_float(0x7fc00000); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16f(uint32_t bits) { return __uint_as_float(bits << 16); }

// Round two floats to e4m3 (nearest-even, saturating); returns the two codes
// (first argument in the low byte) and their values as floats.
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b, float& fa, float& fb) {
  __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(s, __NV_E4M3);
  fa = __half2float(__half(__half_raw{h.x}));
  fb = __half2float(__half(__half_raw{h.y}));
  return static_cast<uint32_t>(s);
}

}  // namespace

template <int KV>
__global__ void __launch_bounds__(kDecThreads, DecCfg<KV>::kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const RowsParams p, const int G) {
  using C = DecCfg<KV>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // B operand(s)
  uint8_t* sA = smem + C::kQBytes;             // A stages
  uint8_t* ctrl = sA + S * C::kTileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;                 // [2]
  uint64_t* tempty = tfull + 2;                // [2]
  uint64_t* qbar = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 260);
  float* w_s = reinterpret_cast<float*>(ctrl + 512);     // 64 floats
  static_assert((2 * S + 5) * 8 <= 256, "control block overflow");

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, b = blockIdx.y;
  const int T = p.W * kPage;
  float* orow = p.out + (long long)b * p.out_stride;
  const int* btrow = p.block_table + (long long)b * p.bt_stride;

  // Prologue that reads no input: it may overlap the previous launch.
  if (tid == 128) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(qbar, KV == DSA_KV_BF16 ? 1 : 128);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&kmap);
    if (KV == DSA_KV_BF16) prefetch_tmap(&qmap);
  }
  griddep_wait();
  griddep_launch_dependents();

  // The row length, and (independent of it, so in parallel) the first
  // tile's block-table entries and, for fp8, the query and head weights.
  // All of these addresses are inside the caller's arrays whatever the
  // length; block-table entries past the length are read but never used.
  const int L = __ldg(p.seqlens + b);
  int bt0 = -1, bt1 = -1;
  if (tid == 128) {
    bt0 = __ldg(btrow + c);
    if (c + G < p.W) bt1 = __ldg(btrow + c + G);
  }
  uint2 qraw[16];
  float wv = 0.f;
  if (KV == DSA_KV_FP8_E4M3 && warp < 4) {
    const uint16_t* qrow = p.q + (long long)b * kHeads * kDim;
#pragma unroll
    for (int hh = 0; hh < 16; ++hh)
      qraw[hh] = __ldg(reinterpret_cast<const uint2*>(qrow + (warp * 16 + hh) * kDim) + lane);
    if (lane < 16) wv = __ldg(p.w + (long long)b * kHeads + warp * 16 + lane);
  }

  const bool bad_len = L > T;
  const int Lc = bad_len ? 0 : max(L, 0);
  const int npv = (Lc + kPage - 1) / kPage;             // valid pages of the row
  const int n_mine = npv > c ? (npv - 1 - c) / G + 1 : 0;

  // -inf (NaN for an over-long row) past the last valid page, split evenly
  // over the row's G CTAs in contiguous 16-byte-aligned chunks.
  {
    const int f0 = npv * kPage;
    int chunk = (T - f0 + G - 1) / G;
    chunk = (chunk + 3) & ~3;
    const long long beg = f0 + (long long)c * chunk;
    const long long end = min(beg + chunk, (long long)T);
    const float fv = bad_len ? nanf_() : -INFINITY;
    const float4 v4 = make_float4(fv, fv, fv, fv);
    if (n_mine == 0 || warp < 4) {
      const int nthr = (n_mine == 0) ? kDecThreads : 128;
      for (long long i = beg + 4 * tid; i < end; i += 4 * nthr)
        *reinterpret_cast<float4*>(orow + i) = v4;
    }
    if (bad_len && c == 0 && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
  }
  if (n_mine == 0) return;
  const int n_tiles = (n_mine + 1) >> 1;

  // Producer: page pair i of this CTA -> stage i % S.  pre0/pre1 are
  // block-table entries already loaded (-2: load here).
  auto issue_tile = [&](int i, int pre0, int pre1) {
    const int s = i % S;
    int phys[2];
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int k = 2 * i + h;
      phys[h] = -1;
      if (k < n_mine) {
        const int pre = h == 0 ? pre0 : pre1;
        const int ph = pre != -2 ? pre : __ldg(btrow + c + k * G);
        if (ph >= 0 && ph < p.num_pages) {
          phys[h] = ph;
          bytes += C::kPageBytes;
        }
      }
    }
    mbar_arrive_expect_tx(&full[s], bytes);
    uint8_t* st = sA + s * C::kTileBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (phys[h] < 0) continue;
      if (KV == DSA_KV_FP8_E4M3) {
        tma_load_3d(st + h * C::kPageBytes, &kmap, &full[s], 0, 0, phys[h]);
      } else {
        // K-block 0 (d 0..63) and K-block 1 (d 64..127), rows of 128 B
        tma_load_3d(st + h * (C::kPageBytes / 2), &kmap, &full[s], 0, 0, phys[h]);
        tma_load_3d(st + C::kTileBytes / 2 + h * (C::kPageBytes / 2), &kmap, &full[s], 64, 0,
                    phys[h]);
      }
    }
  };

  // The first S tiles go out before the setup barrier: this thread
  // initialised the barriers they signal.
  int issued = 0;
  if (tid == 128) {
    if (KV == DSA_KV_BF16) {
      mbar_arrive_expect_tx(qbar, C::kQBytes);
      tma_load_2d(sQ, &qmap, qbar, 0, b * kHeads);
      tma_load_2d(sQ + C::kQBytes / 2, &qmap, qbar, 64, b * kHeads);
    }
    const int first = min(S, n_tiles);
    for (int i = 0; i < first; ++i) issue_tile(i, i == 0 ? bt0 : -2, i == 0 ? bt1 : -2);
    issued = first;
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int i = issued; i < n_tiles; ++i) {
        const int s = i % S;
        if (!mbar_wait_bounded(&empty[s], ((i / S) - 1) & 1, kWaitLimit)) {
          *abort_flag = 1;
          raise_status(p.status, DSA_ERR_TIMEOUT);
          break;
        }
        if (*abort_flag) break;
        issue_tile(i, -2, -2);
        issued = i + 1;
      }
      // never leave the CTA with copies in flight: wait for the last use of
      // every stage (already complete on the normal path)
      for (int i = max(0, issued - S); i < issued; ++i)
        mbar_wait_bounded(&full[i % S], (i / S) & 1, kWaitLimit);
      if (KV == DSA_KV_BF16) mbar_wait_bounded(qbar, 0, kWaitLimit);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc =
          KV == DSA_KV_FP8_E4M3 ? instr_desc(0, 0, 128, kHeads) : instr_desc(1, 1, 128, kHeads);
      const uint32_t sQa = smem_u32(sQ);
      const uint32_t sAa = smem_u32(sA);
      bool ok = mbar_wait_bounded(qbar, 0, kWaitLimit);
      int issued = 0;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int s = i % S, a = i & 1;
        ok = mbar_wait_bounded(&full[s], (i / S) & 1, kWaitLimit);
        if (ok && i >= 2) ok = mbar_wait_bounded(&tempty[a], ((i >> 1) - 1) & 1, kWaitLimit);
        if (!ok || *abort_flag) break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * kHeads;
        const uint32_t st = sAa + s * C::kTileBytes;
        if (KV == DSA_KV_FP8_E4M3) {
          // A: 128 rows x 128 B; B: hi then lo, 64 rows x 128 B each; K = 32 per MMA
#pragma unroll
          for (int term = 0; term < 2; ++term) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(st + 32 * k, 1024);
              const uint64_t bd = smem_desc_sw128(sQa + term * 8192 + 32 * k, 1024);
              mma_f8f6f4(d, ad, bd, idesc, (term | k) != 0);
            }
          }
        } else {
          // two K-blocks of 64 bf16; K = 16 per MMA
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t kb = k >> 2, ko = (k & 3) * 32;
            const uint64_t ad = smem_desc_sw128(st + kb * (C::kTileBytes / 2) + ko, 1024);
            const uint64_t bd = smem_desc_sw128(sQa + kb * (C::kQBytes / 2) + ko, 1024);
            mma_f16(d, ad, bd, idesc, k != 0);
          }
        }
        mma_commit(&empty[s]);
        mma_commit(&tfull[a]);
        issued = i + 1;
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, DSA_ERR_TIMEOUT);
      }
      // the accumulators must be idle before TMEM is released
      if (issued > 0) {
        const int i = issued - 1;
        mbar_wait_bounded(&tfull[i & 1], (i >> 1) & 1, kWaitLimit);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 0-3
    if (KV == DSA_KV_FP8_E4M3) {
      // split q[b] into e4m3 hi + lo with a power-of-two scale per head;
      // warp w owns heads 16w..16w+15, lane l owns d = 4l..4l+3 (loaded above)
#pragma unroll
      for (int hh = 0; hh < 16; ++hh) {
        const int h = warp * 16 + hh;
        float x[4] = {bf16f(qraw[hh].x & 0xffffu), bf16f(qraw[hh].x >> 16),
                      bf16f(qraw[hh].y & 0xffffu), bf16f(qraw[hh].y >> 16)};
        float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        m = warp_max(m);
        int e = 0;
        if (m > 0.f) {
          const int E = ((__float_as_int(m) >> 23) & 0xff) - 127;   // floor(log2 m), m normal
          e = min(max(7 - E, -126), 126);
        }
        const float sc = exp2i(e);
        uint32_t hi = 0, lo = 0;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
          const float a0 = x[j] * sc, a1 = x[j + 1] * sc;
          float h0, h1, l0, l1;
          const uint32_t hc = to_e4m3x2(a0, a1, h0, h1);
          const uint32_t lc = to_e4m3x2(a0 - h0, a1 - h1, l0, l1);
          hi |= hc << (8 * j);
          lo |= lc << (8 * j);
        }
        // row h, bytes [4*lane, 4*lane+4) of 128, 128-byte swizzle
        const uint32_t off = h * 128 + ((((lane >> 2) ^ (h & 7)) << 4) | ((lane & 3) << 2));
        *reinterpret_cast<uint32_t*>(sQ + off) = hi;
        *reinterpret_cast<uint32_t*>(sQ + 8192 + off) = lo;
        const float wh = __shfl_sync(0xffffffffu, wv, hh);
        if (lane == 0) w_s[h] = wh * exp2i(-e);
      }
      fence_proxy_async_smem();
      mbar_arrive(qbar);
    } else {
      if (tid < kHeads) w_s[tid] = __ldg(p.w + (long long)b * kHeads + tid);
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");

    const int r = warp * 32 + lane;            // accumulator row = TMEM lane
    const int half = r >> 6, slot = r & 63;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int a = i & 1;
      const int k = 2 * i + half;
      const bool row_valid = k < n_mine;
      const int page = c + k * G;
      const int t = page * kPage + slot;
      int phys = -1;
      float scale = 1.f;
      if (row_valid) {
        phys = __ldg(btrow + page);
        if (phys >= 0 && phys < p.num_pages && t < Lc && p.kscale != nullptr)
          scale = __ldg(reinterpret_cast<const float*>(p.kscale + (long long)phys * p.page_stride) +
                        slot);
      }
      if (ok) ok = mbar_wait_bounded(&tfull[a], (i >> 1) & 1, kWaitLimit);
      ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);   // warp-uniform for tcgen05.ld
      if (!ok) {
        if (row_valid) orow[t] = t < Lc ? nanf_() : -INFINITY;
        continue;
      }
      tc_fence_after();
      uint32_t v0[32], v1[32];
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + a * kHeads;
      tmem_ld_32x32b_x32(taddr, v0);
      tmem_ld_32x32b_x32(taddr + 32, v1);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[a]);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        const float4 wa = *reinterpret_cast<const float4*>(w_s + h);
        const float4 wb = *reinterpret_cast<const float4*>(w_s + 32 + h);
        acc0 = __ffma2_rn(make_float2(wa.x, wa.y),
                          make_float2(fmaxf(__uint_as_float(v0[h]), 0.f),
                                      fmaxf(__uint_as_float(v0[h + 1]), 0.f)), acc0);
        acc1 = __ffma2_rn(make_float2(wb.x, wb.y),
                          make_float2(fmaxf(__uint_as_float(v1[h]), 0.f),
                                      fmaxf(__uint_as_float(v1[h + 1]), 0.f)), acc1);
        acc0 = __ffma2_rn(make_float2(wa.z, wa.w),
                          make_float2(fmaxf(__uint_as_float(v0[h + 2]), 0.f),
                                      fmaxf(__uint_as_float(v0[h + 3]), 0.f)), acc0);
        acc1 = __ffma2_rn(make_float2(wb.z, wb.w),
                          make_float2(fmaxf(__uint_as_float(v1[h + 2]), 0.f),
                                      fmaxf(__uint_as_float(v1[h + 3]), 0.f)), acc1);
      }
      if (row_valid) {
        float o;
        if (t >= Lc) {
          o = -INFINITY;
        } else if (phys < 0 || phys >= p.num_pages) {
          o = nanf_();
          raise_status(p.status, DSA_ERR_BAD_PAGE);
        } else {
          o = scale * ((acc0.x + acc0.y) + (acc1.x + acc1.y));
        }
        orow[t] = o;
      }
    }
    if (!ok) raise_status(p.status, DSA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 128);
  }
}

// ----------------------------------------------------------------------------
// host side

// CTAs per request, from the launch shape only (never from the lengths, so
// a captured launch stays valid): at most the per-dtype cap and W; and for a
// short table (W <= 64 pages, so no request is long) small enough that all
// B * G CTAs fit in one wave on the GPU.
template <int KV>
int decode_slots(int W, int B, int resident_ctas) {
  int G = W < DecCfg<KV>::kMaxSlots ? W : DecCfg<KV>::kMaxSlots;
  if (W <= 64 && (long long)B * G > resident_ctas) G = resident_ctas / B;
  return G < 1 ? 1 : G;
}

template <int KV>
static cudaError_t launch_decode_t(const RowsParams& p, cudaStream_t stream) {
  // per device: the shared-memory opt-in and the number of resident CTAs
  static int resident_per_dev[kMaxDevices] = {0};
  constexpr int smem = dec_smem_bytes<KV>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (resident_per_dev[dev] == 0) {
    e = cudaFuncSetAttribute(decode_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared storage as shared memory, so that the
    // occupancy below (and at run time) is the shared-memory maximum
    e = cudaFuncSetAttribute(decode_kernel<KV>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<KV>,
                                                           kDecThreads, smem)) != cudaSuccess)
      return e;
    resident_per_dev[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int resident = resident_per_dev[dev];
  CUtensorMap kmap, qmap;
  if (!encode_kcache_map(&kmap, p)) return cudaErrorInvalidValue;
  if (KV == DSA_KV_BF16) {
    if (!encode_q_map(&qmap, p, 64)) return cudaErrorInvalidValue;
  } else {
    memset(&qmap, 0, sizeof qmap);
  }
  const int G = decode_slots<KV>(p.W, p.rows, resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, p.rows);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<KV>, kmap, qmap, p, G);
}

cudaError_t launch_decode(const RowsParams& p, cudaStream_t stream) {
  if (p.kv_dtype == DSA_KV_FP8_E4M3) return launch_decode_t<DSA_KV_FP8_E4M3>(p, stream);
  return launch_decode_t<DSA_KV_BF16>(p, stream);
}

}  // namespace dsa
