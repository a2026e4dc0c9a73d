// topk_sm103.cu -- top-k selection over each row's logits: the positions
// with the k largest logits, which sparse attention then reads.  The pages
// name the consumer ("The Dispatch Decision: Wiring a Triton Kernel into
// Production", section "The Problem That Led Here": the indexer scores the
// cached positions so that only the top-k enter attention); the selection
// itself is a plain definition.
//
// One CTA per row.  Logits become order-preserving 32-bit keys (a larger
// float gives a larger key; NaN, which only an error row holds, the smallest
// key).  A histogram of 2,048 linear bins over the row's range finds the bin
// of the k-th largest logit, and a three-pass radix select (11 + 11 + 10
// bits, shared-memory histograms) within that bin finds the k-th largest key
// K* and how many keys equal to it are needed.  A last pass writes, in position order, every position whose
// key is above K* and the first needed ones equal to it.  Rows of at most k
// valid positions take all of them; the rest of the k outputs is -1 (value
// -inf).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {

namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;

struct TopkParams {
  const float* logits;   // row r at logits + r * ld, positions [0, L_r) valid
  long long ld;
  const int* seqlens;
  int rows;
  int T;                 // W * 64
  int k;
  int* idx;              // row r at idx + r * out_stride, k entries
  float* vals;           // nullable, same layout
  long long out_stride;
  int* status;
  int cache_floats;      // rows up to this length are kept in shared memory
};

__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  if (v != v) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of one value per thread across the block; also returns the
// total.  `ws` holds kTkWarps entries.
__device__ __forceinline__ int block_exclusive_scan(int v, int* ws, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < kTkWarps ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kTkWarps) ws[lane] = s;      // inclusive per-warp prefix
  }
  __syncthreads();
  total = ws[kTkWarps - 1];
  const int base = warp > 0 ? ws[warp - 1] : 0;
  __syncthreads();                            // ws may be reused right away
  return base + x - v;
}

// Finds the bin holding the need-th largest entry of hist[0, nbins) counted
// from the top (nbins <= 2 * kTkThreads): every thread takes two bins, a
// block scan from the top gives each its count above; returns the bin and
// writes the count above it to *above.
__device__ __forceinline__ int find_bin(const uint32_t* hist, int nbins, int need, int* ws,
                                        int* sh_pick, int* above) {
  const int t = threadIdx.x;
  const int b1 = nbins - 1 - 2 * t, b0 = b1 - 1;             // this thread's bins, high first
  const int h1 = b1 >= 0 ? (int)hist[b1] : 0;
  const int h0 = b0 >= 0 ? (int)hist[b0] : 0;
  int total;
  const int before = block_exclusive_scan(h1 + h0, ws, total);   // entries in higher bins
  if (before < need && before + h1 >= need) {
    sh_pick[0] = b1;
    sh_pick[1] = before;
  } else if (before + h1 < need && before + h1 + h0 >= need) {
    sh_pick[0] = b0;
    sh_pick[1] = before + h1;
  }
  __syncthreads();
  *above = sh_pick[1];
  const int bin = sh_pick[0];
  __syncthreads();
  return bin;
}

__global__ void __launch_bounds__(kTkThreads)
    topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) float row_s[];             // the row, when it fits
  __shared__ uint32_t hist[2048];
  __shared__ int ws[kTkWarps];
  __shared__ int sh_pick[2];
  __shared__ float red[2][kTkWarps];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the logits were written by the previous launch
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  const int Lraw = __ldg(p.seqlens + r);
  const bool bad = Lraw > p.T;
  const int L = bad ? 0 : max(Lraw, 0);
  const float* grow = p.logits + (long long)r * p.ld;
  int* orow = p.idx + (long long)r * p.out_stride;
  float* vrow = p.vals ? p.vals + (long long)r * p.out_stride : nullptr;
  if (bad && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
  if (L <= p.k) {
    for (int j = tid; j < p.k; j += kTkThreads) {
      orow[j] = j < L ? j : -1;
      if (vrow) vrow[j] = j < L ? grow[j] : -INFINITY;
    }
    return;
  }

  // ---- the row into shared memory (if it fits), with its range (NaN, an
  // error row's logit, is left out of the range)
  const bool cached = L <= p.cache_floats;
  const int L4 = L / 4;
  float mn = INFINITY, mx = -INFINITY;
  {
    const float4* gr4 = reinterpret_cast<const float4*>(grow);    // rows are 256-byte aligned
    for (int i4 = tid; i4 < L4; i4 += 4 * kTkThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = i4 + u * kTkThreads;
        v[u] = j < L4 ? __ldcg(gr4 + j) : make_float4(NAN, NAN, NAN, NAN);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = i4 + u * kTkThreads;
        if (cached && j < L4) reinterpret_cast<float4*>(row_s)[j] = v[u];
        mn = fminf(mn, fminf(fminf(v[u].x, v[u].y), fminf(v[u].z, v[u].w)));
        mx = fmaxf(mx, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
      }
    }
    for (int i = 4 * L4 + tid; i < L; i += kTkThreads) {
      const float x = grow[i];
      if (cached) row_s[i] = x;
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    red[0][warp] = mn;
    red[1][warp] = mx;
  }
  __syncthreads();
  mn = INFINITY;
  mx = -INFINITY;
#pragma unroll
  for (int w8 = 0; w8 < kTkWarps; ++w8) {
    mn = fminf(mn, red[0][w8]);
    mx = fmaxf(mx, red[1][w8]);
  }
  const float* row = cached ? row_s : grow;             // scalar reads: generic loads
  const float4* s4 = reinterpret_cast<const float4*>(row_s);
  const float4* g4 = reinterpret_cast<const float4*>(grow);
  auto ld4 = [&](int j) -> float4 { return cached ? s4[j] : __ldcg(g4 + j); };

  // ---- the k-th largest key.  Logits crowd into a few sign/exponent
  // values, so a first radix digit would pile the histogram's atomics onto a
  // few bins.  The first pass instead bins linearly between the row's
  // smallest and largest logit (monotone in the logit, so the bin holding the
  // k-th largest, and the count above it, are exact); three radix passes
  // (11 + 11 + 10 bits of the key) then run over that bin's members.  NaN
  // goes to bin 0 with key 0, the smallest.  An infinite or zero range puts
  // everything in bin 0 (still exact).
  const float span = mx - mn;
  const float inv = (span > 0.f && span < INFINITY) ? 2048.f / span : 0.f;
  auto lbin = [&](float x) -> int {
    if (!(x == x)) return 0;
    return min(2047, max(0, (int)((x - mn) * inv)));
  };
  uint32_t prefix = 0, mask = 0;
  int need = p.k;                            // entries still to take at or below the prefix
  int lb = 0;                                // the chosen linear bin
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = pass == 1 ? 21 : pass == 2 ? 10 : 0;
    const int nbins = pass == 3 ? 1024 : 2048;
    for (int b = tid; b < nbins; b += kTkThreads) hist[b] = 0;
    __syncthreads();
    auto count = [&](float x) {
      if (pass == 0) {
        atomicAdd(&hist[lbin(x)], 1u);
        return;
      }
      if (lbin(x) != lb) return;
      const uint32_t key = order_key(x);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
    };
    for (int i4 = tid; i4 < L4; i4 += 4 * kTkThreads) {   // four 16-byte loads in flight
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = i4 + u * kTkThreads;
        v[u] = j < L4 ? ld4(j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (i4 + u * kTkThreads >= L4) continue;
        count(v[u].x);
        count(v[u].y);
        count(v[u].z);
        count(v[u].w);
      }
    }
    for (int i = 4 * L4 + tid; i < L; i += kTkThreads) count(row[i]);   // the last L % 4
    __syncthreads();
    int above;
    const int bin = find_bin(hist, nbins, need, ws, sh_pick, &above);
    if (pass == 0) {
      lb = bin;
    } else {
      prefix |= (uint32_t)bin << shift;
      mask |= (uint32_t)(nbins - 1) << shift;
    }
    need -= above;
  }
  const uint32_t kstar = prefix;             // the k-th largest key; `need` of its copies are taken

  // ---- selection, in position order: every key above K*, the first `need`
  // equal to it.  Thread t scans a contiguous chunk of positions.
  const int chunk = ((L + kTkThreads - 1) / kTkThreads + 3) & ~3;    // whole float4s
  const int c0 = min(L, tid * chunk), c1 = min(L, c0 + chunk);
  int n_gt = 0, n_eq = 0;
  for (int i = c0; i < c1; i += 16) {       // four 16-byte loads in flight
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = i + 4 * u + 3 < c1 ? ld4((i >> 2) + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = i + 4 * u + e;
        if (pos >= c1) continue;
        const uint32_t key = order_key(i + 4 * u + 3 < c1 ? x[e] : row[pos]);
        n_gt += key > kstar;
        n_eq += key == kstar;
      }
    }
  }
  int tot;
  const int eq_before = block_exclusive_scan(n_eq, ws, tot);
  const int eq_take = max(0, min(n_eq, need - eq_before));
  const int out0 = block_exclusive_scan(n_gt + eq_take, ws, tot);
  const int o_end = out0 + n_gt + eq_take;
  int o = out0, eq_seen = 0;
  for (int i = c0; i < c1 && o < o_end; i += 16) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = i + 4 * u + 3 < c1 ? ld4((i >> 2) + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = i + 4 * u + e;
        if (pos >= c1) continue;
        const float val = i + 4 * u + 3 < c1 ? x[e] : row[pos];
        const uint32_t key = order_key(val);
        bool take = key > kstar;
        if (key == kstar) take = eq_seen++ < eq_take;
        if (take) {
          orow[o] = pos;
          if (vrow) vrow[o] = val;
          ++o;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, long long ld, const int* seqlens, int rows, int T,
                        int k, int* idx, float* vals, long long out_stride, int* status,
                        cudaStream_t stream) {
  // shared memory for the row cache: the per-block opt-in less the static
  // arrays, set once per device
  static int cache_per_dev[kMaxDevices] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (cache_per_dev[dev] == 0) {
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    const int bytes = ((optin - 16 * 1024) / 16) * 16;      // leave room for the static arrays
    if ((e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  bytes)) != cudaSuccess)
      return e;
    cache_per_dev[dev] = bytes;
  }
  const int bytes = cache_per_dev[dev];
  const TopkParams p{logits, ld, seqlens, rows, T, k, idx, vals, out_stride, status, bytes / 4};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace dsa
