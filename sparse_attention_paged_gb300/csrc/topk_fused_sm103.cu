// topk_fused_sm103.cu -- the merge step of the fused decode + top-k call:
// per request, the k best positions among the candidates that the decode
// kernel's CTAs left in the request's slots (topk_slots.cuh), written in
// position order with their logits.
//
// The top-k is the logits' consumer: "The Dispatch Decision: Wiring a
// Triton Kernel into Production", section "The Problem That Led Here" (the
// indexer scores the cached positions so that only the best enter sparse
// attention).  The order is the selection's plain definition: larger logit
// first, lower position first among equal logits.
//
// One CTA of 256 threads per request.  The slots of a request list its
// candidates in position order, so "lower position first" is "earlier in
// slot order".  The k-th best key comes from radix selection (8 bits a pass,
// a 256-bin shared histogram, four passes over the candidates, read from
// L2); each thread then owns a contiguous run of the flattened slot space,
// and two block scans give every taken candidate its place in the output.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"
#include "topk_slots.cuh"

namespace dsa {

namespace {

constexpr int kMgThreads = 512;
constexpr int kMgWarps = kMgThreads / 32;
constexpr int kMgMaxSlots = 2048;             // slot offsets kept in shared memory
constexpr int kMgCap = 24 * 1024;             // candidates staged in shared memory
constexpr int kMgSmem = kMgCap * 8;           // their logits and positions: 192 KB

struct MergeParams {
  const float* ws;       // the fused top-k workspace
  const int* seqlens;
  int rows;
  int T;                 // W * 64
  int k;
  int* idx;              // row r at idx + r * out_stride
  float* vals;           // nullable
  long long out_stride;
  int* status;
};

__device__ __forceinline__ int mg_scan(int v, int* scr, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scr[w] = x;
  __syncthreads();
  int base = 0, sum = 0;
#pragma unroll
  for (int j = 0; j < kMgWarps; ++j) {
    const int c = scr[j];
    if (j < w) base += c;
    sum += c;
  }
  __syncthreads();
  *total = sum;
  return base + x - v;
}

// The k best of the candidates i in [0, n) with ok(i), in position order,
// their logits and positions read through val(i) / pos(i); m of them are
// ok.  Written in that order to oidx / oval and padded with -1 / -inf to k.
// Radix selection over 256-bin histograms (one atomic per distinct digit per
// warp), then an ordered compaction: warp w over a contiguous 1/16 of the
// candidates, its lanes on consecutive ones, offsets from warp votes.
template <class Ok, class Val, class Pos>
__device__ void merge_select(int n, int m, int k, Ok ok, Val val, Pos pos, int* oidx,
                             float* oval, int* hist, int* scr) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bool all = m <= k;
  uint32_t prefix = 0, mask = 0;
  int need = min(k, m);                      // still to take among keys matching prefix
  if (!all) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int base = 0; base < n; base += kMgThreads) {
        const int i = base + tid;
        const bool in = i < n && ok(i);
        const uint32_t key = in ? sel_key(val(i)) : 0u;
        const bool mt = in && (key & mask) == prefix;
        const unsigned act = __ballot_sync(0xffffffffu, mt);
        if (mt) {
          const uint32_t d = (key >> shift) & 255u;
          const unsigned peers = __match_any_sync(act, d);
          if (lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
        }
      }
      __syncthreads();
      const int d = 255 - tid;               // one digit per thread (the first 256), high first
      const int h = tid < 256 ? hist[d] : 0;
      int tot;
      const int before = mg_scan(h, scr, &tot);
      if (tid < 256 && before < need && before + h >= need) {
        scr[kMgWarps] = d;
        scr[kMgWarps + 1] = before;
      }
      __syncthreads();
      need -= scr[kMgWarps + 1];
      prefix |= (uint32_t)scr[kMgWarps] << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
  }
  // warp w compacts [b0, b1) in order
  const int per = ((n + kMgWarps - 1) / kMgWarps + 31) & ~31;
  const int b0 = min(w * per, n), b1 = min(b0 + per, n);
  const unsigned lt = (1u << lane) - 1u;
  int gt_w = 0, eq_w = 0;
  for (int i0 = b0; i0 < b1; i0 += 32) {
    const int i = i0 + lane;
    const bool in = i < b1 && ok(i);
    const uint32_t key = in ? sel_key(val(i)) : 0u;
    gt_w += __popc(__ballot_sync(0xffffffffu, in && (all || key > prefix)));
    eq_w += __popc(__ballot_sync(0xffffffffu, in && !all && key == prefix));
  }
  if (lane == 0) {
    scr[kMgWarps + 2 + w] = gt_w;
    scr[2 * kMgWarps + 2 + w] = eq_w;
  }
  __syncthreads();
  int o = 0, e = 0, taken = 0;
  for (int v = 0, ee = 0; v < kMgWarps; ++v) {
    const int eqv = scr[2 * kMgWarps + 2 + v];
    const int tv = scr[kMgWarps + 2 + v] + min(max(need - ee, 0), eqv);
    if (v < w) {
      o += tv;
      e += eqv;
    }
    taken += tv;
    ee += eqv;
  }
  for (int i0 = b0; i0 < b1; i0 += 32) {
    const int i = i0 + lane;
    const bool in = i < b1 && ok(i);
    const float v = in ? val(i) : 0.f;
    const uint32_t key = sel_key(v);
    const bool g = in && (all || key > prefix), q = in && !all && key == prefix;
    const unsigned qb = __ballot_sync(0xffffffffu, q);
    const bool take = g || (q && e + __popc(qb & lt) < need);
    const unsigned tb = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int dst = o + __popc(tb & lt);
      oidx[dst] = pos(i);
      if (oval) oval[dst] = v;
    }
    o += __popc(tb);
    e += __popc(qb);
  }
  for (int j = taken + tid; j < k; j += kMgThreads) {
    oidx[j] = -1;
    if (oval) oval[j] = -INFINITY;
  }
}

__global__ void __launch_bounds__(kMgThreads) topk_merge_kernel(const MergeParams p) {
  extern __shared__ uint8_t mg_smem[];
  __shared__ int hist[256];
  __shared__ int scr[3 * kMgWarps + 2];
  __shared__ int slot_off[kMgMaxSlots + 1];
  float* s_val = reinterpret_cast<float*>(mg_smem);
  int* s_pos = reinterpret_cast<int*>(mg_smem + kMgCap * 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  sm100::griddep_wait();
  const int k = p.k;
  int* oidx = p.idx + (long long)r * p.out_stride;
  float* oval = p.vals ? p.vals + (long long)r * p.out_stride : nullptr;
  const int L = __ldg(p.seqlens + r);
  if (L > p.T) {                             // an over-long row selects nothing
    for (int j = tid; j < k; j += kMgThreads) {
      oidx[j] = -1;
      if (oval) oval[j] = -INFINITY;
    }
    if (tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
    return;
  }
  const int* hdr = reinterpret_cast<const int*>(p.ws);
  const int s0 = L > 0 ? __ldg(hdr + r) : 0, s1 = L > 0 ? __ldg(hdr + r + 1) : 0;
  const int ns = s1 - s0;
  const long long sf = sel_slot_floats(k);
  const float* slots = p.ws + sel_header_floats(p.rows) + (long long)s0 * sf;
  auto count_of = [&](int s) { return __ldg(reinterpret_cast<const int*>(slots + s * sf)); };

  if (ns <= kMgMaxSlots) {
    // slot offsets in slot order: thread t sums slots [t*sp, (t+1)*sp)
    const int sp = (ns + kMgThreads - 1) / kMgThreads;
    const int a = min(tid * sp, ns), b = min(a + sp, ns);
    int mine = 0;
    for (int s = a; s < b; ++s) mine += count_of(s);
    int n;
    int off = mg_scan(mine, scr, &n);
    for (int s = a; s < b; ++s) {
      slot_off[s] = off;
      off += count_of(s);
    }
    if (tid == 0) slot_off[ns] = n;
    __syncthreads();
    if (n <= kMgCap) {
      // stage: a warp per slot, its lanes over the candidates (coalesced)
      for (int s = warp; s < ns; s += kMgWarps) {
        const int c = slot_off[s + 1] - slot_off[s], o = slot_off[s];
        const float* sv = slots + s * sf + kSlotHead;
        const int* spos = reinterpret_cast<const int*>(sv + k);
        for (int j = lane; j < c; j += 32) {
          s_val[o + j] = __ldg(sv + j);
          s_pos[o + j] = __ldg(spos + j);
        }
      }
      __syncthreads();
      // the next launch may start once the candidates are staged (its CTAs
      // would otherwise take SM slots this grid's CTAs still wait for)
      sm100::griddep_launch_dependents();
      merge_select(n, n, k, [](int) { return true; }, [&](int i) { return s_val[i]; },
                   [&](int i) { return s_pos[i]; }, oidx, oval, hist, scr);
      return;
    }
  }
  // rows with more candidates than shared memory holds: read them in place,
  // candidate j of slot s at flat index s * k + j, j below the slot's count
  __syncthreads();
  int m = 0;
  for (int s = tid; s < ns; s += kMgThreads) m += count_of(s);
  int n;
  mg_scan(m, scr, &n);
  sm100::griddep_launch_dependents();
  merge_select(
      ns * k, n, k, [&](int f) { return f % k < count_of(f / k); },
      [&](int f) { return __ldg(slots + (f / k) * sf + kSlotHead + f % k); },
      [&](int f) {
        return __ldg(reinterpret_cast<const int*>(slots + (f / k) * sf + kSlotHead + k) + f % k);
      },
      oidx, oval, hist, scr);
}

}  // namespace

cudaError_t launch_topk_merge(const float* ws, const int* seqlens, int rows, int T, int k,
                              int* idx, float* vals, long long out_stride, int* status,
                              cudaStream_t stream) {
  static bool configured[kMaxDevices] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMgSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  MergeParams mp{ws, seqlens, rows, T, k, idx, vals, out_stride, status};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(kMgThreads);
  cfg.dynamicSmemBytes = kMgSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_merge_kernel, mp);
}

}  // namespace dsa
