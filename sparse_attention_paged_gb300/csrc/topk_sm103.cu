// topk_sm103.cu -- top-k selection over each row's logits: the positions
// with the k largest logits, which sparse attention then reads.  The pages
// name the consumer ("The Dispatch Decision: Wiring a Triton Kernel into
// Production", section "The Problem That Led Here": the indexer scores the
// cached positions so that only the top-k enter attention); the selection
// itself is a plain definition.
//
// One CTA per row, or a cluster of two that splits the row in halves while
// two CTAs per row fit in one wave.  Logits become order-preserving 32-bit
// keys (a larger float gives a larger key; NaN, which only an error row
// holds, the smallest key).  A histogram of 2,048 linear bins over a sampled
// range finds the bin of the k-th largest logit (any monotone binning keeps
// the counts exact); one more pass collects that bin's members into shared
// memory (usually a handful) and records the positions in higher bins as
// warp-vote masks.  The collected keys are ranked directly to find the k-th
// largest key K* and how many keys equal to it are needed (lowest positions
// first); those taken join the masks, from which the last pass writes the
// positions in order.  A bin with many members, or a very long row, takes
// the general path instead: three radix passes (11 + 11 + 10 bits) over the
// collected keys or the whole row, per-warp counts, and a write that
// compares every key.  Each warp owns a contiguous segment, its lanes on
// consecutive float4s, so that shared-memory reads are free of bank
// conflicts and in-order output offsets come from warp votes.  Rows of at
// most k valid positions take all of them; the rest of the k outputs is -1
// (value -inf).
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {

namespace cg = cooperative_groups;

namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
static_assert(kTkWarps == 32, "the per-warp scans run on one warp's lanes");
constexpr int kCand = 2048;                  // keys of the k-th largest's bin kept for the exact passes
constexpr int kRankMax = 128;                // at most this many collected keys: ranked directly
constexpr int kMaskSteps = 16;               // steps of 32 float4s per warp kept as vote masks
static_assert(kTkWarps * kMaskSteps * 4 == 2048, "one mask word per warp, step and element");
static_assert(2 * kRankMax <= kCand / 2, "a pair's collected keys fit in half of the buffer");
constexpr int kStaticSmemReserve = 36 * 1024;  // the kernel's static shared arrays fit in this

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
  int cache_floats;      // a CTA's part of a row up to this length is kept in shared memory
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
// writes the count above it to *above and its own count to *pop.  hist2,
// when given, is added bin by bin (the other half of a row).
__device__ __forceinline__ int find_bin(const uint32_t* hist, const uint32_t* hist2, int nbins,
                                        int need, int* ws, int* sh_pick, int* above, int* pop) {
  const int t = threadIdx.x;
  const int b1 = nbins - 1 - 2 * t, b0 = b1 - 1;             // this thread's bins, high first
  int h1 = b1 >= 0 ? (int)hist[b1] : 0;
  int h0 = b0 >= 0 ? (int)hist[b0] : 0;
  if (hist2 != nullptr) {
    h1 += b1 >= 0 ? (int)hist2[b1] : 0;
    h0 += b0 >= 0 ? (int)hist2[b0] : 0;
  }
  int total;
  const int before = block_exclusive_scan(h1 + h0, ws, total);   // entries in higher bins
  if (before < need && before + h1 >= need) {
    sh_pick[0] = b1;
    sh_pick[1] = before;
    sh_pick[2] = h1;
  } else if (before + h1 < need && before + h1 + h0 >= need) {
    sh_pick[0] = b0;
    sh_pick[1] = before + h1;
    sh_pick[2] = h0;
  }
  __syncthreads();
  *above = sh_pick[1];
  *pop = sh_pick[2];
  const int bin = sh_pick[0];
  __syncthreads();
  return bin;
}

// Warp prefix of a per-lane count in 0..7: the lanes below this one, and
// the warp's total.
__device__ __forceinline__ int warp_prefix(int c, int lane, int& total) {
  const uint32_t b0 = __ballot_sync(0xffffffffu, c & 1);
  const uint32_t b1 = __ballot_sync(0xffffffffu, c & 2);
  const uint32_t b2 = __ballot_sync(0xffffffffu, c & 4);
  const uint32_t lt = (1u << lane) - 1u;
  total = __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
  return __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// kCl CTAs per row (1, or a cluster of 2 that splits the row in halves:
// each reads the other's histogram and receives its collected keys and
// counts through distributed shared memory).
template <int kCl>
__global__ void __launch_bounds__(kTkThreads)
    topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) float row_s[];             // the CTA's part of the row, when it fits
  __shared__ __align__(16) uint32_t hist[2048];
  __shared__ uint32_t cand_key[kCand];
  __shared__ int cand_pos[kCand];
  __shared__ int ws[kTkWarps];
  __shared__ int sh_pick[3];
  __shared__ float red[2][kTkWarps];
  __shared__ int w_gt[kTkWarps], w_eq[kTkWarps], w_out[kTkWarps], w_take[kTkWarps];
  __shared__ int n_cand;
  __shared__ __align__(16) uint32_t tmask[2048];               // vote masks of the positions taken
  // a pair's exchange: the other CTA's collected count and count of
  // positions in bins above lb (written by it), this CTA's count, and the
  // collected positions of the first half that are taken
  __shared__ int peer_n, peer_def, own_def, taken_first;
  const int r = blockIdx.x / kCl, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int crank = kCl > 1 ? (int)cg::this_cluster().block_rank() : 0;
  // the logits were written by the previous launch
  sm100::griddep_wait();
  const int Lraw = __ldg(p.seqlens + r);
  const bool bad = Lraw > p.T;
  const int L = bad ? 0 : max(Lraw, 0);
  const float* grow = p.logits + (long long)r * p.ld;
  int* orow = p.idx + (long long)r * p.out_stride;
  float* vrow = p.vals ? p.vals + (long long)r * p.out_stride : nullptr;
  if (bad && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
  if (L <= p.k) {                            // the whole cluster takes this branch
    if (crank == 0) {
      for (int j = tid; j < p.k; j += kTkThreads) {
        orow[j] = j < L ? j : -1;
        if (vrow) vrow[j] = j < L ? grow[j] : -INFINITY;
      }
    }
    return;
  }

  // The CTA owns float4s [cb4, cb4 + cn4) of the row (its part) and warp w
  // of it float4s [w_beg, w_end); the last float4 may run past L (still
  // inside the row's T >= L floats, or the shared cache, both multiples of
  // 4), and its positions >= L are masked everywhere.  Segments are sized
  // from the largest part, so every CTA of a cluster has the same steps.
  const int n4 = (L + 3) >> 2;
  const int p4 = (n4 + kCl - 1) / kCl;
  int cb4 = min(n4, crank * p4), cn4 = min(n4, cb4 + p4) - cb4;
  int seg4 = (p4 + kTkWarps - 1) / kTkWarps;
  int w_beg = cb4 + min(cn4, warp * seg4), w_end = cb4 + min(cn4, warp * seg4 + seg4);
  bool cached = 4 * cn4 <= p.cache_floats;
  float4* s4 = reinterpret_cast<float4*>(row_s);
  const float4* g4 = reinterpret_cast<const float4*>(grow);    // rows are 256-byte aligned
  auto ld4 = [&](int j) -> float4 { return cached ? s4[j - cb4] : __ldcg(g4 + j); };
  // valid positions in float4 j (0 past the warp's segment)
  auto nvalid = [&](int j) { return j < w_end ? min(4, L - 4 * j) : 0; };
  // every float4 of the warp's segment, four 16-byte loads in flight; fn runs
  // on all lanes of a step (nvalid 0 on the idle ones) so that it may use
  // warp votes; steps wholly past the segment are skipped
  auto visit = [&](auto&& fn) {
    for (int j0 = w_beg; j0 < w_end; j0 += 4 * 32) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * 32 + lane;
        v[u] = j < w_end ? ld4(j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j0 + u * 32 < w_end) fn(j0 + u * 32 + lane, v[u]);   // warp-uniform
    }
  };

  // ---- the bins: 2,048 linear bins over the range of a sample (every
  // lane's first float4), widened by an eighth of its span on each side.
  // Logits crowd into a few sign/exponent values, so a first radix digit
  // would pile the histogram's atomics onto a few bins; linear bins do not.
  // Any binning monotone in the logit keeps the counts exact (values past
  // the range land in the end bins), so the bin of the k-th largest and the
  // count above it are exact; the sample only decides how crowded that bin
  // is.  NaN (an error row's logit, left out of the range) goes to bin 0 with
  // key 0, the smallest.  A zero or infinite range puts everything in bin 0
  // (still exact).
  const int j_first = w_beg + lane;
  const float4 v_first = j_first < w_end ? __ldcg(g4 + j_first) : make_float4(0.f, 0.f, 0.f, 0.f);
  float mn = INFINITY, mx = -INFINITY;
  {
    const int nv = nvalid(j_first);
    const float x[4] = {v_first.x, v_first.y, v_first.z, v_first.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e < nv) {
        mn = fminf(mn, x[e]);
        mx = fmaxf(mx, x[e]);
      }
    }
  }
  if constexpr (kCl > 1) {
    // the other half's sample too, read from global memory, so that both
    // CTAs of the pair bin over the same range without an exchange
    const int o_cb4 = min(n4, (1 - crank) * p4), o_cn4 = min(n4, o_cb4 + p4) - o_cb4;
    const int jo = o_cb4 + min(o_cn4, warp * seg4) + lane;
    if (jo < o_cb4 + min(o_cn4, warp * seg4 + seg4)) {
      const float4 v = __ldcg(g4 + jo);
      const float x[4] = {v.x, v.y, v.z, v.w};
      const int nv = min(4, L - 4 * jo);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < nv) {
          mn = fminf(mn, x[e]);
          mx = fmaxf(mx, x[e]);
        }
      }
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
  for (int b = tid; b < 2048; b += kTkThreads) hist[b] = 0;
  if (tid == 0) {
    // (the other CTA of a pair writes peer_n / peer_def only after both
    // have passed the histogram barrier, so these are cleared first)
    n_cand = 0;
    peer_n = 0;
    peer_def = 0;
    own_def = 0;
    taken_first = 0;
  }
  __syncthreads();
  mn = INFINITY;
  mx = -INFINITY;
#pragma unroll
  for (int w8 = 0; w8 < kTkWarps; ++w8) {
    mn = fminf(mn, red[0][w8]);
    mx = fmaxf(mx, red[1][w8]);
  }
  float span = mx - mn, lo = mn;
  if (span > 0.f && span < INFINITY) {
    lo = mn - 0.125f * span;
    span *= 1.25f;
  }
  const float inv = (span > 0.f && span < INFINITY) ? 2048.f / span : 0.f;
  auto lbin = [&](float x) -> int {
    if (!(x == x)) return 0;
    return min(2047, max(0, (int)((x - lo) * inv)));
  };

  // ---- one pass over the row: into shared memory (if it fits), the
  // histogram, and each position's bin (16 bits, when the row and its bins
  // fit)
  bool bins_cached = 6 * cn4 <= p.cache_floats;
  uint2* b2 = reinterpret_cast<uint2*>(row_s + 4 * cn4);      // four bins per float4
  auto bin_float4 = [&](int j, float4 v) {
    const int nv = nvalid(j);
    if (nv == 0) return;
    if (cached) s4[j - cb4] = v;
    const float x[4] = {v.x, v.y, v.z, v.w};
    uint32_t bq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      bq[e] = (uint32_t)lbin(x[e]);
      if (e < nv) atomicAdd(&hist[bq[e]], 1u);
    }
    if (bins_cached) b2[j - cb4] = make_uint2(bq[0] | (bq[1] << 16), bq[2] | (bq[3] << 16));
  };
  bin_float4(j_first, v_first);
  for (int j0 = w_beg + 32; j0 < w_end; j0 += 8 * 32) {      // eight 16-byte loads in flight
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * 32 + lane;
      v[u] = j < w_end ? __ldcg(g4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) bin_float4(j0 + u * 32 + lane, v[u]);
  }
  __syncthreads();
  int need = p.k;                            // entries still to take at or below the prefix
  int above, pop;
  const uint32_t* hist_peer = nullptr;
  if constexpr (kCl > 1) {                   // both halves' histograms complete
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    hist_peer = cluster.map_shared_rank(hist, 1 - crank);
  }
  const int lb = find_bin(hist, hist_peer, 2048, need, ws, sh_pick, &above, &pop);
  need -= above;

  // ---- the k-th largest key K* among the members of bin lb: the collected
  // keys, or the whole row by radix passes when the bin holds more than
  // kCand of them.
  //
  // The usual case ("fast": at most kRankMax members and a segment of at
  // most kMaskSteps steps) ranks the collected keys directly and records
  // the positions taken as warp-vote masks, one word per (warp, step,
  // element of the float4): positions in bins above lb while the row is
  // collected, then the collected ones that make the cut.
  const bool collect = pop <= kCand;
  const int S = (seg4 + 31) >> 5;            // steps of 32 float4s in a warp's segment
  const bool fast = pop <= kRankMax && S <= kMaskSteps;
  if (kCl > 1 && !fast) {
    // the general path runs on the cluster's first CTA alone, over the
    // whole row, read from global memory (its histogram is reused once the
    // other CTA has read it)
    if constexpr (kCl > 1) cg::this_cluster().sync();
    if (crank != 0) return;
    cb4 = 0;
    cn4 = n4;
    seg4 = (n4 + kTkWarps - 1) / kTkWarps;
    w_beg = min(n4, warp * seg4);
    w_end = min(n4, w_beg + seg4);
    cached = false;
    bins_cached = false;
  }
  auto mask_word = [&](int w, int step, int e) -> uint32_t& {
    return tmask[(w * kMaskSteps + step) * 4 + e];
  };
  if (fast) {                                // each warp clears its own words
    for (int i = lane; i < kMaskSteps * 4; i += 32) tmask[warp * kMaskSteps * 4 + i] = 0u;
    __syncwarp();
  }
  int n_gt_bins = 0;                         // this lane's positions in bins above lb
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t* peer_key = nullptr;              // a pair on the fast path: the other CTA's buffers
  int* peer_pos = nullptr;
  if constexpr (kCl > 1) {
    if (fast) {
      peer_key = cg::this_cluster().map_shared_rank(cand_key, 1 - crank);
      peer_pos = cg::this_cluster().map_shared_rank(cand_pos, 1 - crank);
    }
  }
  // one step of the collection: b[e] is the bin of position 4j+e (-1 past
  // the segment); x_of() gives the float4, read only by lanes holding a
  // member of bin lb
  auto collect_step = [&](int j, const int (&b)[4], auto&& x_of) {
    bool c[4], d[4];
    bool any = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      d[e] = b[e] > lb;
      n_gt_bins += d[e];
      c[e] = b[e] == lb;
      any |= c[e];
    }
    if (fast) {
      const uint32_t m0 = __ballot_sync(0xffffffffu, d[0]);
      const uint32_t m1 = __ballot_sync(0xffffffffu, d[1]);
      const uint32_t m2 = __ballot_sync(0xffffffffu, d[2]);
      const uint32_t m3 = __ballot_sync(0xffffffffu, d[3]);
      if (lane < 4)
        mask_word(warp, (j - lane - w_beg) >> 5, lane) =
            lane == 0 ? m0 : lane == 1 ? m1 : lane == 2 ? m2 : m3;
    }
    if (__ballot_sync(0xffffffffu, any) == 0u) return;     // warp-uniform: the usual case
    const float4 v = any ? x_of() : make_float4(0.f, 0.f, 0.f, 0.f);
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t m = __ballot_sync(0xffffffffu, c[e]);
      if (m) {                                            // warp-uniform
        const int leader = __ffs(m) - 1;
        int base = 0;
        if (lane == leader) base = atomicAdd(&n_cand, __popc(m));
        base = __shfl_sync(0xffffffffu, base, leader);
        const int i = base + __popc(m & lt);
        if (c[e] && i < kCand) {
          cand_key[i] = order_key(x[e]);
          cand_pos[i] = 4 * j + e;
          if (peer_key != nullptr) {                      // a pair: the other CTA's copy
            peer_key[kCand / 2 + i] = cand_key[i];
            peer_pos[kCand / 2 + i] = cand_pos[i];
          }
        }
      }
    }
  };
  if (collect && bins_cached) {
    for (int j0 = w_beg; j0 < w_end; j0 += 4 * 32) {       // four 8-byte loads in flight
      uint2 bb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * 32 + lane;
        bb[u] = j < w_end ? b2[j - cb4] : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (j0 + u * 32 >= w_end) break;                  // warp-uniform: past the segment
        const int j = j0 + u * 32 + lane;
        const int nv = nvalid(j);
        int b[4] = {(int)(bb[u].x & 0xffffu), (int)(bb[u].x >> 16), (int)(bb[u].y & 0xffffu),
                    (int)(bb[u].y >> 16)};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e >= nv) b[e] = -1;
        collect_step(j, b, [&] { return s4[j - cb4]; });
      }
    }
  } else if (collect) {
    visit([&](int j, float4 v) {
      const float x[4] = {v.x, v.y, v.z, v.w};
      const int nv = nvalid(j);
      int b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) b[e] = e < nv ? lbin(x[e]) : -1;
      collect_step(j, b, [&] { return v; });
    });
  }
  int nc = min(pop, kCand);
  auto warp_of = [&](int pos) { return ((pos >> 2) - cb4) / seg4; };
  uint32_t kstar = 0;
  int part_base = 0;                         // outputs of the parts before this CTA's
  if (fast) {
    if constexpr (kCl > 1) {
      // each CTA has pushed its collected keys into the other's buffer (at
      // kCand / 2); now its counts, then the pair's barrier: after it
      // neither CTA touches the other's shared memory
      cg::cluster_group cluster = cg::this_cluster();
      const int g = warp_sum(n_gt_bins);
      if (lane == 0) atomicAdd(&own_def, g);
      __syncthreads();
      if (tid == 0) {
        *cluster.map_shared_rank(&peer_n, 1 - crank) = n_cand;
        *cluster.map_shared_rank(&peer_def, 1 - crank) = own_def;
      }
      cluster.sync();                        // both halves collected and pushed
      const int n_own = n_cand, n_other = peer_n;
      for (int i = tid; i < n_other; i += kTkThreads) {   // the other half's keys after this one's
        cand_key[n_own + i] = cand_key[kCand / 2 + i];
        cand_pos[n_own + i] = cand_pos[kCand / 2 + i];
      }
      if (crank == 1) part_base = peer_def;
      nc = n_own + n_other;
    }
    // thread i ranks collected key i: the keys above it, equal to it, and
    // equal to it at a lower position; every thread holding a copy of the
    // need-th largest writes the same pair
    __syncthreads();                         // the collected keys and the masks are in place
    uint32_t key = 0;
    int pos = 0, eq_lower = 0;
    if (tid < nc) {
      key = cand_key[tid];
      pos = cand_pos[tid];
      int gt = 0, eq = 0;
      for (int i = 0; i < nc; ++i) {
        const uint32_t o = cand_key[i];
        gt += o > key;
        eq += o == key;
        eq_lower += o == key && cand_pos[i] < pos;
      }
      if (gt < need && need <= gt + eq) {
        sh_pick[0] = (int)key;
        sh_pick[1] = gt;
      }
    }
    __syncthreads();
    kstar = (uint32_t)sh_pick[0];
    need -= sh_pick[1];                      // copies of K* taken, lowest positions first
    if (tid < nc && (key > kstar || (key == kstar && eq_lower < need))) {
      const int j = pos >> 2;
      if (j >= cb4 && j < cb4 + cn4) {         // this CTA's part: into its masks
        const int w = warp_of(pos), rel = j - cb4 - w * seg4;
        atomicOr(&mask_word(w, rel >> 5, pos & 3), 1u << (rel & 31));
      } else if (j < cb4) {                    // the first part's: its outputs come first
        atomicAdd(&taken_first, 1);
      }
    }
    __syncthreads();
    if (kCl > 1 && crank == 1) part_base += taken_first;
    int cnt = 0;
    for (int i = lane; i < S * 4; i += 32) cnt += __popc(tmask[warp * kMaskSteps * 4 + i]);
    cnt = warp_sum(cnt);
    if (lane == 0) {
      w_gt[warp] = cnt;
      w_eq[warp] = 0;
    }
  } else {
    // three radix passes (11 + 11 + 10 bits)
    uint32_t prefix = 0, mask = 0;
#pragma unroll 1
    for (int pass = 1; pass < 4; ++pass) {
      const int shift = pass == 1 ? 21 : pass == 2 ? 10 : 0;
      const int nbins = pass == 3 ? 1024 : 2048;
      __syncthreads();                       // the previous pass's hist reads are done
      for (int b = tid; b < nbins; b += kTkThreads) hist[b] = 0;
      __syncthreads();
      if (collect) {
        for (int i = tid; i < nc; i += kTkThreads) {
          const uint32_t key = cand_key[i];
          if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
        }
      } else {
        visit([&](int j, float4 v) {
          const float x[4] = {v.x, v.y, v.z, v.w};
          const int nv = nvalid(j);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (e >= nv || lbin(x[e]) != lb) continue;
            const uint32_t key = order_key(x[e]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
          }
        });
      }
      __syncthreads();
      const int bin = find_bin(hist, nullptr, nbins, need, ws, sh_pick, &above, &pop);
      prefix |= (uint32_t)bin << shift;
      mask |= (uint32_t)(nbins - 1) << shift;
      need -= above;
    }
    kstar = prefix;                          // the k-th largest key; `need` of its copies are taken
    // per warp: positions above K*, and equal to it
    if (collect) {
      const int g = warp_sum(n_gt_bins);
      if (lane == 0) {
        w_gt[warp] = g;
        w_eq[warp] = 0;
      }
      __syncthreads();
      for (int i = tid; i < nc; i += kTkThreads) {
        const uint32_t key = cand_key[i];
        if (key > kstar) atomicAdd(&w_gt[warp_of(cand_pos[i])], 1);
        else if (key == kstar) atomicAdd(&w_eq[warp_of(cand_pos[i])], 1);
      }
    } else {
      int n_gt = 0, n_eq = 0;
      visit([&](int j, float4 v) {
        const float x[4] = {v.x, v.y, v.z, v.w};
        const int nv = nvalid(j);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e >= nv) continue;
          const uint32_t key = order_key(x[e]);
          n_gt += key > kstar;
          n_eq += key == kstar;
        }
      });
      n_gt = warp_sum(n_gt);
      n_eq = warp_sum(n_eq);
      if (lane == 0) {
        w_gt[warp] = n_gt;
        w_eq[warp] = n_eq;
      }
    }
  }
  __syncthreads();
  // warp 0: the copies of K* each warp takes (the first `need` in position
  // order) and each warp's first output slot
  if (warp == 0) {
    const int g = w_gt[lane], q = w_eq[lane];
    int qs = q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, qs, o);
      if (lane >= o) qs += y;
    }
    const int take = max(0, min(q, need - (qs - q)));
    int ts = g + take;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ts, o);
      if (lane >= o) ts += y;
    }
    w_out[lane] = part_base + ts - (g + take);
    w_take[lane] = take;
  }
  __syncthreads();

  // ---- the selection, in position order
  // Only now may the next launch start: its CTAs, started earlier, would
  // take SM slots this grid's CTAs (most of an SM's shared memory each) are
  // still waiting for (measured: 0.5-1.5 us per call with a decode next).
  sm100::griddep_launch_dependents();
  int o = w_out[warp];
  const int o_end = o + w_gt[warp] + w_take[warp];
  const int o_lim = min(o_end, p.k);         // the counts say o_end <= k; never write past k
  if (fast) {
    // from the masks: lane l's positions of a step follow those of lanes < l
    const int steps = (w_end - w_beg + 31) >> 5;
    for (int step = 0; step < steps && o < o_end; ++step) {        // warp-uniform
      const uint4 m4 = *reinterpret_cast<const uint4*>(&mask_word(warp, step, 0));
      const uint32_t M[4] = {m4.x, m4.y, m4.z, m4.w};
      const int tot = __popc(M[0]) + __popc(M[1]) + __popc(M[2]) + __popc(M[3]);
      if (tot == 0) continue;
      if (((M[0] | M[1] | M[2] | M[3]) >> lane) & 1u) {
        const int j = w_beg + step * 32 + lane;
        int oo = o + __popc(M[0] & lt) + __popc(M[1] & lt) + __popc(M[2] & lt) + __popc(M[3] & lt);
        const float4 v = ld4(j);
        const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((M[e] >> lane) & 1u) {
            if (oo < o_lim) {
              orow[oo] = 4 * j + e;
              if (vrow) vrow[oo] = x[e];
            }
            ++oo;
          }
        }
      }
      o += tot;
    }
    return;
  }
  // from the keys: every key above K*, the first w_take[warp] equal to it
  const int eq_take = w_take[warp];
  int eq_seen = 0;
  for (int j0 = w_beg; j0 < w_end && o < o_end; j0 += 4 * 32) {   // warp-uniform
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * 32 + lane;
      v[u] = j < w_end ? ld4(j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (j0 + u * 32 >= w_end) break;       // warp-uniform: past the segment
      const int j = j0 + u * 32 + lane;
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      bool gt[4], eq[4];
      int c_eq = 0;
      const int nv = nvalid(j);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = order_key(x[e]);
        gt[e] = e < nv && key > kstar;
        eq[e] = e < nv && key == kstar;
        c_eq += eq[e];
      }
      int tot_eq = 0, rank = eq_seen;
      if (__ballot_sync(0xffffffffu, c_eq != 0) != 0u)        // warp-uniform: a tie in this step
        rank += warp_prefix(c_eq, lane, tot_eq);
      bool take[4];
      int c_take = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        take[e] = gt[e] || (eq[e] && rank < eq_take);
        rank += eq[e];
        c_take += take[e];
      }
      int tot_take;
      int oo = o + warp_prefix(c_take, lane, tot_take);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (take[e]) {
          if (oo < o_lim) {
            orow[oo] = 4 * j + e;
            if (vrow) vrow[oo] = x[e];
          }
          ++oo;
        }
      }
      eq_seen += tot_eq;
      o += tot_take;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, long long ld, const int* seqlens, int rows, int T,
                        int k, int* idx, float* vals, long long out_stride, int* status,
                        cudaStream_t stream) {
  // shared memory for the row cache: the per-block opt-in less the static
  // arrays; and the SM count.  Set once per device.
  static int cache_per_dev[kMaxDevices] = {0};
  static int sms_per_dev[kMaxDevices] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (cache_per_dev[dev] == 0) {
    int optin = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const int bytes = ((optin - kStaticSmemReserve) / 16) * 16;   // room for the static arrays
    if ((e = cudaFuncSetAttribute(topk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  bytes)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  bytes)) != cudaSuccess)
      return e;
    sms_per_dev[dev] = sms;
    cache_per_dev[dev] = bytes;
  }
  const int bytes = cache_per_dev[dev];
  const TopkParams p{logits, ld, seqlens, rows, T, k, idx, vals, out_stride, status, bytes / 4};
  // two CTAs per row (one cluster each) while they all fit in one wave of
  // one CTA per SM; else one CTA per row
  const bool pairs = 2ll * rows <= sms_per_dev[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pairs ? 2 * rows : rows);
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = pairs ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pairs ? 2 : 1;
  return pairs ? cudaLaunchKernelEx(&cfg, topk_kernel<2>, p)
               : cudaLaunchKernelEx(&cfg, topk_kernel<1>, p);
}

}  // namespace dsa
