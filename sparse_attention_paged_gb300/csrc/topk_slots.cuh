// topk_slots.cuh -- the candidate slots of the fused decode + top-k call.
//
// In the fused form the decode kernel keeps no logits in global memory.  A
// persistent CTA of the balanced decode owns a contiguous slice of the
// call's valid (row, page) units; its pages of one row form a segment, cut
// into chunks of at most kSelChunkPages pages counted from the segment's
// first page (a two-page tile never straddles two chunks).  When a chunk is
// complete the CTA writes the chunk's best min(k, n) positions (largest
// logit first, lower position first among equal logits) with their logits
// into a slot of the caller's workspace.  Every chunk has its own slot, so
// the slots of a row, in slot order, list the row's candidates in position
// order; the merge kernel then selects the row's k best among them.  Taking
// each chunk's k best loses nothing: a position that k others of its own
// chunk beat cannot be among the row's k best.
//
// Workspace layout (floats): [row slot offsets S, B + 1 ints, padded to a
// multiple of 4][slots].  Row r's slots are S[r] .. S[r+1]-1.  A slot is
// kSlotHead + 2 * k floats: the count n (an int) at 0, the n logits at
// kSlotHead, the n positions (ints) at kSlotHead + k.
#pragma once

#include "dsa_common.cuh"

namespace dsa {

constexpr int kSelChunkPages = 32;                 // pages per chunk
constexpr int kSelChunk = kSelChunkPages * kPage;  // 2,048 positions
constexpr int kSelMaxK = kSelChunk;                // the fused form's largest k (a chunk)
constexpr int kSlotHead = 4;                       // floats before a slot's logits

__host__ __device__ __forceinline__ long long sel_slot_floats(int k) {
  return kSlotHead + 2ll * k;
}

__host__ __device__ __forceinline__ long long sel_header_floats(int rows) {
  return ((long long)rows + 1 + 3) & ~3ll;
}

// The balanced decode's slicing: CTA c of R owns units [c*N/R, (c+1)*N/R),
// computed as c*q + (c*r)/R with N = q*R + r (32-bit arithmetic: c*q <= N
// and c*r < R*R).
struct Slicer {
  int N, R, q, r;
  __device__ __forceinline__ Slicer(int N_, int R_) : N(N_), R(R_), q(N_ / R_), r(N_ % R_) {}
  __device__ __forceinline__ int begin(int c) const { return c * q + (c * r) / R; }
  // the CTA whose slice holds unit u (0 <= u < N): the largest c with
  // begin(c) <= u
  __device__ __forceinline__ int cta_of(int u) const {
    int c = (int)(((long long)(u + 1) * R - 1) / N);
    c = min(max(c, 0), R - 1);
    while (c > 0 && begin(c) > u) --c;
    while (c + 1 < R && begin(c + 1) <= u) ++c;
    return c;
  }
  // chunks of the row of units [v0, v1) that CTA c holds
  __device__ __forceinline__ int chunks_of(int c, int v0, int v1) const {
    const int a = max(begin(c), v0), b = min(begin(c + 1), v1);
    return b > a ? (b - a + kSelChunkPages - 1) / kSelChunkPages : 0;
  }
  // chunks of the row of units [v0, v1) held by its CTAs before CTA c_stop
  // (all of them for c_stop >= R)
  __device__ __forceinline__ int row_chunks(int v0, int v1, int c_stop) const {
    if (v1 <= v0) return 0;
    const int c0 = cta_of(v0), c1 = cta_of(v1 - 1);
    int n = 0;
    for (int c = c0; c <= c1 && c < c_stop; ++c) n += chunks_of(c, v0, v1);
    return n;
  }
};

// Order-preserving 32-bit key of a logit: a larger logit gives a larger
// key; NaN (an error position) the smallest.
__device__ __forceinline__ uint32_t sel_key(float v) {
  const uint32_t u = __float_as_uint(v);
  if (v != v) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dsa
