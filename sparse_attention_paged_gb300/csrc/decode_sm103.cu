// decode_sm103.cu -- decode kernel of the DSA indexer paged MQA-logits for
// GB300 (sm_103a): TMA page gathers through the block table, tcgen05 MMA with
// the accumulator in TMEM, and a fused ReLU / head-weight / scale epilogue.
//
// The grid is fixed by the launch shape (B, W) alone, never by the lengths,
// so a launch can be captured in a CUDA graph and replayed with new lengths
// and tables ("The Moment the Context-Length Tax Vanished: Committing the
// O(actual) Triton Indexer", section "The Commit: Engineering as
// Narrative").  Only pages below each row's length are read, so the work is
// O(actual length); the fixed-shape output past the length is -inf.  Two ways
// of handing out the valid pages, chosen from (B, W):
//
//  * per-request (W <= 64, or many rows): grid (G, B); CTA (c, b) owns pages
//    c, c+G, c+2G, ... of request b.  With G = W this is one CTA per
//    (request, page) ("The Dispatch Wire: Connecting a Triton Indexer Kernel
//    to Production Inference", section "The Reasoning and Decision-Making");
//    a CTA whose first page lies past the request's length only writes -inf
//    and exits.  G is capped so that the few pages of a short table are
//    pipelined by one CTA instead of each paying a CTA's start-up latency.
//  * balanced (long tables): one persistent CTA per resident slot; the valid
//    (request, page) pairs of all rows, in row order, are split into
//    contiguous slices of equal cost (prefix sums of the rows' valid page
//    counts, computed by every CTA; with fp8 keys a row start costs a few
//    pages more, as the CTA splits that row's query itself), and the
//    positions past each length are split evenly.  No CTA is the tail of a
//    long request.  A slice can cross rows; the query operand is
//    double-buffered per row segment.
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
// split once per row segment into two e4m3 terms with a power-of-two scale
// per head: q * 2^e_h = hi + lo * 2^-5, hi = e4m3(q * 2^e_h), lo = e4m3((q *
// 2^e_h - hi) * 2^5), with 2^e_h folded into the head weight.  The two terms
// accumulate in TMEM apart (the lo term's 2^-5 is applied in the epilogue),
// so hi + lo * 2^-5 reproduces every bf16 value whose magnitude is at least
// 2^-14 of its head's maximum exactly, and the rest to within 2^-22 of it.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"
#include "tensor_maps.cuh"
#include "topk_slots.cuh"

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
#define DSA_DEC_FP8_STAGES 4
#endif
#ifndef DSA_DEC_BF16_STAGES
#define DSA_DEC_BF16_STAGES 2
#endif
#ifndef DSA_DEC_CTAS
#define DSA_DEC_CTAS 2
#endif
constexpr int kDecThreads = 192;          // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kCtasPerSm = DSA_DEC_CTAS;
#ifndef DSA_WAIT_LIMIT_CYCLES
#define DSA_WAIT_LIMIT_CYCLES 2000000000ll
#endif
constexpr long long kWaitLimit = DSA_WAIT_LIMIT_CYCLES;   // ~1 s of SM clock: bound on any wait
constexpr int kMaxRowsBalanced = 384;     // balanced mode keeps per-row prefix sums in smem

template <int KV>
struct DecCfg;

template <>
struct DecCfg<DSA_KV_FP8_E4M3> {
  static constexpr int kStages = DSA_DEC_FP8_STAGES;
  static constexpr int kMaxSlots = DSA_DEC_FP8_SLOTS;     // G cap: CTAs per request
  static constexpr int kPageBytes = kPage * kDim;         // 8 KB of e4m3 rows
  static constexpr int kTileBytes = 2 * kPageBytes;       // 128 rows x 128 B
  static constexpr int kQBytes = 2 * kHeads * kDim;       // hi + lo: 16 KB
};

template <>
struct DecCfg<DSA_KV_BF16> {
  static constexpr int kStages = DSA_DEC_BF16_STAGES;
  static constexpr int kMaxSlots = DSA_DEC_BF16_SLOTS;
  static constexpr int kPageBytes = kPage * kDim * 2;     // 16 KB
  static constexpr int kTileBytes = 2 * kPageBytes;       // 2 K-blocks x 128 rows x 128 B
  static constexpr int kQBytes = kHeads * kDim * 2;       // 16 KB
};

// Shared memory: [2 query-operand buffers][A stages][control block].
// Control block: barriers at +0, TMEM slot +256, abort flag +260, head
// weights [2][64] at +512, row lengths at +1024, valid-page prefix sums and
// fill-page prefix sums after them (balanced mode).
constexpr int kCtrlLens = 1024;
constexpr int kCtrlPv = kCtrlLens + 4 * kMaxRowsBalanced;
constexpr int kCtrlPf = kCtrlPv + 4 * (kMaxRowsBalanced + 1);
constexpr int kCtrlBytes = kCtrlPf + 4 * (kMaxRowsBalanced + 1);

// The auxiliary region: with the fill, blocks of -inf and of NaN (the
// sources of the bulk copies that write it); with the fused top-k, a chunk's
// logits, a 256-bin histogram and scan scratch.
constexpr int kFillBlock = 4096;
constexpr int kNanBlock = 1024;
constexpr int kSelHist = kSelChunk * 4;            // byte offsets in the region
constexpr int kSelScratch = kSelHist + 256 * 4;
constexpr int kSelBytes = kSelScratch + 64;
// The logits kernel needs the fill blocks; the fused top-k's kernel (SEL)
// the chunk buffer.
template <bool SEL>
constexpr int aux_bytes() {
  return SEL ? kSelBytes : kFillBlock + kNanBlock;
}

template <int KV, bool SEL>
constexpr int dec_smem_bytes() {
  using C = DecCfg<KV>;
  return 1024 /* alignment slack */ + 2 * C::kQBytes + C::kStages * C::kTileBytes +
         aux_bytes<SEL>() + kCtrlBytes;
}

__device__ __forceinline__ float nanf_() { return __int_as_float(0x7fc00000); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 2^e as a float, e in [-126, 127].
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// fp8 keys: the query's lo term is held times kLoScale, in a TMEM
// accumulator of its own; TMEM columns of one CTA: two accumulator buffers
// of 64 heads (bf16), each with a second one for the lo term (fp8)
constexpr float kLoScale = 32.f;
template <int KV>
constexpr uint32_t dec_tmem_cols() { return KV == DSA_KV_FP8_E4M3 ? 256u : 128u; }

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

// Valid pages of a row of length L in a table of W pages (0 for an
// over-long row, which is written NaN by the fill).
__device__ __forceinline__ int valid_pages(int L, int W) {
  if (L > W * kPage || L <= 0) return 0;
  return (L + kPage - 1) / kPage;
}

// The CTA's tiles, in order.  A tile is one or two pages of one row; the
// segment index counts row changes.
struct Tiles {
  // per-request mode
  int G, c, n_mine;
  // balanced mode
  int u, u1;
  const int* Pv;      // exclusive prefix sums of valid pages, rows + 1 entries
  int rows;
  bool balanced;
  // current tile
  int row, seg, pg0, pg1;   // pg1 < 0: single page

  __device__ void init_request(int G_, int c_, int b, int n_mine_) {
    balanced = false;
    G = G_;
    c = c_;
    n_mine = n_mine_;
    u = 0;
    row = b;
    seg = 0;
    set_request();
  }
  __device__ void set_request() {
    pg0 = 2 * u < n_mine ? c + 2 * u * G : -1;
    pg1 = 2 * u + 1 < n_mine ? c + (2 * u + 1) * G : -1;
  }
  __device__ void init_balanced(const int* Pv_, int rows_, int u0, int u1_) {
    balanced = true;
    Pv = Pv_;
    rows = rows_;
    u = u0;
    u1 = u1_;
    seg = 0;
    row = 0;
    if (u < u1) {
      // the row holding unit u0: largest r with Pv[r] <= u0 (and Pv[r+1] > u0)
      int lo = 0, hi = rows - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (Pv[mid] <= u) lo = mid; else hi = mid - 1;
      }
      row = lo;
    }
    set_balanced();
  }
  __device__ void set_balanced() {
    if (u >= u1) {
      pg0 = pg1 = -1;
      return;
    }
    pg0 = u - Pv[row];
    pg1 = (u + 1 < u1 && u + 1 < Pv[row + 1]) ? pg0 + 1 : -1;
  }
  __device__ bool valid() const { return pg0 >= 0; }
  __device__ void next() {
    if (!balanced) {
      ++u;
      set_request();
      return;
    }
    u += pg1 >= 0 ? 2 : 1;
    if (u < u1 && u >= Pv[row + 1]) {
      do {
        ++row;
      } while (Pv[row + 1] <= u);
      ++seg;
    }
    set_balanced();
  }
  // row of segment seg+1 of this CTA, or -1 (balanced mode only)
  __device__ int next_segment_row() const {
    if (!balanced) return -1;
    int r = row + 1;
    while (r < rows && Pv[r + 1] == Pv[r]) ++r;
    return (r < rows && Pv[r] < u1) ? r : -1;
  }
};

// Barrier of the four epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Exclusive prefix sum over the 128 epilogue threads (four warps); `scr`
// holds 4 ints.  Returns this thread's prefix; *total gets the sum.
__device__ __forceinline__ int epi_scan(int v, int* scr, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scr[w] = x;
  epi_sync();
  int base = 0, sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = scr[j];
    if (j < w) base += c;
    sum += c;
  }
  epi_sync();                                 // scr may be reused at once
  *total = sum;
  return base + x - v;
}

// A complete chunk of the fused top-k: its n logits are buf[0, n) (position
// p0 + i at i).  Writes its best min(k, n) -- largest logit first, lower
// position first among equal logits -- into `slot` in position order, with
// the count.  The k-th best key is found by radix selection, 8 bits a pass
// over a 256-bin histogram (one atomic per distinct digit per warp); the
// taken positions are then compacted in order, each warp over a contiguous
// quarter of the chunk, its lanes on consecutive entries.  Called by the 128
// epilogue threads together.
__device__ void select_chunk(const float* buf, int n, int p0, int k, float* slot, int* hist,
                             int* scr) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  float* vals = slot + kSlotHead;
  int* poss = reinterpret_cast<int*>(slot + kSlotHead + k);
  if (n <= k) {
    for (int i = tid; i < n; i += 128) {
      vals[i] = buf[i];
      poss[i] = p0 + i;
    }
    if (tid == 0) *reinterpret_cast<int*>(slot) = n;
    return;
  }
  uint32_t prefix = 0, mask = 0;
  int need = k;                               // still to take among keys matching prefix
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    hist[tid] = 0;
    hist[tid + 128] = 0;
    epi_sync();
    for (int base = 0; base < n; base += 128) {
      const int i = base + tid;
      const uint32_t key = i < n ? sel_key(buf[i]) : 0u;
      const bool m = i < n && (key & mask) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, m);
      if (m) {
        const uint32_t d = (key >> shift) & 255u;
        const unsigned peers = __match_any_sync(act, d);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
      }
    }
    epi_sync();
    const int d1 = 255 - 2 * tid, d0 = d1 - 1;   // this thread's digits, high first
    const int h1 = hist[d1], h0 = hist[d0];
    int tot;
    const int before = epi_scan(h1 + h0, scr, &tot);   // keys in higher digits
    if (before < need && before + h1 >= need) {
      scr[4] = d1;
      scr[5] = before;
    } else if (before + h1 < need && before + h1 + h0 >= need) {
      scr[4] = d0;
      scr[5] = before + h1;
    }
    epi_sync();
    const uint32_t digit = (uint32_t)scr[4];
    need -= scr[5];
    prefix |= digit << shift;
    mask |= 0xFFu << shift;
    epi_sync();                               // hist and scr[4..5] are reused
  }
  // prefix is the k-th best key; `need` keys equal to it are taken, the
  // lowest positions first.  Warp w compacts [b0, b1).
  const int per = ((n + 3) / 4 + 31) & ~31;
  const int b0 = min(w * per, n), b1 = min(b0 + per, n);
  const unsigned lt = (1u << lane) - 1u;
  int gt_w = 0, eq_w = 0;
  for (int i0 = b0; i0 < b1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < b1 ? sel_key(buf[i]) : 0u;
    gt_w += __popc(__ballot_sync(0xffffffffu, i < b1 && key > prefix));
    eq_w += __popc(__ballot_sync(0xffffffffu, i < b1 && key == prefix));
  }
  if (lane == 0) {
    scr[8 + w] = gt_w;
    scr[12 + w] = eq_w;
  }
  epi_sync();
  int o = 0, e = 0;                           // taken, and equal keys, before this warp
  for (int v = 0; v < w; ++v) {
    const int eqv = scr[12 + v];
    o += scr[8 + v] + min(max(need - e, 0), eqv);
    e += eqv;
  }
  for (int i0 = b0; i0 < b1; i0 += 32) {
    const int i = i0 + lane;
    const float v = i < b1 ? buf[i] : 0.f;
    const uint32_t key = sel_key(v);
    const bool g = i < b1 && key > prefix, q = i < b1 && key == prefix;
    const unsigned qb = __ballot_sync(0xffffffffu, q);
    const bool take = g || (q && e + __popc(qb & lt) < need);
    const unsigned tb = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int dst = o + __popc(tb & lt);
      vals[dst] = v;
      poss[dst] = p0 + i;
    }
    o += __popc(tb);
    e += __popc(qb);
  }
  if (tid == 0) *reinterpret_cast<int*>(slot) = k;
}

}  // namespace

// SEL: the fused top-k's instance (the epilogue keeps each chunk's logits in
// shared memory and selects its best; no fill).  The logits instance carries
// none of that code.
template <int KV, bool SEL>
__global__ void __launch_bounds__(kDecThreads, kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const RowsParams p, const int G, const int balanced, const int early_tmem) {
  using C = DecCfg<KV>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // 2 x B operand (row segments alternate)
  uint8_t* sA = smem + 2 * C::kQBytes;         // A stages
  uint8_t* sAux = sA + S * C::kTileBytes;    // [aux_bytes<SEL>()]
  uint8_t* sInf = sAux;                       // fill: [kFillBlock] -inf
  uint8_t* sNan = sAux + kFillBlock;          // fill: [kNanBlock] NaN
  uint8_t* ctrl = sAux + aux_bytes<SEL>();
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;                 // [2] accumulator ready
  uint64_t* tempty = tfull + 2;                // [2] accumulator drained
  uint64_t* qbar = tempty + 2;                 // [2] query operand ready
  uint64_t* bempty = qbar + 2;                 // [2] query operand no longer read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 260);
  int* slice_s = reinterpret_cast<int*>(ctrl + 264);    // balanced: this CTA's [u0, u1)
  volatile int* tiles_out = reinterpret_cast<volatile int*>(ctrl + 272);  // producer: tiles issued
  float* w_s = reinterpret_cast<float*>(ctrl + 512);     // [2][64]
  int* lens_s = reinterpret_cast<int*>(ctrl + kCtrlLens);
  int* Pv = reinterpret_cast<int*>(ctrl + kCtrlPv);
  int* Pf = reinterpret_cast<int*>(ctrl + kCtrlPf);
  static_assert((2 * S + 8) * 8 <= 256, "control block overflow");

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int T = p.W * kPage;

  // Prologue that reads no input: it may overlap the previous launch.
  if (tid == 128) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
      mbar_init(&qbar[a], KV == DSA_KV_BF16 ? 1 : 128);
      mbar_init(&bempty[a], 1);
    }
    *abort_flag = 0;
    *tiles_out = 0;
    fence_barrier_init();
    prefetch_tmap(&kmap);
    if (KV == DSA_KV_BF16) prefetch_tmap(&qmap);
  }
  // With more than one CTA per SM, the tensor memory is taken before the
  // wait for the previous launch: an SM was measured to start a launch's
  // second CTA only once its first had allocated and given up the
  // allocation permit (~3 us later in balanced mode, after the lengths'
  // prefix sums).  A CTA that then leaves before the main body frees it.
  if (early_tmem && warp == 5) {
    tmem_alloc(tmem_slot, dec_tmem_cols<KV>());
    tmem_relinquish();
  }
  // the blocks of -inf / NaN the balanced mode's fill is copied from (the
  // logits instance; written before the wait, as they read no input)
  if (!SEL && warp == 4 && balanced) {
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const float4 qnan = make_float4(nanf_(), nanf_(), nanf_(), nanf_());
    for (int j = lane; j < kFillBlock / 16; j += 32) reinterpret_cast<float4*>(sInf)[j] = ninf;
    for (int j = lane; j < kNanBlock / 16; j += 32) reinterpret_cast<float4*>(sNan)[j] = qnan;
    fence_proxy_async_smem();
    __syncwarp();
  }
  auto leave_early = [&]() {
    if (!early_tmem) return;
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
      tc_fence_after();
      tmem_dealloc(*tmem_slot, dec_tmem_cols<KV>());
    }
  };
  griddep_wait();
  griddep_launch_dependents();

  // fp8 query split, done by warps 0-3 (warp w owns heads 16w..16w+15, lane
  // l owns d = 4l..4l+3): q_load fetches row r's query and head weights,
  // q_convert writes q * 2^e_h = hi + lo * 2^-5 into query buffer sb as two
  // e4m3 terms (K-major, 128-byte swizzle) and the weights w_h * 2^-e_h
  auto q_load = [&](int r, uint2 (&raw)[16], float& wv) {
    const uint16_t* qrow = p.q + (long long)r * kHeads * kDim;
#pragma unroll
    for (int hh = 0; hh < 16; ++hh)
      raw[hh] = __ldg(reinterpret_cast<const uint2*>(qrow + (warp * 16 + hh) * kDim) + lane);
    wv = lane < 16 ? __ldg(p.w + (long long)r * kHeads + warp * 16 + lane) : 0.f;
  };
  auto q_convert = [&](const uint2 (&raw)[16], float wv, int sb) {
    float* ws = w_s + sb * kHeads;
    uint8_t* qb = sQ + sb * C::kQBytes;
#pragma unroll
    for (int hh = 0; hh < 16; ++hh) {
      const int h = warp * 16 + hh;
      float x[4] = {bf16f(raw[hh].x & 0xffffu), bf16f(raw[hh].x >> 16),
                    bf16f(raw[hh].y & 0xffffu), bf16f(raw[hh].y >> 16)};
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
        // the residual is exact in fp32 and below 2^3 (hi's half step for
        // |a| < 2^8): times 2^5 it stays within e4m3's range
        const uint32_t lc = to_e4m3x2((a0 - h0) * kLoScale, (a1 - h1) * kLoScale, l0, l1);
        hi |= hc << (8 * j);
        lo |= lc << (8 * j);
      }
      // row h, bytes [4*lane, 4*lane+4) of 128, 128-byte swizzle
      const uint32_t off = h * 128 + ((((lane >> 2) ^ (h & 7)) << 4) | ((lane & 3) << 2));
      *reinterpret_cast<uint32_t*>(qb + off) = hi;
      *reinterpret_cast<uint32_t*>(qb + 8192 + off) = lo;
      const float wh = __shfl_sync(0xffffffffu, wv, hh);
      if (lane == 0) ws[h] = wh * exp2i(-e);
    }
    fence_proxy_async_smem();
    mbar_arrive(&qbar[sb]);
  };
  uint2 q0raw[16];           // fp8: the first segment's query, loaded first of all
  float q0w = 0.f;

  // This CTA's share of the fill.  Per-request mode: floats [fill_beg,
  // fill_end) of row blockIdx.y; balanced mode: fill pages [fill_f0,
  // fill_f1) of the call (Pf holds the rows' fill-page prefix sums).
  long long fill_beg = 0, fill_end = 0;
  bool fill_bad = false;
  int fill_f0 = 0, fill_f1 = 0;
  int my_pages = 0;                   // pages this CTA loads (pacing of the fill)

  // Calls f(first float, count, over-long row) for each contiguous piece of
  // this CTA's share of the fill (each starts 16-byte aligned and counts a
  // multiple of 4 floats); raises DSA_ERR_BAD_SEQLEN for an over-long row.
  auto for_each_fill_range = [&](bool report, auto&& f) {
    if (!balanced) {
      if (fill_end > fill_beg)
        f(p.out + (long long)blockIdx.y * p.out_stride + fill_beg, fill_end - fill_beg, fill_bad);
      return;
    }
    const int B = p.rows;
    if (fill_f0 >= fill_f1) return;
    int lo = 0, hi = B - 1;
    while (lo < hi) {      // row holding fill page fill_f0
      const int mid = (lo + hi + 1) >> 1;
      if (Pf[mid] <= fill_f0) lo = mid; else hi = mid - 1;
    }
    for (int r = lo, fp = fill_f0; fp < fill_f1 && r < B; ++r) {
      const int nf = Pf[r + 1] - Pf[r];
      if (nf == 0) continue;
      const int a = fp - Pf[r];                      // first fill page of row r in range
      const int e = min(fill_f1 - Pf[r], nf);        // one past the last
      const bool bad = lens_s[r] > T;
      const int first_page = p.W - nf;               // = valid pages of row r
      f(p.out + (long long)r * p.out_stride + (long long)(first_page + a) * kPage,
        (long long)(e - a) * kPage, bad);
      if (bad && a == 0 && report) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
      fp = Pf[r] + e;
    }
  };

  Tiles tiles;
  int early_ph[2] = {-1, -1};   // balanced mode: the first tile's table entries (producer lane 0)
  if (!balanced) {
    // ---------------------------------------------------------------- per-request
    const int b = blockIdx.y, c = blockIdx.x;
    const int L = __ldg(p.seqlens + b);
    const int npv = valid_pages(L, p.W);
    const int n_mine = npv > c ? (npv - 1 - c) / G + 1 : 0;
    if (KV == DSA_KV_FP8_E4M3 && tid < 128 && n_mine > 0) q_load(b, q0raw, q0w);
    {
      // -inf (NaN for an over-long row) past the last valid page, split over
      // the row's G CTAs in contiguous 16-byte-aligned chunks
      fill_bad = L > T;
      const int f0 = npv * kPage;
      int chunk = (T - f0 + G - 1) / G;
      chunk = (chunk + 3) & ~3;
      fill_beg = f0 + (long long)c * chunk;
      fill_end = p.fill ? min(fill_beg + chunk, (long long)T) : fill_beg;
      if (fill_bad && c == 0 && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
    }
    // per-request mode: the epilogue warps write the CTA's share with
    // streaming stores (its share is small; measured faster here than the
    // producer's bulk copies, whose set-up every one of the many CTAs pays)
    if (n_mine > 0 && tid < 128) {
      const float fv = fill_bad ? nanf_() : -INFINITY;
      const float4 v4 = make_float4(fv, fv, fv, fv);
      float* orow = p.out + (long long)b * p.out_stride;
      for (long long i = fill_beg + 4 * tid; i < fill_end; i += 4 * 128)
        __stcs(reinterpret_cast<float4*>(orow + i), v4);
    }
    if (n_mine > 0) fill_end = fill_beg;    // nothing left for the producer
    if (n_mine == 0) {
      const float fv = fill_bad ? nanf_() : -INFINITY;
      const float4 v4 = make_float4(fv, fv, fv, fv);
      float* orow = p.out + (long long)b * p.out_stride;
      for (long long i = fill_beg + 4 * tid; i < fill_end; i += 4 * kDecThreads)
        __stcs(reinterpret_cast<float4*>(orow + i), v4);
      leave_early();
      return;
    }
    if (tid == 0) lens_s[0] = L;
    my_pages = n_mine;
    tiles.init_request(G, c, b, n_mine);
  } else {
    // ---------------------------------------------------------------- balanced
    const int B = p.rows;
    for (int j = tid; j < B; j += kDecThreads) lens_s[j] = __ldg(p.seqlens + j);
    __syncthreads();
    if (warp == 0) {
      // exclusive prefix sums of valid pages, and the count of non-empty
      // rows; a row's fill pages are W minus its valid pages, so their
      // prefix sums follow: Pf[j] = j * W - Pv[j]
      int run_v = 0, n_rows = 0;
      for (int base = 0; base < B; base += 32) {
        const int j = base + lane;
        const int v = j < B ? valid_pages(lens_s[j], p.W) : 0;
        n_rows += __popc(__ballot_sync(0xffffffffu, v > 0));
        int sv = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int tv = __shfl_up_sync(0xffffffffu, sv, o);
          if (lane >= o) sv += tv;
        }
        if (j < B) {
          Pv[j] = run_v + sv - v;
          Pf[j] = (int)((long long)j * p.W - (run_v + sv - v));
        }
        run_v += __shfl_sync(0xffffffffu, sv, 31);
      }
      if (lane == 0) {
        Pv[B] = run_v;
        Pf[B] = (int)((long long)B * p.W - run_v);
      }
      __syncwarp();
      // fp8 keys: this CTA's pages [u0, u1) balance pages plus a weight Y
      // per row start (a row segment's query is loaded and split by the
      // CTA itself), Y = min(6, pages per CTA / 4) so that short slices are
      // not swamped by it; each CTA takes the units whose weighted starts
      // fall in [k * NW / R, (k + 1) * NW / R), a row's first unit weighing
      // 1 + Y.  bf16 keys (the query comes by TMA) and the fused top-k (its
      // slots follow the plain split) take Y = 0, the plain split.
      const int Rg = gridDim.x;
      const int Y = (KV == DSA_KV_FP8_E4M3 && !SEL) ? min(6, run_v / Rg / 4) : 0;
      // the two slice ends k * NW / R and (k + 1) * NW / R, as c * q +
      // (c * r) / R with NW = q * R + r (c * r < R * R), found in one pass
      // over the rows; a row's count of non-empty rows before it comes from
      // a ballot
      const long long NW = run_v + (long long)Y * n_rows;
      long long q;
      unsigned r;
      if (NW < (1ll << 31)) {            // the usual case: a 32-bit division
        const unsigned nw = (unsigned)NW, q32 = nw / (unsigned)Rg;
        q = q32;
        r = nw - q32 * (unsigned)Rg;
      } else {
        q = NW / Rg;
        r = (unsigned)(NW - q * Rg);
      }
      long long xe[2];
      int ue[2] = {run_v, run_v};
      bool found[2] = {false, false};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const unsigned c = blockIdx.x + e;
        xe[e] = (long long)c * q + (long long)(c * r / (unsigned)Rg);
      }
      int nb = 0;
      for (int base = 0; base < B && !(found[0] && found[1]); base += 32) {
        const int j = base + lane;
        const int len = j < B ? Pv[j + 1] - Pv[j] : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, len > 0);
        const int before = nb + __popc(bal & ((1u << lane) - 1u));
        const long long pw = Pv[min(j, B)] + (long long)Y * before;   // the row's weighted start
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (found[e]) continue;                                     // warp-uniform
          const unsigned hb = __ballot_sync(0xffffffffu, len > 0 && xe[e] < pw + len + Y);
          if (hb) {
            const int src = __ffs(hb) - 1;
            int uu = 0;
            if (lane == src) {
              const long long i = xe[e] <= pw ? 0 : max(1ll, xe[e] - pw - Y);
              uu = Pv[j] + (int)min(i, (long long)len);
            }
            ue[e] = __shfl_sync(0xffffffffu, uu, src);
            found[e] = true;
          }
        }
        nb += __popc(bal);
      }
      if (lane == 0) {
        slice_s[0] = ue[0];
        slice_s[1] = ue[1];
      }
      if (SEL) {
        // fused top-k: exclusive prefix sums of the rows' chunk counts (the
        // rows' first slots) replace the fill prefix sums
        __syncwarp();
        const Slicer sl(max(run_v, 1), gridDim.x);
        int run_s = 0;
        for (int base = 0; base < B; base += 32) {
          const int j = base + lane;
          const int cnt = j < B ? sl.row_chunks(Pv[j], Pv[j + 1], 1 << 30) : 0;
          int sc = cnt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o) sc += t;
          }
          if (j < B) Pf[j] = run_s + sc - cnt;
          run_s += __shfl_sync(0xffffffffu, sc, 31);
        }
        if (lane == 0) Pf[B] = run_s;
        __syncwarp();
        if (blockIdx.x == 0) {
          int* hdr = reinterpret_cast<int*>(p.sel_ws);
          for (int j = lane; j <= B; j += 32) hdr[j] = Pf[j];
        }
      }
    }
    __syncthreads();
    // this CTA's fill pages [k * F / R, (k + 1) * F / R), as c * q + (c * r) / R
    const unsigned R = gridDim.x, k = blockIdx.x;
    const int F = p.fill ? Pf[B] : 0;
    const int u0 = slice_s[0], u1 = slice_s[1];
    const int fq = F / (int)R;
    const unsigned fr = (unsigned)(F - fq * (int)R);
    const int f0 = (int)k * fq + (int)(k * fr / R), f1 = (int)(k + 1) * fq + (int)((k + 1) * fr / R);
    if (u0 < u1) {
      tiles.init_balanced(Pv, B, u0, u1);
      if (KV == DSA_KV_FP8_E4M3 && tid < 128) q_load(tiles.row, q0raw, q0w);
      if (KV == DSA_KV_FP8_E4M3 && tid == 128) {
        // the producer's first tile: its table entries, read now (fp8 keys:
        // measured 0.1 us faster on short slices; bf16 keys, whose first
        // tile waits behind its query load anyway, measured 0.8 us slower)
        const int* btrow = p.block_table + (long long)tiles.row * p.bt_stride;
        early_ph[0] = __ldg(btrow + tiles.pg0);
        if (tiles.pg1 >= 0) early_ph[1] = __ldg(btrow + tiles.pg1);
      }
    }

    fill_f0 = f0;
    fill_f1 = f1;
    my_pages = u1 - u0;
    if (u0 >= u1) {
      // no pages: the whole CTA writes its share of the fill
      for_each_fill_range(tid == 0, [&](float* dst, long long n, bool bad) {
        const float fv = bad ? nanf_() : -INFINITY;
        const float4 v4 = make_float4(fv, fv, fv, fv);
        for (long long i = 4 * tid; i < n; i += 4 * kDecThreads)
          __stcs(reinterpret_cast<float4*>(dst + i), v4);
      });
      leave_early();
      return;
    }
  }

  if (!early_tmem && warp == 5) {
    tmem_alloc(tmem_slot, dec_tmem_cols<KV>());
    tmem_relinquish();
  }
  // Barrier 2: the TMEM address (and, in per-request mode, the barrier
  // initialisation) reaches the MMA and epilogue warps.  The producer only
  // arrives: it uses neither, and starts loading pages at once.
  if (warp == 4) {
    asm volatile("bar.arrive 2, %0;" ::"n"(kDecThreads) : "memory");
  } else {
    tc_fence_before();
    asm volatile("bar.sync 2, %0;" ::"n"(kDecThreads) : "memory");
    tc_fence_after();
  }
  const uint32_t tmem_base = warp == 4 ? 0u : *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    // The fill goes out as bulk copies from blocks of -inf / NaN in shared
    // memory.  Lanes 1-31 issue them all at once (copies from one thread
    // complete one after another; from 31 they overlap) once lane 0 has
    // issued its last page loads: the page reads stream first, and the
    // writes, absorbed by L2, drain while the last tiles are processed
    // (config 3: 28.2 us, against 30.2 us when released after the first S
    // tiles and 32.6 us at once).  bf16 keys, CTA with a long
    // page stream (16 pages or more): lane 0 issues them instead, in step
    // with its page loads, a share after every tile from the S-th on, so
    // that DRAM serves a steady mix of reads and writes (measured ~1% faster
    // on 2,048-page tables).  fp8 keys keep the burst alone: with the paced
    // loop compiled in, their short calls were measured slower even where
    // it never ran.  (Pacing lanes 1-31 by lane 0's progress, or the whole
    // warp issuing the burst between lane 0's first and later stages, was
    // also slower.)
    const bool any_fill = balanced ? fill_f0 < fill_f1 : fill_end > fill_beg;
    // this CTA's tiles; the paced fill starts after the first S of them
    const int n_tiles = max((my_pages + 1) / 2, 1);
    const int first_fill = min(S, n_tiles);
    constexpr bool kCanPace = KV == DSA_KV_BF16;
    const bool paced = kCanPace && any_fill && my_pages >= 16;
    const bool burst = any_fill && !paced;

    // lane 0's share of the fill (paced): a cursor over the ranges, the
    // current one f_n floats from f_dst (NaN for an over-long row), the next
    // one starting at fill page f_fp in row f_row or later
    float* f_dst = nullptr;
    long long f_n = 0;
    bool f_bad = false;
    int f_row = 0, f_fp = fill_f0;
    if (!balanced) {
      f_dst = p.out + (long long)blockIdx.y * p.out_stride + fill_beg;
      f_n = paced ? max(fill_end - fill_beg, 0ll) : 0;
      f_bad = fill_bad;
    } else if (paced && lane == 0) {
      int lo = 0, hi = p.rows - 1;
      while (lo < hi) {      // row holding fill page fill_f0
        const int mid = (lo + hi + 1) >> 1;
        if (Pf[mid] <= fill_f0) lo = mid; else hi = mid - 1;
      }
      f_row = lo;
    } else {
      f_fp = fill_f1;        // nothing for the cursor
    }
    auto next_range = [&]() -> bool {
      if (!balanced || f_fp >= fill_f1) return false;
      while (f_row < p.rows && Pf[f_row + 1] <= f_fp) ++f_row;
      if (f_row >= p.rows) return false;
      const int nf = Pf[f_row + 1] - Pf[f_row];
      const int a = f_fp - Pf[f_row];                  // first fill page of the row in range
      const int e = min(fill_f1 - Pf[f_row], nf);      // one past the last
      f_bad = lens_s[f_row] > T;
      if (f_bad && a == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
      f_dst = p.out + (long long)f_row * p.out_stride + (long long)(p.W - nf + a) * kPage;
      f_n = (long long)(e - a) * kPage;
      f_fp = Pf[f_row] + e;
      return true;
    };
    // issue `budget` more floats of lane 0's share (a multiple of 4; < 0 = all)
    auto issue_fill = [&](long long budget) {
      bool any = false;
      while (budget != 0) {
        if (f_n == 0 && !next_range()) break;
        long long n = min(f_n, (long long)((f_bad ? kNanBlock : kFillBlock) / 4));
        if (budget > 0) n = min(n, budget);
        bulk_store(f_dst, f_bad ? sNan : sInf, (uint32_t)(4 * n));
        f_dst += n;
        f_n -= n;
        if (budget > 0) budget -= n;
        any = true;
      }
      if (any) bulk_commit();
    };
    // the paced share per loaded page, from the first stages on
    long long per_page = 0;
    if (paced) {
      const long long fill_total =
          balanced ? (long long)(fill_f1 - fill_f0) * kPage : max(fill_end - fill_beg, 0ll);
      const long long paced_pages = max(my_pages - 2 * (first_fill - 1), 1);
      per_page = ((fill_total + paced_pages - 1) / paced_pages + kPage - 1) / kPage * kPage;
    }

    // lane 0's page loop, compiled with and without the paced fill
    int issued = 0, seg_loaded = -1;
    bool ok = true;
    auto page_loop = [&](auto paced_c) {
      constexpr bool kPaced = decltype(paced_c)::value;
      Tiles it = tiles;
      for (int i = 0; it.valid(); ++i, it.next()) {
        if (KV == DSA_KV_BF16 && it.seg != seg_loaded) {
          // query of this row segment -> buffer seg % 2, once segment seg-2
          // (the buffer's previous user) has finished its MMAs
          const int sb = it.seg & 1;
          if (it.seg >= 2) ok = mbar_wait_bounded(&bempty[sb], ((it.seg - 2) >> 1) & 1, kWaitLimit);
          if (!ok) break;
          mbar_arrive_expect_tx(&qbar[sb], C::kQBytes);
          tma_load_2d(sQ + sb * C::kQBytes, &qmap, &qbar[sb], 0, it.row * kHeads);
          tma_load_2d(sQ + sb * C::kQBytes + C::kQBytes / 2, &qmap, &qbar[sb], kHalfRowUnits,
                      it.row * kHeads);
          seg_loaded = it.seg;
        }
        const int s = i % S;
        if (i >= S) ok = mbar_wait_bounded(&empty[s], ((i / S) - 1) & 1, kWaitLimit);
        if (!ok || *abort_flag) break;
#ifdef DSA_TEST_SKIP_FIRST_TILE
        // test builds only: never deliver the first tile, so that the MMA's
        // bounded wait for it runs out and the call reports DSA_ERR_TIMEOUT
        if (i == 0) {
          issued = i + 1;
          continue;
        }
#endif
        const int* btrow = p.block_table + (long long)it.row * p.bt_stride;
        int phys[2];
        uint32_t bytes = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int pg = h == 0 ? it.pg0 : it.pg1;
          phys[h] = -1;
          if (pg >= 0) {
            const int ph = (KV == DSA_KV_FP8_E4M3 && balanced && i == 0) ? early_ph[h]
                                                                        : __ldg(btrow + pg);
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
            tma_load_3d(st + C::kTileBytes / 2 + h * (C::kPageBytes / 2), &kmap, &full[s],
                        kHalfRowUnits, 0, phys[h]);
          }
        }
        issued = i + 1;
        *tiles_out = i + 1;
        if (kPaced && i + 1 >= first_fill) issue_fill(per_page * (it.pg1 >= 0 ? 2 : 1));
      }
    };
    if (lane != 0) {
      if (burst) {
        // wait (bounded: ~0.5 s) for lane 0's last page loads, then issue
        // this lane's chunks: chunk c of the CTA's share (4 KB, or 1 KB of
        // NaN) goes to lane 1 + c % 31
        for (int spin = 0; *tiles_out < n_tiles && spin < (1 << 22); ++spin) __nanosleep(128);
        int c = 0;
        bool any = false;
        for_each_fill_range(lane == 1, [&](float* dst, long long n, bool bad) {
          const long long blk = (bad ? kNanBlock : kFillBlock) / 4;
          for (long long j = 0; j < n; j += blk, ++c) {
            if (c % 31 != lane - 1) continue;
            bulk_store(dst + j, bad ? sNan : sInf, (uint32_t)(4 * min(blk, n - j)));
            any = true;
          }
        });
        if (any) bulk_commit();
      }
    } else {
      if (kCanPace && paced) page_loop(BoolC<kCanPace>{});
      else page_loop(BoolC<false>{});
      *tiles_out = 1 << 30;                  // release the lanes' fill
      if (paced) issue_fill(-1);             // the rest of lane 0's share
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, DSA_ERR_TIMEOUT);
      }
      // never leave the CTA with copies in flight: wait for the last use of
      // every stage and query buffer (already complete on the normal path)
      for (int i = max(0, issued - S); i < issued; ++i)
        mbar_wait_bounded(&full[i % S], (i / S) & 1, kWaitLimit);
      if (KV == DSA_KV_BF16 && seg_loaded >= 0) {
        for (int sg = max(0, seg_loaded - 1); sg <= seg_loaded; ++sg)
          mbar_wait_bounded(&qbar[sg & 1], (sg >> 1) & 1, kWaitLimit);
      }
    }
    if (any_fill) bulk_wait_reads();         // the fill blocks are read: the CTA may exit
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc =
          KV == DSA_KV_FP8_E4M3 ? instr_desc(0, 0, 128, kHeads) : instr_desc(1, 1, 128, kHeads);
      const uint32_t sQa = smem_u32(sQ);
      const uint32_t sAa = smem_u32(sA);
      Tiles it = tiles;
      int issued = 0, seg_ready = -1;
      bool ok = true;
      for (int i = 0; it.valid(); ++i) {
        const int s = i % S, a = i & 1, seg = it.seg;
        if (seg != seg_ready) {
          ok = mbar_wait_bounded(&qbar[seg & 1], (seg >> 1) & 1, kWaitLimit);
          seg_ready = seg;
        }
        if (ok) ok = mbar_wait_bounded(&full[s], (i / S) & 1, kWaitLimit);
        if (ok && i >= 2) ok = mbar_wait_bounded(&tempty[a], ((i >> 1) - 1) & 1, kWaitLimit);
        if (!ok || *abort_flag) break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * kHeads;
        const uint32_t st = sAa + s * C::kTileBytes;
        const uint32_t bq = sQa + (seg & 1) * C::kQBytes;
        if (KV == DSA_KV_FP8_E4M3) {
          // A: 128 rows x 128 B; B: hi then lo, 64 rows x 128 B each; K = 32
          // per MMA; the lo term into its own accumulator, 128 columns on
#pragma unroll
          for (int term = 0; term < 2; ++term) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(st + 32 * k, 1024);
              const uint64_t bd = smem_desc_sw128(bq + term * 8192 + 32 * k, 1024);
              mma_f8f6f4(d + term * 128, ad, bd, idesc, k != 0);
            }
          }
        } else {
          // two K-blocks of 64 bf16; K = 16 per MMA
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t kb = k >> 2, ko = (k & 3) * 32;
            const uint64_t ad = smem_desc_sw128(st + kb * (C::kTileBytes / 2) + ko, 1024);
            const uint64_t bd = smem_desc_sw128(bq + kb * (C::kQBytes / 2) + ko, 1024);
            mma_f16(d, ad, bd, idesc, k != 0);
          }
        }
        mma_commit(&empty[s]);
        mma_commit(&tfull[a]);
        issued = i + 1;
        it.next();
        if (!it.valid() || it.seg != seg) mma_commit(&bempty[seg & 1]);   // query buffer free
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
    // ------------------------------------------------------------ warps 0-3
    // Prepare row r's query operand in buffer sb: fp8 splits q into e4m3 hi
    // + lo with a power-of-two scale per head (warp w owns heads 16w..16w+15,
    // lane l owns d = 4l..4l+3); both dtypes stage the head weights.
    auto prepare = [&](int r, int sb) {
      if (KV == DSA_KV_FP8_E4M3) {
        uint2 qraw[16];
        float wv;
        q_load(r, qraw, wv);
        q_convert(qraw, wv, sb);
      } else {
        if (tid < kHeads) w_s[sb * kHeads + tid] = __ldg(p.w + (long long)r * kHeads + tid);
      }
    };

    bool ok = true;
    // segments 0 and 1 use fresh buffers; segment 0's query was loaded
    // before the fill (fp8)
    if (KV == DSA_KV_FP8_E4M3) q_convert(q0raw, q0w, 0);
    else prepare(tiles.row, 0);
    const int r1 = tiles.next_segment_row();
    if (r1 >= 0) prepare(r1, 1);
    asm volatile("bar.sync 1, 128;" ::: "memory");

    const int r = warp * 32 + lane;            // accumulator row = TMEM lane
    const int half = r >> 6, slot = r & 63;
    // fused top-k: the open chunk (row, first position, valid positions so
    // far, its slot); chunk_row < 0 = none open
    const bool sel = SEL && balanced;          // the host launches it only so
    float* selbuf = reinterpret_cast<float*>(sAux);
    int* selhist = reinterpret_cast<int*>(sAux + kSelHist);
    int* selscr = reinterpret_cast<int*>(sAux + kSelScratch);
    int chunk_row = -1, chunk_seg = -1, chunk_c = -1, chunk_p0 = 0, chunk_n = 0, seg_first = 0;
    int seg_slot0 = 0;                         // the segment's first slot
    float* chunk_slot = nullptr;
    auto flush_chunk = [&]() {
      epi_sync();                              // every logit of the chunk is in selbuf
      select_chunk(selbuf, chunk_n, chunk_p0, p.sel_k, chunk_slot, selhist, selscr);
      epi_sync();                              // selbuf is free again
      chunk_row = -1;
    };
    Tiles it = tiles;
    int cur_seg = 0;
    for (int i = 0; it.valid(); ++i, it.next()) {
      const int a = i & 1;
      if (it.seg != cur_seg) {
        // entering segment s >= 1: segment s+1 may take over buffer
        // (s+1) % 2 once segment s-1's MMAs are done (they are: their
        // accumulators have been read)
        cur_seg = it.seg;
        const int rn = it.next_segment_row();
        if (rn >= 0) {
          const int sb = (cur_seg + 1) & 1;
          if (ok) ok = mbar_wait_bounded(&bempty[sb], ((cur_seg - 1) >> 1) & 1, kWaitLimit);
          ok = __all_sync(0xffffffffu, ok);
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (ok) prepare(rn, sb);
          asm volatile("bar.sync 1, 128;" ::: "memory");
        }
      }
      const int row = it.row;
      const int L = balanced ? lens_s[row] : lens_s[0];
      const int Lc = L > T ? 0 : max(L, 0);
      if (sel) {
        // the tile's chunk: pages counted from the segment's first page, in
        // groups of kSelChunkPages (tiles pair pages from the segment's
        // first, so a tile never straddles two chunks)
        const bool new_seg = it.seg != chunk_seg;
        if (new_seg) seg_first = it.pg0;
        const int c = (it.pg0 - seg_first) / kSelChunkPages;
        if (chunk_row >= 0 && (new_seg || c != chunk_c)) flush_chunk();
        if (new_seg) {
          // slots of the row's chunks held by the CTAs before this one
          const Slicer sl(max(Pv[p.rows], 1), gridDim.x);
          seg_slot0 = Pf[row] + sl.row_chunks(Pv[row], Pv[row + 1], blockIdx.x);
        }
        if (chunk_row < 0) {
          chunk_row = row;
          chunk_seg = it.seg;
          chunk_c = c;
          chunk_p0 = (seg_first + c * kSelChunkPages) * kPage;
          chunk_n = 0;
          chunk_slot = p.sel_ws + sel_header_floats(p.rows) + (long long)(seg_slot0 + c) *
                                                                sel_slot_floats(p.sel_k);
        }
        const int last_pg = it.pg1 >= 0 ? it.pg1 : it.pg0;
        chunk_n = max(chunk_n, min((last_pg + 1) * kPage, Lc) - chunk_p0);
      }
      const int pg = half ? it.pg1 : it.pg0;
      const bool row_valid = pg >= 0;
      const int t = pg * kPage + slot;
      const int* btrow = p.block_table + (long long)row * p.bt_stride;
      int phys = -1;
      float scale = 1.f;
      if (row_valid) {
        phys = __ldg(btrow + pg);
        if (phys >= 0 && phys < p.num_pages && t < Lc && p.kscale != nullptr)
          scale = __ldg(reinterpret_cast<const float*>(p.kscale + (long long)phys * p.page_stride) +
                        slot);
      }
      if (ok) ok = mbar_wait_bounded(&tfull[a], (i >> 1) & 1, kWaitLimit);
      ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);   // warp-uniform for tcgen05.ld
      float* orow = p.out + (long long)row * p.out_stride;
      if (!ok) {
        if (sel) {
          if (row_valid && t < Lc) selbuf[t - chunk_p0] = nanf_();
        } else if (row_valid) {
          orow[t] = t < Lc ? nanf_() : -INFINITY;
        }
        continue;
      }
      tc_fence_after();
      const float* ws = w_s + (cur_seg & 1) * kHeads;
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + a * kHeads;
      if (KV == DSA_KV_FP8_E4M3) {
        // S = hi + lo * 2^-5, 16 heads at a time (heads 0-31 to one partial
        // sum, 32-63 to the other, as below); the next 16 heads' loads are
        // in flight while the current ones are summed
        uint32_t vh[2][16], vl[2][16];
        tmem_ld_32x32b_x16(taddr, vh[0]);
        tmem_ld_32x32b_x16(taddr + 128, vl[0]);
        tmem_ld_wait(vh[0], vl[0]);
        const float2 lsc = make_float2(1.f / kLoScale, 1.f / kLoScale);
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          const int cb = part & 1;
          if (part < 3) {
            tmem_ld_32x32b_x16(taddr + 16 * (part + 1), vh[cb ^ 1]);
            tmem_ld_32x32b_x16(taddr + 128 + 16 * (part + 1), vl[cb ^ 1]);
          }
          float2& acc = part < 2 ? acc0 : acc1;
#pragma unroll
          for (int h = 0; h < 16; h += 2) {
            const float2 wv = *reinterpret_cast<const float2*>(ws + 16 * part + h);
            const float2 sv = __ffma2_rn(
                make_float2(__uint_as_float(vl[cb][h]), __uint_as_float(vl[cb][h + 1])), lsc,
                make_float2(__uint_as_float(vh[cb][h]), __uint_as_float(vh[cb][h + 1])));
            acc = __ffma2_rn(wv, make_float2(fmaxf(sv.x, 0.f), fmaxf(sv.y, 0.f)), acc);
          }
          if (part < 3) tmem_ld_wait(vh[cb ^ 1], vl[cb ^ 1]);
          if (part == 2) {
            // every column is in registers: the accumulator buffer is free
            tc_fence_before();
            mbar_arrive(&tempty[a]);
          }
        }
      } else {
      uint32_t v0[32], v1[32];
      tmem_ld_32x32b_x32(taddr, v0);
      tmem_ld_32x32b_x32(taddr + 32, v1);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[a]);
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        const float4 wa = *reinterpret_cast<const float4*>(ws + h);
        const float4 wb = *reinterpret_cast<const float4*>(ws + 32 + h);
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
        if (!sel) orow[t] = o;
        else if (t < Lc) selbuf[t - chunk_p0] = o;
      }
    }
    if (sel && chunk_row >= 0) flush_chunk();
    if (!ok) raise_status(p.status, DSA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, dec_tmem_cols<KV>());
  }
}

// ----------------------------------------------------------------------------
// host side

bool decode_is_balanced(int W, int rows) { return W > 64 && rows <= kMaxRowsBalanced; }

// CTAs per request in per-request mode, from the launch shape only: at most
// the per-dtype cap and W.  For a short table (W <= 64 pages, so no request
// is long) about two CTAs per SM in total, the resident limit: each CTA
// pipelines a few pages instead of paying its start-up latency for one.
// (Measured: B=16/32 rows 5.3 / 5.4 us per launch at two per SM, 5.8 at one;
// before the tensor memory was taken ahead of the dependent-launch wait, an
// SM started its second CTA ~1.4 us late and one per SM was faster.)
template <int KV>
int decode_slots(int W, int B, int sms) {
  int G = W < DecCfg<KV>::kMaxSlots ? W : DecCfg<KV>::kMaxSlots;
  if (W <= 64) {
    const int g = 2 * sms / B > 1 ? 2 * sms / B : 1;
    if (G > g) G = g;
  }
  return G < 1 ? 1 : G;
}

// Per device: the shared-memory opt-in, the SM count and the CTAs the
// balanced mode keeps resident (its grid), set up once.
template <int KV, bool SEL>
static cudaError_t decode_device_setup(int* dev_out, int* resident, int* sms) {
  static int resident_per_dev[kMaxDevices] = {0};
  static int sms_per_dev[kMaxDevices] = {0};
  constexpr int smem = dec_smem_bytes<KV, SEL>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (sms_per_dev[dev] == 0) {
    e = cudaFuncSetAttribute(decode_kernel<KV, SEL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<KV, SEL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int n_sm = 0, smem_sm = 0;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
        cudaSuccess)
      return e;
    // resident CTAs per SM from the shared-memory budget (1 KB of it is
    // reserved per CTA) and the launch bounds
    int per_sm = smem_sm / (smem + 1024);
    if (per_sm > kCtasPerSm) per_sm = kCtasPerSm;
    if (n_sm < 1) n_sm = 1;
    resident_per_dev[dev] = n_sm * (per_sm > 0 ? per_sm : 1);
    sms_per_dev[dev] = n_sm;
  }
  *dev_out = dev;
  *resident = resident_per_dev[dev];
  *sms = sms_per_dev[dev];
  return cudaSuccess;
}

template <int KV, bool SEL>
static cudaError_t launch_decode_t(const RowsParams& p, cudaStream_t stream) {
  int dev = 0, resident = 0, sms = 0;
  cudaError_t e = decode_device_setup<KV, SEL>(&dev, &resident, &sms);
  if (e != cudaSuccess) return e;
  CUtensorMap kmap, qmap;
  if (!encode_kcache_map(&kmap, p)) return cudaErrorInvalidValue;
  if (KV == DSA_KV_BF16) {
    if (!encode_q_map(&qmap, p, 64)) return cudaErrorInvalidValue;
  } else {
    memset(&qmap, 0, sizeof qmap);
  }
  const int balanced = decode_is_balanced(p.W, p.rows) ? 1 : 0;
  const int G = decode_slots<KV>(p.W, p.rows, sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = balanced ? dim3(resident, 1) : dim3(G, p.rows);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = dec_smem_bytes<KV, SEL>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // more CTAs than SMs: take the tensor memory early (see the kernel)
  const int early_tmem = (long long)cfg.gridDim.x * cfg.gridDim.y > sms ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_kernel<KV, SEL>, kmap, qmap, p, G, balanced, early_tmem);
}

// The balanced grid of the current device for keys of kv_dtype.
cudaError_t decode_balanced_ctas(int kv_dtype, int* ctas) {
  int dev = 0, sms = 0;
  if (kv_dtype == DSA_KV_FP8_E4M3)
    return decode_device_setup<DSA_KV_FP8_E4M3, true>(&dev, ctas, &sms);
  return decode_device_setup<DSA_KV_BF16, true>(&dev, ctas, &sms);
}

cudaError_t launch_decode(const RowsParams& p, cudaStream_t stream) {
  if (p.sel_k > 0) {
    if (p.kv_dtype == DSA_KV_FP8_E4M3) return launch_decode_t<DSA_KV_FP8_E4M3, true>(p, stream);
    return launch_decode_t<DSA_KV_BF16, true>(p, stream);
  }
  if (p.kv_dtype == DSA_KV_FP8_E4M3) return launch_decode_t<DSA_KV_FP8_E4M3, false>(p, stream);
  return launch_decode_t<DSA_KV_BF16, false>(p, stream);
}

}  // namespace dsa
