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
//    (request, page) pairs of all rows, in row order, are split into equal
//    contiguous slices (prefix sums of the rows' valid page counts, computed
//    by every CTA), and the positions past each length are split the same
//    way.  No CTA is the tail of a long request.  A slice can cross rows; the
//    query operand is double-buffered per row segment.
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
// per head: q * 2^e_h = hi + lo, hi = e4m3(q * 2^e_h), lo = e4m3(q * 2^e_h -
// hi), with 2^e_h folded into the head weight.  hi + lo reproduces every
// bf16 value whose magnitude is at least ~2^-10 of its head's maximum
// exactly, and the rest to within 2^-18 of the head's maximum.
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
#define DSA_DEC_FP8_STAGES 4
#endif
#ifndef DSA_DEC_BF16_STAGES
#define DSA_DEC_BF16_STAGES 2
#endif
#ifndef DSA_DEC_CTAS
#define DSA_DEC_CTAS 2
#endif
#ifndef DSA_DEC_SMALL_PER_SM
#define DSA_DEC_SMALL_PER_SM 1
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

template <int KV>
constexpr int dec_smem_bytes() {
  using C = DecCfg<KV>;
  return 1024 /* alignment slack */ + 2 * C::kQBytes + C::kStages * C::kTileBytes + kCtrlBytes;
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

}  // namespace

template <int KV>
__global__ void __launch_bounds__(kDecThreads, kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const RowsParams p, const int G, const int balanced) {
  using C = DecCfg<KV>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // 2 x B operand (row segments alternate)
  uint8_t* sA = smem + 2 * C::kQBytes;         // A stages
  uint8_t* ctrl = sA + S * C::kTileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;                 // [2] accumulator ready
  uint64_t* tempty = tfull + 2;                // [2] accumulator drained
  uint64_t* qbar = tempty + 2;                 // [2] query operand ready
  uint64_t* bempty = qbar + 2;                 // [2] query operand no longer read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 260);
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
    fence_barrier_init();
    prefetch_tmap(&kmap);
    if (KV == DSA_KV_BF16) prefetch_tmap(&qmap);
  }
  griddep_wait();
  griddep_launch_dependents();

  Tiles tiles;
  if (!balanced) {
    // ---------------------------------------------------------------- per-request
    const int b = blockIdx.y, c = blockIdx.x;
    const int L = __ldg(p.seqlens + b);
    const int npv = valid_pages(L, p.W);
    const int n_mine = npv > c ? (npv - 1 - c) / G + 1 : 0;
    if (tid < 128 || n_mine == 0) {
      // -inf (NaN for an over-long row) past the last valid page, split over
      // the row's G CTAs in contiguous 16-byte-aligned chunks
      const bool bad = L > T;
      const int f0 = npv * kPage;
      int chunk = (T - f0 + G - 1) / G;
      chunk = (chunk + 3) & ~3;
      const long long beg = f0 + (long long)c * chunk;
      const long long end = p.fill ? min(beg + chunk, (long long)T) : beg;
      const float fv = bad ? nanf_() : -INFINITY;
      const float4 v4 = make_float4(fv, fv, fv, fv);
      const int nthr = n_mine == 0 ? kDecThreads : 128;
      float* orow = p.out + (long long)b * p.out_stride;
      for (long long i = beg + 4 * tid; i < end; i += 4 * nthr)
        __stcs(reinterpret_cast<float4*>(orow + i), v4);
      if (bad && c == 0 && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
    }
    if (n_mine == 0) return;
    if (tid == 0) lens_s[0] = L;
    tiles.init_request(G, c, b, n_mine);
  } else {
    // ---------------------------------------------------------------- balanced
    const int B = p.rows;
    for (int j = tid; j < B; j += kDecThreads) lens_s[j] = __ldg(p.seqlens + j);
    __syncthreads();
    if (warp == 0) {
      // exclusive prefix sums of valid pages and of fill pages (W - valid)
      int run_v = 0, run_f = 0;
      for (int base = 0; base < B; base += 32) {
        const int j = base + lane;
        const int v = j < B ? valid_pages(lens_s[j], p.W) : 0;
        const int f = j < B ? p.W - v : 0;
        int sv = v, sf = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int tv = __shfl_up_sync(0xffffffffu, sv, o);
          const int tf = __shfl_up_sync(0xffffffffu, sf, o);
          if (lane >= o) {
            sv += tv;
            sf += tf;
          }
        }
        if (j < B) {
          Pv[j] = run_v + sv - v;
          Pf[j] = run_f + sf - f;
        }
        run_v += __shfl_sync(0xffffffffu, sv, 31);
        run_f += __shfl_sync(0xffffffffu, sf, 31);
      }
      if (lane == 0) {
        Pv[B] = run_v;
        Pf[B] = run_f;
      }
    }
    __syncthreads();
    const long long R = gridDim.x, k = blockIdx.x;
    const long long N = Pv[B], F = p.fill ? Pf[B] : 0;
    const int u0 = (int)(k * N / R), u1 = (int)((k + 1) * N / R);
    const int f0 = (int)(k * F / R), f1 = (int)((k + 1) * F / R);

    // this CTA's share of the fill: fill pages [f0, f1) in row order; fill
    // page i of row r is page valid_pages(L_r) + i of that row
    if (f0 < f1 && (tid < 128 || u0 >= u1)) {
      const int nthr = u0 >= u1 ? kDecThreads : 128;
      int lo = 0, hi = B - 1;
      while (lo < hi) {      // row holding fill page f0
        const int mid = (lo + hi + 1) >> 1;
        if (Pf[mid] <= f0) lo = mid; else hi = mid - 1;
      }
      for (int r = lo, f = f0; f < f1 && r < B; ++r) {
        const int nf = Pf[r + 1] - Pf[r];
        if (nf == 0) continue;
        const int a = f - Pf[r];                       // first fill page of row r in range
        const int e = min(f1 - Pf[r], nf);             // one past the last
        const int L = lens_s[r];
        const bool bad = L > T;
        const int first_page = p.W - nf;               // = valid pages of row r
        const float fv = bad ? nanf_() : -INFINITY;
        const float4 v4 = make_float4(fv, fv, fv, fv);
        float* orow = p.out + (long long)r * p.out_stride;
        const long long beg = (long long)(first_page + a) * kPage;
        const long long end = (long long)(first_page + e) * kPage;
        for (long long i = beg + 4 * tid; i < end; i += 4 * nthr)
          __stcs(reinterpret_cast<float4*>(orow + i), v4);
        if (bad && a == 0 && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
        f = Pf[r] + e;
      }
    }
    if (u0 >= u1) return;
    tiles.init_balanced(Pv, B, u0, u1);
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
      Tiles it = tiles;
      int issued = 0, seg_loaded = -1;
      bool ok = true;
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
            const int ph = __ldg(btrow + pg);
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
      }
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
          // A: 128 rows x 128 B; B: hi then lo, 64 rows x 128 B each; K = 32 per MMA
#pragma unroll
          for (int term = 0; term < 2; ++term) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(st + 32 * k, 1024);
              const uint64_t bd = smem_desc_sw128(bq + term * 8192 + 32 * k, 1024);
              mma_f8f6f4(d, ad, bd, idesc, (term | k) != 0);
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
      float* ws = w_s + sb * kHeads;
      if (KV == DSA_KV_FP8_E4M3) {
        const uint16_t* qrow = p.q + (long long)r * kHeads * kDim;
        uint2 qraw[16];
#pragma unroll
        for (int hh = 0; hh < 16; ++hh)
          qraw[hh] = __ldg(reinterpret_cast<const uint2*>(qrow + (warp * 16 + hh) * kDim) + lane);
        const float wv = lane < 16 ? __ldg(p.w + (long long)r * kHeads + warp * 16 + lane) : 0.f;
        uint8_t* qb = sQ + sb * C::kQBytes;
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
          *reinterpret_cast<uint32_t*>(qb + off) = hi;
          *reinterpret_cast<uint32_t*>(qb + 8192 + off) = lo;
          const float wh = __shfl_sync(0xffffffffu, wv, hh);
          if (lane == 0) ws[h] = wh * exp2i(-e);
        }
        fence_proxy_async_smem();
        mbar_arrive(&qbar[sb]);
      } else {
        if (tid < kHeads) ws[tid] = __ldg(p.w + (long long)r * kHeads + tid);
      }
    };

    bool ok = true;
    // segments 0 and 1 use fresh buffers
    prepare(tiles.row, 0);
    const int r1 = tiles.next_segment_row();
    if (r1 >= 0) prepare(r1, 1);
    asm volatile("bar.sync 1, 128;" ::: "memory");

    const int r = warp * 32 + lane;            // accumulator row = TMEM lane
    const int half = r >> 6, slot = r & 63;
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
      const float* ws = w_s + (cur_seg & 1) * kHeads;
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
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

// CTAs per request in per-request mode, from the launch shape only: at most
// the per-dtype cap and W; for a short table (W <= 64 pages, so no request is
// long) about DSA_DEC_SMALL_PER_SM CTAs per SM in total, so that each CTA
// pipelines a few pages instead of paying its start-up latency for one.
template <int KV>
int decode_slots(int W, int B, int sms) {
  int G = W < DecCfg<KV>::kMaxSlots ? W : DecCfg<KV>::kMaxSlots;
  const long long budget = (long long)sms * DSA_DEC_SMALL_PER_SM;
  if (W <= 64 && (long long)B * G > budget) G = (int)(budget / B);
  return G < 1 ? 1 : G;
}

template <int KV>
static cudaError_t launch_decode_t(const RowsParams& p, cudaStream_t stream) {
  // per device: the shared-memory opt-in, the SM count and the resident CTAs
  static int resident_per_dev[kMaxDevices] = {0};
  static int sms_per_dev[kMaxDevices] = {0};
  constexpr int smem = dec_smem_bytes<KV>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (sms_per_dev[dev] == 0) {
    e = cudaFuncSetAttribute(decode_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<KV>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int sms = 0, smem_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
        cudaSuccess)
      return e;
    // resident CTAs per SM from the shared-memory budget (1 KB of it is
    // reserved per CTA) and the launch bounds
    int per_sm = smem_sm / (smem + 1024);
    if (per_sm > kCtasPerSm) per_sm = kCtasPerSm;
    if (sms < 1) sms = 1;
    resident_per_dev[dev] = sms * (per_sm > 0 ? per_sm : 1);
    sms_per_dev[dev] = sms;
  }
  CUtensorMap kmap, qmap;
  if (!encode_kcache_map(&kmap, p)) return cudaErrorInvalidValue;
  if (KV == DSA_KV_BF16) {
    if (!encode_q_map(&qmap, p, 64)) return cudaErrorInvalidValue;
  } else {
    memset(&qmap, 0, sizeof qmap);
  }
  const int balanced = (p.W > 64 && p.rows <= kMaxRowsBalanced) ? 1 : 0;
  const int G = decode_slots<KV>(p.W, p.rows, sms_per_dev[dev]);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = balanced ? dim3(resident_per_dev[dev], 1) : dim3(G, p.rows);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<KV>, kmap, qmap, p, G, balanced);
}

cudaError_t launch_decode(const RowsParams& p, cudaStream_t stream) {
  if (p.kv_dtype == DSA_KV_FP8_E4M3) return launch_decode_t<DSA_KV_FP8_E4M3>(p, stream);
  return launch_decode_t<DSA_KV_BF16>(p, stream);
}

}  // namespace dsa
