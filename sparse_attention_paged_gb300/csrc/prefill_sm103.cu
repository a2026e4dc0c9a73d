// prefill_sm103.cu -- prefill kernel of the DSA indexer paged MQA-logits for
// GB300 (sm_103a): n_q query tokens of one request share one block table;
// query i may see the positions below its length L_i (causal limit + 1).
//
// The keys are read page by page from the paged cache through TMA; no
// gathered [queries, pages, ...] copy is ever formed ("The Dispatch
// Decision: Wiring a Triton Kernel into Production", section "The Problem
// That Led Here": the materialised gather of a 22K-context, 4,096-query
// prefill is what ran out of memory).
//
// Work: items (query tile j of 4 queries, position tile of 128 positions),
// only for position tiles below the tile's largest length.  A persistent
// grid of one CTA per SM splits the item list evenly (a block-wide prefix
// sum over the per-tile lengths), so the causal triangle's skipped tiles cost
// nothing and every SM gets the same number of MMAs.
//
// Per item: tcgen05 MMA with M = 128 positions, N = 256 (4 queries x 64
// heads), K = 128, f32 accumulator in TMEM, double-buffered (2 x 256
// columns); 16 epilogue warps (four per TMEM lane quadrant, one query each)
// apply ReLU, the head weights (packed f32x2 FMAs) and the position scale and
// store one coalesced 128-byte row segment per warp.
//
// Keys in bf16: kind::f16, the query tile loaded by TMA.  Keys in fp8
// (e4m3): the stored codes are the A operand as they are (kind::f8f6f4, one
// 8 KB box per page); the query tile is split by the epilogue warps into two
// e4m3 terms (hi + lo) with a power-of-two scale per head, folded into the
// head weights, and both terms accumulate into the same TMEM columns.
#include <cuda.h>
#include <cuda_fp16.h>
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

constexpr int kQT = 4;                        // queries per tile (N = 256)
constexpr int kN = kQT * kHeads;              // 256
constexpr int kTileM = 128;                   // positions per tile
constexpr int kEpiWarps = 16;                 // 4 per TMEM lane quadrant, one query each
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = (kEpiWarps + 2) * 32;  // + TMA warp + MMA warp
constexpr int kBox = kPage * 128;             // 8 KB: one page's 64 rows of 128 bytes
constexpr int kBBytes = kN * kDim * 2;        // 64 KB: 2 x 256 rows x 128 B (bf16 K-blocks / e4m3 hi, lo)
constexpr int kCtrl = 10240;
constexpr int kCtrlReq = 4352;                // request map (tile0, row0) in the control block
constexpr int kCtrlWScan = kCtrlReq + 8 * (kMaxPrefillRequests + 1);   // [kThreads] long long
// The persistent split balances cost, not items: an item weighs 16, a query
// tile adds a fixed kTileChangeW (its query tile's load, weights and set-up:
// about two items) and 1/20 per 64-position page of its rows' tail, which
// the epilogue writes with -inf when it starts the tile.  CTAs on tiles of
// short contexts (frequent tile changes, long tails) so take fewer items.
// (Weights chosen by measurement among 0..64 per tile and 0..2/5 per page.)
#ifndef DSA_PF_TILE_W
#define DSA_PF_TILE_W 32
#endif
#ifndef DSA_PF_FILL_W_NUM
#define DSA_PF_FILL_W_NUM 1
#endif
#ifndef DSA_PF_FILL_W_DEN
#define DSA_PF_FILL_W_DEN 20
#endif
constexpr long long kTileChangeW = DSA_PF_TILE_W;
constexpr int kBtSmem = 4096;                 // block-table entries kept in shared memory
constexpr long long kWaitLimit = 2000000000ll;   // ~1 s of SM clock: bound on any wait

template <int KV>
struct PfCfg;
template <>
struct PfCfg<DSA_KV_BF16> {
  static constexpr int kStages = 4;
  static constexpr int kABytes = kTileM * kDim * 2;   // 32 KB: 2 K-blocks x 128 rows x 128 B
  static constexpr int kOps = 4;                      // boxes per item: page x K-block
};
template <>
struct PfCfg<DSA_KV_FP8_E4M3> {
  static constexpr int kStages = 8;
  static constexpr int kABytes = kTileM * kDim;       // 16 KB: 128 rows x 128 B
  static constexpr int kOps = 2;                      // boxes per item: one per page
};
template <int KV>
constexpr int pf_smem_bytes() {
  return 1024 + kBBytes + PfCfg<KV>::kStages * PfCfg<KV>::kABytes + kCtrl + 4 * kBtSmem;
}

__device__ __forceinline__ float nanf_() { return __int_as_float(0x7fc00000); }

// max(s, 0) * 2^-64 for |s| < 2^64, computed on the FMA pipe (a saturating
// multiply clamps to [0, 1]); the caller scales its weighted sum by 2^64.
__device__ __forceinline__ float relu_sat(float s) {
  float r;
  asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(r) : "f"(s), "f"(5.421010862427522e-20f));   // 2^-64
  return r;
}
constexpr float kTwo64 = 18446744073709551616.0f;   // 2^64

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Two floats to e4m3 (nearest-even, saturating): the two codes (first
// argument in the low byte) and their values.
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b, float& fa, float& fb) {
  __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(s, __NV_E4M3);
  fa = __half2float(__half(__half_raw{h.x}));
  fb = __half2float(__half(__half_raw{h.y}));
  return (uint32_t)s;
}

// A query tile: up to kQT consecutive query rows of one request, and the
// request's block-table row.
struct QTile {
  int row0;          // first query row
  int n;             // rows in the tile (1..kQT)
  const int* bt;     // the request's block-table row
  int req;           // the request (0 for a one-request call)
};

struct Lens {
  int T;
  int nq;
  int nqt;
  const int* seqlens;
  // several requests (n_req > 0): request b's query tiles are tiles
  // tile0[b] .. tile0[b+1]-1 and its rows row0[b] .. row0[b+1]-1, its table
  // row at bt + b * bt_stride; n_req = 0: one request, tile j = rows 4j..
  int n_req;
  const int* tile0;  // shared memory
  const int* row0;   // shared memory
  const int* bt;
  long long bt_stride;
  __device__ __forceinline__ QTile tile(int j) const {
    if (n_req == 0) return {kQT * j, min(kQT, nq - kQT * j), bt, 0};
    int lo = 0, hi = n_req - 1;          // the request holding tile j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile0[mid] <= j) lo = mid; else hi = mid - 1;
    }
    const int r0 = row0[lo] + kQT * (j - tile0[lo]);
    return {r0, min(kQT, row0[lo + 1] - r0), bt + (long long)lo * bt_stride, lo};
  }
  // length of query i clamped to [0, T]; an over-long row counts as 0 here
  // (it is written NaN by the fill)
  __device__ __forceinline__ int valid(int i) const {
    if (i >= nq) return 0;
    const int L = __ldg(seqlens + i);
    return (L > T) ? 0 : max(L, 0);
  }
  // largest valid length among the queries of query tile j
  __device__ __forceinline__ int lmax(int j) const {
    const QTile t = tile(j);
    int m = 0;
#pragma unroll
    for (int q = 0; q < kQT; ++q) m = max(m, q < t.n ? valid(t.row0 + q) : 0);
    return m;
  }
  __device__ __forceinline__ int tiles(int j) const { return (lmax(j) + kTileM - 1) / kTileM; }
};

// Walks a CTA's contiguous slice of the item list (query-tile major).
struct ItemIter {
  int j, pt, ntl, lmax;
  const Lens* lens;
  __device__ void init(const Lens* l, int j0, int pt0) {
    lens = l;
    j = j0;
    pt = pt0;
    lmax = l->lmax(j0);
    ntl = (lmax + kTileM - 1) / kTileM;
  }
  __device__ void next() {
    if (++pt < ntl) return;
    pt = 0;
    do {
      if (++j >= lens->nqt) {   // past the end of the list
        ntl = lmax = 0;
        return;
      }
      lmax = lens->lmax(j);
      ntl = (lmax + kTileM - 1) / kTileM;
    } while (ntl == 0);
  }
};

}  // namespace

template <int KV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                   const RowsParams p, const __grid_constant__ PrefillRequests rq) {
  constexpr int kStages = PfCfg<KV>::kStages;
  constexpr int kABytes = PfCfg<KV>::kABytes;
  constexpr bool kFp8 = KV == DSA_KV_FP8_E4M3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sA = smem + kBBytes;
  uint8_t* ctrl = sA + kStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;   // [2]
  uint64_t* tempty = tfull + 2;        // [2]
  uint64_t* bfull = tempty + 2;
  uint64_t* bempty = bfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 260);
  int* sm_misc = reinterpret_cast<int*>(ctrl + 272);       // total, start j, start pt
  int* scan = reinterpret_cast<int*>(ctrl + 2048);         // [kThreads]
  int* bt_s = reinterpret_cast<int*>(ctrl + kCtrl);        // [kBtSmem] the shared table row
  int* e_s = scan;                                          // fp8: [256] per-head exponents (after the split)
  int* rq_tile0 = reinterpret_cast<int*>(ctrl + kCtrlReq);  // [kMaxPrefillRequests + 1]
  int* rq_row0 = rq_tile0 + kMaxPrefillRequests + 1;        // [kMaxPrefillRequests + 1]
  static_assert((2 * kStages + 6) * 8 <= 256, "control block");
  static_assert(2048 + kThreads * 4 <= kCtrlReq, "control block");
  static_assert(kCtrlWScan + 8 * kThreads <= kCtrl && kCtrlWScan % 8 == 0, "control block");
  long long* wscan = reinterpret_cast<long long*>(ctrl + kCtrlWScan);   // [kThreads]
  long long* sm_wtot = reinterpret_cast<long long*>(ctrl + 304);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.W * kPage;
  const int n_qt = rq.n_req > 0 ? rq.tile0[rq.n_req] : (p.rows + kQT - 1) / kQT;
  for (int b = tid; b <= rq.n_req; b += kThreads) {   // the request map, to shared memory
    rq_tile0[b] = rq.tile0[b];
    rq_row0[b] = rq.row0[b];
  }
  const Lens lens{T, p.rows, n_qt, p.seqlens, rq.n_req, rq_tile0, rq_row0, p.block_table,
                  p.bt_stride};
  const int P = gridDim.x, k = blockIdx.x;
  const bool shared_row = rq.n_req == 0;   // one request: every query reads table row 0

  // nothing above reads the call's inputs; from here on they may have been
  // written by the previous launch in the stream
  griddep_wait();
  griddep_launch_dependents();

  // Page ids come from shared memory: one request's table row (its first
  // kBtSmem entries), or every request's row when they fit together (request
  // b's at b * W); else from each tile's own row (L1-cached loads).
  const bool all_rows = !shared_row && rq.n_req * p.W <= kBtSmem;
  if (shared_row) {
    for (int j = tid; j < min(p.W, kBtSmem); j += kThreads) bt_s[j] = __ldg(p.block_table + j);
  } else if (all_rows) {
    for (int j = tid; j < rq.n_req * p.W; j += kThreads) {
      const int b = j / p.W, e = j - b * p.W;
      bt_s[j] = __ldg(p.block_table + (long long)b * p.bt_stride + e);
    }
  }
  __syncthreads();
  auto page_id = [&](const QTile& tq, int page) {
    if (shared_row) return page < kBtSmem ? bt_s[page] : __ldg(tq.bt + page);
    return all_rows ? bt_s[tq.req * p.W + page] : __ldg(tq.bt + page);
  };

  // ---- fill: rows of query tiles without any position tile (every length
  // <= 0, or over-long rows) are written here; the other tiles' tails are
  // written by the CTA that owns their first item.
  for (int j = k; j < n_qt; j += P) {
    if (lens.tiles(j) != 0) continue;
    const QTile qt = lens.tile(j);
    for (int q = 0; q < qt.n; ++q) {
      const int i = qt.row0 + q;
      const bool bad = __ldg(p.seqlens + i) > T;
      const float fv = bad ? nanf_() : -INFINITY;
      float* orow = p.out + (long long)i * p.out_stride;
      for (int t = 4 * tid; t < T; t += 4 * kThreads)
        *reinterpret_cast<float4*>(orow + t) = make_float4(fv, fv, fv, fv);
      if (bad && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
    }
  }

  // ---- this CTA's slice of the item list: an equal share of the cost
  auto tile_weight = [&](int j, int nt) -> long long {
    if (nt == 0) return 0;
    const long long tail = (long long)lens.tile(j).n * max(p.W - 2 * nt, 0);
    return 16ll * nt + kTileChangeW + tail * DSA_PF_FILL_W_NUM / DSA_PF_FILL_W_DEN;
  };
  {
    const int j0 = (int)((long long)tid * n_qt / kThreads);
    const int j1 = (int)((long long)(tid + 1) * n_qt / kThreads);
    int part = 0;
    long long wpart = 0;
    for (int j = j0; j < j1; ++j) {
      const int nt = lens.tiles(j);
      part += nt;
      wpart += tile_weight(j, nt);
    }
    scan[tid] = part;
    wscan[tid] = wpart;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      long long wrun = 0;
      for (int i = 0; i < kThreads; ++i) {
        const int v = scan[i];
        const long long wv = wscan[i];
        scan[i] = run;
        wscan[i] = wrun;
        run += v;
        wrun += wv;
      }
      sm_misc[0] = run;
      sm_misc[1] = -1;
      sm_misc[6] = run;          // item bounds of this CTA (found below)
      sm_misc[7] = run;
      *sm_wtot = wrun;
    }
    __syncthreads();
    // this CTA's items: from the first item whose cost range starts at or
    // after k * TW / P up to the next CTA's first
    const long long TW = *sm_wtot;
    for (int e = 0; e < 2; ++e) {
      const long long x = (long long)(k + e) * TW / P;
      if (wpart > 0 && x >= wscan[tid] && x < wscan[tid] + wpart) {
        long long acc = wscan[tid];
        int ia = scan[tid];
        for (int j = j0; j < j1; ++j) {
          const int nt = lens.tiles(j);
          const long long wt = tile_weight(j, nt);
          if (x < acc + wt) {
            // item 0 covers [acc, acc + wt - 16 (nt - 1)), item pt > 0 the
            // 16 units after its predecessor
            const long long f = wt - 16ll * nt;
            int pt = 0;
            if (x > acc) pt = (int)min((long long)nt, max(1ll, (x - acc - f + 15) / 16));
            sm_misc[6 + e] = ia + pt;
            break;
          }
          acc += wt;
          ia += nt;
        }
      }
    }
    __syncthreads();
    const int start = sm_misc[6];
    if (part > 0 && start >= scan[tid] && start < scan[tid] + part) {
      int acc = scan[tid];
      for (int j = j0; j < j1; ++j) {
        const int n = lens.tiles(j);
        if (start < acc + n) {
          sm_misc[1] = j;
          sm_misc[2] = start - acc;
          break;
        }
        acc += n;
      }
    }
    __syncthreads();
  }
  const int n_items = sm_misc[7] - sm_misc[6];
  if (n_items <= 0) return;
  const int j_start = sm_misc[1], pt_start = sm_misc[2];

  if (tid == kEpiWarps * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps * 32);
    }
    mbar_init(bfull, kFp8 ? kEpiThreads : 1);    // fp8: the epilogue threads write B
    mbar_init(bempty, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kEpiWarps + 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kEpiWarps) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp walks the item list.  Lane 0 waits on and arms the
    // barriers; every copy of an item is issued by a lane of its own (a
    // little faster than one lane issuing all four).
    if (lane == 0) {
      prefetch_tmap(&kmap);
      if (!kFp8) prefetch_tmap(&qmap);
    }
    ItemIter it;
    it.init(&lens, j_start, pt_start);
    int nb = 0, issued = 0, cur_j = -1, tq_j = -1;
    QTile tq = {0, 0, p.block_table, 0};
    bool ok = true;
    for (int i = 0; i < n_items; ++i, it.next()) {
      if (it.j != tq_j) {             // the query tile's rows and table row
        tq = lens.tile(it.j);
        tq_j = it.j;
      }
      if (!kFp8 && it.j != cur_j) {   // new query tile: reload B once the MMA is done with it
        if (lane == 0) {
          if (nb > 0) ok = mbar_wait_bounded(bempty, (nb - 1) & 1, kWaitLimit);
          ok = ok && *abort_flag == 0;
          if (ok) mbar_arrive_expect_tx(bfull, kBBytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < 2)
          tma_load_2d(sB + lane * (kBBytes / 2), &qmap, bfull, lane * kHalfRowUnits,
                      tq.row0 * kHeads);
        cur_j = it.j;
        ++nb;
      }
      const int s = i % kStages;
      if (lane == 0) {
        if (i >= kStages) ok = mbar_wait_bounded(&empty[s], ((i / kStages) - 1) & 1, kWaitLimit);
        ok = ok && *abort_flag == 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // lane l < kOps: page (l & 1) of the tile; bf16: K-block (l >> 1)
      int phys = -1;
      if (lane < PfCfg<KV>::kOps) {
        const int page = 2 * it.pt + (lane & 1);
        if (page * kPage < it.lmax) {     // a page some query of the tile needs
          const int ph = page_id(tq, page);
          if (ph >= 0 && ph < p.num_pages) phys = ph;
        }
      }
      const unsigned have = __ballot_sync(0xffffffffu, phys >= 0);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], __popc(have) * kBox);
      __syncwarp();
      if (phys >= 0) {
        if (kFp8)
          tma_load_3d(sA + s * kABytes + lane * kBox, &kmap, &full[s], 0, 0, phys);
        else
          tma_load_3d(sA + s * kABytes + (lane >> 1) * (kABytes / 2) + (lane & 1) * kBox, &kmap,
                      &full[s], (lane >> 1) * kHalfRowUnits, 0, phys);
      }
      issued = i + 1;
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, DSA_ERR_TIMEOUT);
      }
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, kWaitLimit);
      if (nb > 0) mbar_wait_bounded(bfull, (nb - 1) & 1, kWaitLimit);
    }
  } else if (warp == kEpiWarps + 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = kFp8 ? instr_desc(0, 0, kTileM, kN) : instr_desc(1, 1, kTileM, kN);
      const uint32_t sAa = smem_u32(sA), sBa = smem_u32(sB);
      ItemIter it;
      it.init(&lens, j_start, pt_start);
      int nb = 0, issued = 0, cur_j = -1;
      bool ok = true;
      for (int i = 0; i < n_items; ++i) {
        const int s = i % kStages, a = i & 1;
        if (it.j != cur_j) {
          ok = mbar_wait_bounded(bfull, nb & 1, kWaitLimit);
          cur_j = it.j;
          ++nb;
        }
        if (ok) ok = mbar_wait_bounded(&full[s], (i / kStages) & 1, kWaitLimit);
        if (ok && i >= 2) ok = mbar_wait_bounded(&tempty[a], ((i >> 1) - 1) & 1, kWaitLimit);
        if (!ok || *abort_flag) break;
        tc_fence_after();
        const uint32_t d = tmem_base + a * kN;
        const uint32_t st = sAa + s * kABytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (kFp8) {
            // hi then lo term; K = 32 per MMA within the 128-byte rows
            const uint32_t term = kk >> 2, ko = (kk & 3) * 32;
            const uint64_t ad = smem_desc_sw128(st + ko, 1024);
            const uint64_t bd = smem_desc_sw128(sBa + term * (kBBytes / 2) + ko, 1024);
            mma_f8f6f4(d, ad, bd, idesc, kk != 0);
          } else {
            const uint32_t kb = kk >> 2, ko = (kk & 3) * 32;
            const uint64_t ad = smem_desc_sw128(st + kb * (kABytes / 2) + ko, 1024);
            const uint64_t bd = smem_desc_sw128(sBa + kb * (kBBytes / 2) + ko, 1024);
            mma_f16(d, ad, bd, idesc, kk != 0);
          }
        }
        mma_commit(&empty[s]);
        mma_commit(&tfull[a]);
        issued = i + 1;
        it.next();
        if (i + 1 == n_items || it.j != cur_j) mma_commit(bempty);   // B free after these MMAs
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, DSA_ERR_TIMEOUT);
      }
      if (issued > 0) {
        const int i = issued - 1;
        mbar_wait_bounded(&tfull[i & 1], (i >> 1) & 1, kWaitLimit);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int quad = warp & 3;                // TMEM lane quadrant
    const int qt = warp >> 2;                 // query of the tile this warp reduces
    // Accumulator reads use the 16x256b shape: thread (g = lane / 4,
    // c = lane % 4) sees rows g, g+8 (first read) and g+16, g+24 (second)
    // of the quadrant, always at heads 8j + 2c, 8j + 2c + 1 (j < 8), so its
    // 16 weights stay in registers for a whole query tile.  A reduce-scatter
    // over the four threads of a row group leaves thread lane with the full
    // sum of row g + 8 * (2 * (c & 1) + (c >> 1)).
    const int cq = lane & 3;
    const int r = quad * 32 + (lane >> 2) + 8 * (2 * (cq & 1) + (cq >> 1));
    // fp8: split query tile j into e4m3 hi + lo terms in B (row q*64 + h,
    // 128-byte swizzle; hi at +0, lo at +32 KB) with a power-of-two scale
    // 2^e per head (the head's largest |q| lands in [128, 256)), e in e_s.
    // Threads 2t and 2t+1 take row t, 64 values each.
    auto split_queries = [&](const QTile& tq) {
      const int row = tid >> 1, half = tid & 1;
      const int qi = tq.row0 + (row >> 6);
      const bool live = (row >> 6) < tq.n;
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + ((long long)(live ? qi : 0) * kHeads + (row & 63)) * kDim + half * 64);
      // pass 1: the head's largest |q| (as float bits: non-negative floats
      // order as integers); pass 2 below re-reads the same 128 bytes (L1)
      uint32_t mb = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)      // a bf16 pair: low value in bits 0-15
          mb = max(mb, max((w4[u] << 17) >> 1, (w4[u] >> 16 << 17) >> 1));
      }
      float m = __uint_as_float(mb);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      int e = 0;
      if (m > 0.f) {
        const int E = ((__float_as_int(m) >> 23) & 0xff) - 127;   // floor(log2 m), m normal
        e = min(max(7 - E, -126), 126);
      }
      const float sc = exp2i(e);
      if (half == 0) e_s[row] = e;
      uint8_t* hb = sB + row * 128;
      uint8_t* lb = sB + kBBytes / 2 + row * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {           // 16 values = one 16-byte chunk of each term
        const uint4 v0 = live ? __ldg(src + 2 * cc) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 v1 = live ? __ldg(src + 2 * cc + 1) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t src8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float a0 = __uint_as_float(src8[u] << 16) * sc;
          const float a1 = __uint_as_float(src8[u] & 0xffff0000u) * sc;
          float h0, h1, l0, l1;
          const uint32_t hc = to_e4m3x2(a0, a1, h0, h1);
          const uint32_t lc = to_e4m3x2(a0 - h0, a1 - h1, l0, l1);
          hi[u >> 1] |= hc << (16 * (u & 1));
          lo[u >> 1] |= lc << (16 * (u & 1));
        }
        const int phys_chunk = (half * 4 + cc) ^ (row & 7);
        *reinterpret_cast<uint4*>(hb + phys_chunk * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(lb + phys_chunk * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bfull);
    };
    ItemIter it;
    it.init(&lens, j_start, pt_start);
    int cur_j = -1;
    QTile tqe = {0, 0, p.block_table, 0};
    int Lq = 0, Lmax = 0;
    float2 wreg[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) wreg[j] = make_float2(0.f, 0.f);
    bool badq = false;
    bool ok = true;
    int nb = 0;           // fp8: query tiles split so far
    for (int i = 0; i < n_items; ++i, it.next()) {
      const int a = i & 1;
      if (it.j != cur_j) {
        cur_j = it.j;
        tqe = lens.tile(cur_j);
        if (kFp8) {
          // every thread is past its reads of the previous e_s; the MMA is
          // done with the previous B (its last accumulator has been read)
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
          if (nb > 0 && ok) ok = mbar_wait_bounded(bempty, (nb - 1) & 1, kWaitLimit);
          ++nb;
          split_queries(tqe);
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
        }
        const int qi = tqe.row0 + qt;
        if (qt < tqe.n) {
          const float* wr = p.w + (long long)qi * kHeads + 2 * cq;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            wreg[j] = make_float2(__ldg(wr + 8 * j), __ldg(wr + 8 * j + 1));
            if (kFp8) {     // undo the split's per-head scale
              wreg[j].x *= exp2i(-e_s[qt * kHeads + 8 * j + 2 * cq]);
              wreg[j].y *= exp2i(-e_s[qt * kHeads + 8 * j + 2 * cq + 1]);
            }
          }
        }
        const int L = qt < tqe.n ? __ldg(p.seqlens + qi) : 0;
        badq = L > T;
        Lq = badq ? 0 : max(L, 0);
        Lmax = it.lmax;
        // the tail of this query tile past its last position tile
        if (it.pt == 0) {
          const int f0 = it.ntl * kTileM;
          for (int q = 0; q < tqe.n; ++q) {
            const int qf = tqe.row0 + q;
            const bool bad = __ldg(p.seqlens + qf) > T;
            const float fv = bad ? nanf_() : -INFINITY;
            float* orow = p.out + (long long)qf * p.out_stride;
            for (int t = f0 + 4 * tid; t < T; t += 4 * kEpiThreads)
              *reinterpret_cast<float4*>(orow + t) = make_float4(fv, fv, fv, fv);
            if (bad && tid == 0) raise_status(p.status, DSA_ERR_BAD_SEQLEN);
          }
        }
      }
      const int t = it.pt * kTileM + r;
      const int page = t / kPage, slot = t % kPage;
      const bool in_table = t < T;
      int phys = -1;
      float scale = 1.f;
      if (in_table && t < Lmax) {
        phys = page_id(tqe, page);
        if (phys >= 0 && phys < p.num_pages && p.kscale != nullptr)
          scale = __ldg(reinterpret_cast<const float*>(p.kscale + (long long)phys * p.page_stride) +
                        slot);
      }
      if (ok) ok = mbar_wait_bounded(&tfull[a], (i >> 1) & 1, kWaitLimit);
      ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);
      float res = 0.f;
      if (ok) {
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + a * kN + qt * kHeads;
        float part[4];      // this thread's 16 heads of rows g, g+8, g+16, g+24
        // four quarters (lane half x repeats 0-3 / 4-7), each load in flight
        // while the quarter before it is summed
        uint32_t v[2][16];
        tmem_ld_16x256b_x4(taddr, v[0]);
        tmem_ld_wait(v[0]);
        float2 f0 = make_float2(0.f, 0.f), f1 = f0, s0 = f0, s1 = f0;
#pragma unroll
        for (int qr = 0; qr < 4; ++qr) {
          const int half = qr >> 1, rep0 = (qr & 1) * 4, cb = qr & 1;
          if (qr < 3) {
            const int nh = (qr + 1) >> 1, nr = ((qr + 1) & 1) * 4;
            tmem_ld_16x256b_x4(taddr + ((uint32_t)(16 * nh) << 16) + 8 * nr, v[cb ^ 1]);
          }
          // ReLU split over two pipes: even repeats by fmax (ALU pipe), odd
          // ones by sat(s * 2^-64) (FMA pipe) in their own sums, scaled back
          // by 2^64.
#pragma unroll
          for (int j = 0; j < 4; j += 2) {
            const uint32_t* u = v[cb];
            f0 = __ffma2_rn(wreg[rep0 + j], make_float2(fmaxf(__uint_as_float(u[4 * j]), 0.f),
                                                        fmaxf(__uint_as_float(u[4 * j + 1]), 0.f)), f0);
            f1 = __ffma2_rn(wreg[rep0 + j], make_float2(fmaxf(__uint_as_float(u[4 * j + 2]), 0.f),
                                                        fmaxf(__uint_as_float(u[4 * j + 3]), 0.f)), f1);
            s0 = __ffma2_rn(wreg[rep0 + j + 1], make_float2(relu_sat(__uint_as_float(u[4 * j + 4])),
                                                            relu_sat(__uint_as_float(u[4 * j + 5]))), s0);
            s1 = __ffma2_rn(wreg[rep0 + j + 1], make_float2(relu_sat(__uint_as_float(u[4 * j + 6])),
                                                            relu_sat(__uint_as_float(u[4 * j + 7]))), s1);
          }
          if (qr < 3) tmem_ld_wait(v[cb ^ 1]);
          if (qr == 2) {
            // every column is in registers: the accumulator buffer is free
            tc_fence_before();
            mbar_arrive(&tempty[a]);
          }
          if (qr & 1) {
            part[2 * half] = (f0.x + f0.y) + kTwo64 * (s0.x + s0.y);
            part[2 * half + 1] = (f1.x + f1.y) + kTwo64 * (s1.x + s1.y);
            f0 = f1 = s0 = s1 = make_float2(0.f, 0.f);
          }
        }
        // reduce-scatter over c: bit 0 picks rows {g+16, g+24} or {g, g+8},
        // bit 1 the second or first of the pair
        const bool b0 = cq & 1, b1 = cq & 2;
        const float ra = __shfl_xor_sync(0xffffffffu, b0 ? part[0] : part[2], 1);
        const float rb = __shfl_xor_sync(0xffffffffu, b0 ? part[1] : part[3], 1);
        const float k0 = (b0 ? part[2] : part[0]) + ra;
        const float k1 = (b0 ? part[3] : part[1]) + rb;
        res = (b1 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
      }
      const int qi = tqe.row0 + qt;
      if (in_table && qt < tqe.n) {
        float o;
        if (badq) {
          o = nanf_();
        } else if (t >= Lq) {
          o = -INFINITY;
        } else if (!ok || phys < 0 || phys >= p.num_pages) {
          o = nanf_();
          if (ok) raise_status(p.status, DSA_ERR_BAD_PAGE);
        } else {
          o = scale * res;
        }
        p.out[(long long)qi * p.out_stride + t] = o;
      }
    }
    if (!ok) raise_status(p.status, DSA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kEpiWarps + 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int KV>
static cudaError_t launch_prefill_t(const RowsParams& p, const PrefillRequests& rq,
                                    cudaStream_t stream) {
  // per device: the shared-memory opt-in and the SM count (one CTA per SM)
  static int sms_per_dev[kMaxDevices] = {0};
  constexpr int smem = pf_smem_bytes<KV>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (sms_per_dev[dev] == 0) {
    e = cudaFuncSetAttribute(prefill_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_kernel<KV>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    sms_per_dev[dev] = sms > 0 ? sms : 1;
  }
  CUtensorMap kmap, qmap;
  if (!encode_kcache_map(&kmap, p)) return cudaErrorInvalidValue;
  if (KV == DSA_KV_BF16) {
    if (!encode_q_map(&qmap, p, kN)) return cudaErrorInvalidValue;
  } else {
    memset(&qmap, 0, sizeof qmap);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms_per_dev[dev]);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<KV>, kmap, qmap, p, rq);
}

cudaError_t launch_prefill(const RowsParams& p, const PrefillRequests& rq, cudaStream_t stream) {
  if (p.kv_dtype == DSA_KV_FP8_E4M3) return launch_prefill_t<DSA_KV_FP8_E4M3>(p, rq, stream);
  return launch_prefill_t<DSA_KV_BF16>(p, rq, stream);
}

}  // namespace dsa
