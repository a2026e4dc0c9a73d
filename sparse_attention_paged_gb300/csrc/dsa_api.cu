// dsa_api.cu -- the C ABI declared in include/dsa_indexer.h: argument
// checks, parameter packing and the single kernel launch of each call.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_common.cuh"
#include "dsa_indexer.h"
#include "topk_slots.cuh"

namespace dsa {
cudaError_t launch_decode(const RowsParams& p, cudaStream_t stream);
cudaError_t launch_prefill(const RowsParams& p, const PrefillRequests& rq, cudaStream_t stream);
cudaError_t launch_topk(const float* logits, long long ld, const int* seqlens, int rows, int T,
                        int k, int* idx, float* vals, long long out_stride, int* status,
                        cudaStream_t stream);
cudaError_t launch_topk_merge(const float* ws, const int* seqlens, int rows, int T, int k,
                              int* idx, float* vals, long long out_stride, int* status,
                              cudaStream_t stream);
bool decode_is_balanced(int W, int rows);
cudaError_t decode_balanced_ctas(int kv_dtype, int* ctas);
long long static_scratch_floats();
cudaError_t static_scratch(float** ptr);
cudaError_t launch_store(const uint16_t* k, const int* slots, int n, uint8_t* kcache,
                         long long page_stride, int num_pages, int kv_dtype, int* status,
                         cudaStream_t stream);
}

namespace {

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Host-side checks shared by both entry points.  Returns DSA_OK and fills
// `p`, or an error code (nothing is launched on error).
int check_and_pack(const void* q, const float* w, const void* kcache,
                   const void* kscale, long long page_stride, int num_pages,
                   int kv_dtype, const int* block_table, long long bt_stride,
                   const int* seqlens, int rows, int H, int D, int page_size,
                   int W, float* out, long long out_stride, int* dev_status,
                   dsa::RowsParams* p) {
  if (rows < 0 || W <= 0) return DSA_ERR_INVALID_ARG;
  if (H != dsa::kHeads || D != dsa::kDim || page_size != dsa::kPage)
    return DSA_ERR_UNSUPPORTED;
  if (kv_dtype != DSA_KV_FP8_E4M3 && kv_dtype != DSA_KV_BF16)
    return DSA_ERR_INVALID_ARG;
  if (rows > 0 && (!q || !w || !kcache || !block_table || !seqlens || !out))
    return DSA_ERR_INVALID_ARG;
  if (num_pages <= 0) return DSA_ERR_INVALID_ARG;
  const long long key_bytes =
      (long long)dsa::kPage * dsa::kDim * (kv_dtype == DSA_KV_BF16 ? 2 : 1);
  if (page_stride < key_bytes) return DSA_ERR_INVALID_ARG;
  if (bt_stride != 0 && bt_stride < W) return DSA_ERR_INVALID_ARG;
  if (bt_stride < 0) return DSA_ERR_INVALID_ARG;
  if (out_stride < (long long)W * dsa::kPage) return DSA_ERR_INVALID_ARG;
  if (page_stride % 16 != 0 || out_stride % 4 != 0) return DSA_ERR_MISALIGNED;
  if (!aligned(q, 16) || !aligned(kcache, 16) || !aligned(out, 16) ||
      !aligned(w, 4) || !aligned(block_table, 4) || !aligned(seqlens, 4))
    return DSA_ERR_MISALIGNED;
  if (kscale && !aligned(kscale, 16)) return DSA_ERR_MISALIGNED;

  p->q = static_cast<const uint16_t*>(q);
  p->w = w;
  p->kcache = static_cast<const uint8_t*>(kcache);
  p->kscale = static_cast<const uint8_t*>(kscale);
  p->page_stride = page_stride;
  p->num_pages = num_pages;
  p->kv_dtype = kv_dtype;
  p->block_table = block_table;
  p->bt_stride = bt_stride;
  p->seqlens = seqlens;
  p->rows = rows;
  p->W = W;
  p->out = out;
  p->out_stride = out_stride;
  p->status = dev_status;
  p->fill = 1;
  p->sel_k = 0;
  p->sel_ws = nullptr;
  return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_indexer_logits_decode(const void* q, const float* w,
                              const void* kcache, const void* kscale,
                              long long page_stride_bytes, int num_pages,
                              int kv_dtype, const int* block_table,
                              long long bt_stride, const int* seqlens, int B,
                              int H, int D, int page_size, int W, float* out,
                              long long out_stride, int* dev_status,
                              void* stream) {
  dsa::RowsParams p;
  int st = check_and_pack(q, w, kcache, kscale, page_stride_bytes, num_pages,
                          kv_dtype, block_table, bt_stride, seqlens, B, H, D,
                          page_size, W, out, out_stride, dev_status, &p);
  if (st != DSA_OK) return st;
  if (B == 0) return DSA_OK;
  if (B > 65535) return DSA_ERR_UNSUPPORTED;
  cudaError_t e = dsa::launch_decode(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_indexer_logits_prefill(const void* q, const float* w,
                               const void* kcache, const void* kscale,
                               long long page_stride_bytes, int num_pages,
                               int kv_dtype, const int* block_table,
                               long long bt_stride, const int* seqlens,
                               int n_q, int H, int D, int page_size, int W,
                               float* out, long long out_stride,
                               int* dev_status, void* stream) {
  dsa::RowsParams p;
  int st = check_and_pack(q, w, kcache, kscale, page_stride_bytes, num_pages,
                          kv_dtype, block_table, bt_stride, seqlens, n_q, H, D,
                          page_size, W, out, out_stride, dev_status, &p);
  if (st != DSA_OK) return st;
  if (n_q == 0) return DSA_OK;
  cudaError_t e;
  if (bt_stride == 0) {
    // one request's queries over one shared table: the query-tile kernel
    dsa::PrefillRequests one;
    one.n_req = 0;
    e = dsa::launch_prefill(p, one, static_cast<cudaStream_t>(stream));
  } else {
    // per-query table rows (several requests, multi-token decode): every
    // query token is a row of the decode kernel, with its own table row,
    // length and query
    if (n_q > 65535) return DSA_ERR_UNSUPPORTED;
    e = dsa::launch_decode(p, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_indexer_logits_prefill_varlen(const void* q, const float* w, const void* kcache,
                                      const void* kscale, long long page_stride_bytes,
                                      int num_pages, int kv_dtype, const int* block_table,
                                      long long bt_stride, const int* cu_q, int n_req,
                                      const int* seqlens, int H, int D, int page_size, int W,
                                      float* out, long long out_stride, int* dev_status,
                                      void* stream) {
  // the request boundaries are host data: checked here, before any launch
  if (n_req < 0 || (n_req > 0 && cu_q == nullptr)) return DSA_ERR_INVALID_ARG;
  if (n_req > 0 && cu_q[0] != 0) return DSA_ERR_INVALID_ARG;
  for (int b = 0; b < n_req; ++b)
    if (cu_q[b + 1] < cu_q[b]) return DSA_ERR_INVALID_ARG;
  const int n_q = n_req > 0 ? cu_q[n_req] : 0;
  dsa::RowsParams p;
  int st = check_and_pack(q, w, kcache, kscale, page_stride_bytes, num_pages, kv_dtype,
                          block_table, bt_stride, seqlens, n_q, H, D, page_size, W, out,
                          out_stride, dev_status, &p);
  if (st != DSA_OK) return st;
  // the query-tile kernel over up to kMaxPrefillRequests requests per launch
  // (one launch for most calls): each request's query tiles read its own
  // table row
  static_assert(sizeof(dsa::PrefillRequests) <= 2048, "request map fits the kernel parameters");
  for (int b0 = 0; b0 < n_req; b0 += dsa::kMaxPrefillRequests) {
    const int nb = n_req - b0 < dsa::kMaxPrefillRequests ? n_req - b0 : dsa::kMaxPrefillRequests;
    const int a = cu_q[b0], rows = cu_q[b0 + nb] - a;
    if (rows == 0) continue;
    dsa::PrefillRequests rq;
    rq.n_req = nb;
    int tiles = 0;
    for (int b = 0; b < nb; ++b) {
      rq.tile0[b] = tiles;
      rq.row0[b] = cu_q[b0 + b] - a;
      tiles += (cu_q[b0 + b + 1] - cu_q[b0 + b] + 3) / 4;
    }
    rq.tile0[nb] = tiles;
    rq.row0[nb] = rows;
    dsa::RowsParams pb = p;
    pb.q = p.q + (long long)a * dsa::kHeads * dsa::kDim;
    pb.w = p.w + (long long)a * dsa::kHeads;
    pb.seqlens = p.seqlens + a;
    pb.out = p.out + (long long)a * p.out_stride;
    pb.block_table = p.block_table + (long long)b0 * bt_stride;
    pb.bt_stride = bt_stride;
    pb.rows = rows;
    if (dsa::launch_prefill(pb, rq, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

int dsa_indexer_topk_decode_form(const void* q, const float* w, const void* kcache,
                                 const void* kscale, long long page_stride_bytes, int num_pages,
                                 int kv_dtype, const int* block_table, long long bt_stride,
                                 const int* seqlens, int B, int H, int D, int page_size, int W,
                                 int k_top, int* topk_idx, float* topk_val, long long topk_stride,
                                 float* workspace, long long workspace_floats, int* dev_status,
                                 int form, void* stream) {
  dsa::RowsParams p;
  const long long T = (long long)W * dsa::kPage;
  int st = check_and_pack(q, w, kcache, kscale, page_stride_bytes, num_pages, kv_dtype,
                          block_table, bt_stride, seqlens, B, H, D, page_size, W, workspace, T,
                          dev_status, &p);
  if (st != DSA_OK) return st;
  if (k_top < 1 || !topk_idx || topk_stride < k_top) return DSA_ERR_INVALID_ARG;
  if (form != DSA_TOPK_AUTO && form != DSA_TOPK_TWO_PASS && form != DSA_TOPK_FUSED)
    return DSA_ERR_INVALID_ARG;
  if (B > 0 && workspace_floats < (long long)B * T) return DSA_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || (topk_val && !aligned(topk_val, 4))) return DSA_ERR_MISALIGNED;
  if (B == 0) return DSA_OK;
  if (B > 65535) return DSA_ERR_UNSUPPORTED;
  p.fill = 0;      // the selection reads only t < L
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the fused form (on request only: the two-pass form measured faster on
  // every batch tried): the balanced decode, k small enough that a chunk
  // keeps at most half of its positions, and the slots within the workspace
  bool fused = false;
  if (form == DSA_TOPK_FUSED && k_top <= dsa::kSelMaxK && dsa::decode_is_balanced(W, B)) {
    int ctas = 0;
    if (dsa::decode_balanced_ctas(kv_dtype, &ctas) != cudaSuccess) return DSA_ERR_CUDA;
    const long long slots = (long long)ctas + B + ((long long)B * W + dsa::kSelChunkPages - 1) /
                                                       dsa::kSelChunkPages;
    fused = dsa::sel_header_floats(B) + slots * dsa::sel_slot_floats(k_top) <= workspace_floats;
  }
  if (form == DSA_TOPK_FUSED && !fused) return DSA_ERR_UNSUPPORTED;
  cudaError_t e;
  if (fused) {
    p.sel_k = k_top;
    p.sel_ws = workspace;
    e = dsa::launch_decode(p, s);
    if (e == cudaSuccess)
      e = dsa::launch_topk_merge(workspace, seqlens, B, (int)T, k_top, topk_idx, topk_val,
                                 topk_stride, dev_status, s);
  } else {
    e = dsa::launch_decode(p, s);
    if (e == cudaSuccess)
      e = dsa::launch_topk(workspace, T, seqlens, B, (int)T, k_top, topk_idx, topk_val,
                           topk_stride, dev_status, s);
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_indexer_topk_decode(const void* q, const float* w, const void* kcache,
                            const void* kscale, long long page_stride_bytes, int num_pages,
                            int kv_dtype, const int* block_table, long long bt_stride,
                            const int* seqlens, int B, int H, int D, int page_size, int W,
                            int k_top, int* topk_idx, float* topk_val, long long topk_stride,
                            float* workspace, long long workspace_floats, int* dev_status,
                            void* stream) {
  return dsa_indexer_topk_decode_form(q, w, kcache, kscale, page_stride_bytes, num_pages,
                                      kv_dtype, block_table, bt_stride, seqlens, B, H, D,
                                      page_size, W, k_top, topk_idx, topk_val, topk_stride,
                                      workspace, workspace_floats, dev_status, DSA_TOPK_AUTO,
                                      stream);
}

int dsa_indexer_topk_decode_static(const void* q, const float* w, const void* kcache,
                                   const void* kscale, long long page_stride_bytes,
                                   int num_pages, int kv_dtype, const int* block_table,
                                   long long bt_stride, const int* seqlens, int B, int H, int D,
                                   int page_size, int W, int k_top, int* topk_idx,
                                   float* topk_val, long long topk_stride, int* dev_status,
                                   void* stream) {
  // size first: an oversized call is refused before any device work; every
  // other argument is checked by the workspace entry point, as for a call
  // with a caller workspace (B = 0 passes no workspace and launches nothing)
  if (B > 0 && W > 0 && (long long)B * W * dsa::kPage > dsa::static_scratch_floats())
    return DSA_ERR_UNSUPPORTED;
  float* ws = nullptr;
  if (B > 0 && W > 0 && dsa::static_scratch(&ws) != cudaSuccess) return DSA_ERR_CUDA;
  return dsa_indexer_topk_decode(q, w, kcache, kscale, page_stride_bytes, num_pages, kv_dtype,
                                 block_table, bt_stride, seqlens, B, H, D, page_size, W, k_top,
                                 topk_idx, topk_val, topk_stride, ws,
                                 ws != nullptr ? dsa::static_scratch_floats() : 0, dev_status,
                                 stream);
}

int dsa_kcache_store(const void* k, const int* slot_mapping, int n, void* kcache,
                     long long page_stride_bytes, int num_pages, int kv_dtype, int D,
                     int page_size, int* dev_status, void* stream) {
  if (D != dsa::kDim || page_size != dsa::kPage) return DSA_ERR_UNSUPPORTED;
  if (kv_dtype != DSA_KV_FP8_E4M3 && kv_dtype != DSA_KV_BF16) return DSA_ERR_INVALID_ARG;
  if (n < 0 || num_pages <= 0) return DSA_ERR_INVALID_ARG;
  if (n > 0 && (!k || !slot_mapping || !kcache)) return DSA_ERR_INVALID_ARG;
  // fp8: codes then scales in one page; bf16: the values
  const long long need = kv_dtype == DSA_KV_FP8_E4M3
                             ? (long long)dsa::kPage * (dsa::kDim + 4)
                             : (long long)dsa::kPage * dsa::kDim * 2;
  if (page_stride_bytes < need) return DSA_ERR_INVALID_ARG;
  if (page_stride_bytes % 16 != 0 || !aligned(k, 16) || !aligned(kcache, 16) ||
      !aligned(slot_mapping, 4))
    return DSA_ERR_MISALIGNED;
  if (n == 0) return DSA_OK;
  cudaError_t e = dsa::launch_store(static_cast<const uint16_t*>(k), slot_mapping, n,
                                    static_cast<uint8_t*>(kcache), page_stride_bytes, num_pages,
                                    kv_dtype, dev_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: invalid argument";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: unsupported shape or mode";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED: pointer or stride misaligned";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: CUDA launch failed";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a device wait exceeded its bound";
    case DSA_ERR_BAD_PAGE: return "DSA_ERR_BAD_PAGE: block-table entry outside the pool";
    case DSA_ERR_BAD_SEQLEN: return "DSA_ERR_BAD_SEQLEN: length exceeds the block table";
    default: return "unknown dsa status";
  }
}

int dsa_indexer_abi_version(void) { return DSA_INDEXER_ABI_VERSION; }

}  // extern "C"
