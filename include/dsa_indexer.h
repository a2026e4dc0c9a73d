/*
 * dsa_indexer.h -- C ABI of the GB300 (sm_103a) DSA indexer paged
 * MQA-logits library, libdsa_indexer.so.
 *
 * The operation.  For every row r (a decode request, or a prefill query
 * token) and every cached key position t in [0, W*64):
 *
 *     out[r, t] = scale(t) * sum_{h<64} w[r, h] * max(0, q[r, h, :] . k(t))
 *                                                      if t <  seqlens[r]
 *     out[r, t] = -inf                                 if t >= seqlens[r]
 *
 * The per-head dot, the ReLU, the per-head weights and the per-position
 * scale are the ingredients listed on "The Dispatch Wire: Connecting a
 * Triton Indexer Kernel to Production Inference", section "The Road to This
 * Message".  The -inf rule is the "inf-pattern" criterion of "The Final Gate:
 * Validating a Custom Triton Indexer Kernel Before Production Deployment",
 * section "What the Test Output Reveals".  The output shape is fixed
 * ([rows, W*64]) and work past seqlens[r] is skipped inside the kernel, so a
 * call can be captured in a CUDA graph and replayed with new lengths and
 * block tables: "The Moment the Context-Length Tax Vanished: Committing the
 * O(actual) Triton Indexer", section "The Commit: Engineering as Narrative".
 *
 * The key cache.  Keys live in physical pages of 64 positions x D = 128
 * values.  Position t of row r is slot (t % 64) of physical page
 * block_table[r][t / 64] (the page table of "The Final Gate ...", section
 * "Assumptions and Knowledge Required").  Page p starts at
 * (char*)kcache + p * page_stride_bytes and holds its 64 key rows
 * position-major (D values per position, contiguous):
 *   DSA_KV_FP8_E4M3  OCP e4m3 ("e4m3fn") bytes, 128 bytes per position.  The
 *                    fused page of "The Dispatch Wire ...", section "The
 *                    Reasoning and Decision-Making", is 8,448 bytes: 8,192
 *                    bytes of keys then 64 fp32 scales, i.e.
 *                    page_stride_bytes = 8448 and kscale = kcache + 8192.
 *   DSA_KV_BF16      bf16, 256 bytes per position, 16,384 bytes per page,
 *                    no quantisation ("The Dispatch Decision: Wiring a Triton
 *                    Kernel into Production", section "The Problem That Led
 *                    Here"); pass kscale = NULL for scale 1.
 * kscale, when not NULL, is the address of page 0's 64 fp32 scales; page p's
 * are at (char*)kscale + p * page_stride_bytes.  NULL means scale(t) = 1.
 *
 * Common rules for the indexer entry points.
 *   Memory.   Every pointer except `stream` is a DEVICE pointer owned by the
 *             caller (the varlen prefill's request offsets are host data).
 *             The library allocates nothing, never synchronises and
 *             launches one kernel per call on `stream` (a cudaStream_t;
 *             NULL = legacy default stream); the top-k calls launch two, the
 *             varlen prefill one per 128 requests.  All calls are legal inside
 *             stream capture.  Every kernel is launched with
 *             programmatic dependent launch allowed: its set-up may overlap
 *             the tail of the previous kernel in the stream, but it reads no
 *             argument array before that kernel has completed.
 *   Shapes.   Only H = 64, D = 128 and page_size = 64 are supported
 *             (DSA_ERR_UNSUPPORTED otherwise).  W >= 1.  Rows may be 0 (no
 *             launch, DSA_OK).
 *   Layouts.  q: bf16 [rows, 64, 128] contiguous.  w: fp32 [rows, 64]
 *             contiguous.  block_table: int32, row r at
 *             block_table + r * bt_stride, W entries used (bt_stride = 0
 *             means every row shares row 0; otherwise bt_stride >= W).
 *             seqlens: int32 [rows].  out: fp32, row r at
 *             out + r * out_stride, W*64 entries written (out_stride >=
 *             W*64).
 *   Alignment. q, kcache and out 16-byte aligned; kscale 16-byte aligned;
 *             page_stride_bytes a multiple of 16 and at least the key bytes
 *             of a page (8,192 fp8, 16,384 bf16); out_stride a multiple of
 *             4 (DSA_ERR_MISALIGNED otherwise).
 *   Host errors.  Invalid arguments are reported by the return value and
 *             nothing is launched.  A launch failure returns DSA_ERR_CUDA.
 *   Data errors (found by the kernel; never a trap or a fault):
 *             - seqlens[r] > W*64: the whole row is written NaN, status
 *               DSA_ERR_BAD_SEQLEN;
 *             - a block-table entry outside [0, num_pages) that a valid
 *               position needs: that page's valid positions are NaN, status
 *               DSA_ERR_BAD_PAGE;
 *             - an internal wait that does not complete within its bound:
 *               the affected outputs are NaN, status DSA_ERR_TIMEOUT.
 *             The status is stored with atomicMax into *dev_status when
 *             dev_status is not NULL; the library never clears it (zero it
 *             before the call to read a fresh status).  seqlens[r] <= 0 is
 *             not an error: the row is all -inf.  Entries of the block table
 *             at or past ceil(seqlens[r] / 64) are never used as page ids and
 *             may hold any value (decode may load the first entries of a row
 *             before it knows the row's length; all W entries of every row
 *             must therefore be readable memory).
 */
#ifndef DSA_INDEXER_H
#define DSA_INDEXER_H

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_INDEXER_ABI_VERSION 1

typedef enum {
  DSA_KV_FP8_E4M3 = 0,
  DSA_KV_BF16 = 1
} dsa_kv_dtype_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,
  DSA_ERR_UNSUPPORTED = 2,
  DSA_ERR_MISALIGNED = 3,
  DSA_ERR_CUDA = 4,
  DSA_ERR_TIMEOUT = 5,
  DSA_ERR_BAD_PAGE = 6,
  DSA_ERR_BAD_SEQLEN = 7
} dsa_status_t;

/*
 * Decode: B requests, one query token each.  Row b uses q[b], w[b], block
 * table row b and length seqlens[b].  The grid is fixed by (B, W) alone, so
 * the launch does not depend on the lengths: "The Dispatch Wire ...",
 * section "The Reasoning and Decision-Making" (one program per request and
 * page, early exit past the request's length).
 */
int dsa_indexer_logits_decode(const void* q, const float* w,
                              const void* kcache, const void* kscale,
                              long long page_stride_bytes, int num_pages,
                              int kv_dtype, const int* block_table,
                              long long bt_stride, const int* seqlens, int B,
                              int H, int D, int page_size, int W, float* out,
                              long long out_stride, int* dev_status,
                              void* stream);

/*
 * Prefill: n_q query tokens.  Query i uses q[i], w[i], block-table row i
 * (bt_stride = 0: all queries share row 0, the one-request prefill of "The
 * Dispatch Decision ...", section "The Problem That Led Here") and length
 * seqlens[i] = its causal limit + 1.  Keys are read page by page from the
 * cache: no gathered copy is made.  A shared row (bt_stride = 0) runs the
 * query-tile kernel, which reuses each key tile for four query tokens (fp8
 * keys: the query is split into two e4m3 terms, as in decode).  Per-query
 * rows (bt_stride >= W: several requests in one call, or multi-token
 * decode) run the decode kernel with one row per query token; there
 * n_q <= 65535 (DSA_ERR_UNSUPPORTED otherwise).  Range (query-tile kernel,
 * bf16 keys): half of the heads
 * take their ReLU as a saturating multiply by 2^-64 with the weight scaled
 * by 2^64, so results are defined for |w[i, h]| < 2^64 and per-head dots
 * |q . k| < 2^64.
 */
int dsa_indexer_logits_prefill(const void* q, const float* w,
                               const void* kcache, const void* kscale,
                               long long page_stride_bytes, int num_pages,
                               int kv_dtype, const int* block_table,
                               long long bt_stride, const int* seqlens,
                               int n_q, int H, int D, int page_size, int W,
                               float* out, long long out_stride,
                               int* dev_status, void* stream);

/*
 * Prefill of several requests in one call, with a table row per request:
 * the query tokens of request b are rows [cu_q[b], cu_q[b+1]) of q, w,
 * seqlens and out, and read the keys through block-table row b
 * (block_table + b * bt_stride; bt_stride >= W, or 0 for one row shared by
 * all requests).  Query i may see the positions t < seqlens[i] (its causal
 * limit + 1), as in dsa_indexer_logits_prefill; positions past it hold
 * -inf.  No gathered per-query copy of the keys is made ("The Dispatch
 * Decision ...", section "The Problem That Led Here": the materialised
 * [query tokens, pages, ...] gather is what ran out of memory).
 *
 * cu_q is a HOST array of n_req + 1 offsets: cu_q[0] = 0, non-decreasing
 * (DSA_ERR_INVALID_ARG otherwise, checked before any launch); n_q =
 * cu_q[n_req] rows in all.  The requests' query tiles run in one launch of
 * the query-tile kernel of dsa_indexer_logits_prefill (up to 128 requests a
 * launch; more run as further launches, in request order, on `stream`),
 * each tile reading its own request's table row, so requests of many tokens
 * reuse each key tile four times; requests of one or a few tokens are
 * better served by per-query rows.  Other arguments, layouts, alignment,
 * range and device errors as for dsa_indexer_logits_prefill.  DSA_ERR_CUDA
 * from a launch may leave the earlier groups of requests launched.
 */
int dsa_indexer_logits_prefill_varlen(const void* q, const float* w, const void* kcache,
                                      const void* kscale, long long page_stride_bytes,
                                      int num_pages, int kv_dtype, const int* block_table,
                                      long long bt_stride, const int* cu_q, int n_req,
                                      const int* seqlens, int H, int D, int page_size, int W,
                                      float* out, long long out_stride, int* dev_status,
                                      void* stream);

/* How the top-k decode computes its selection (dsa_indexer_topk_decode_form). */
typedef enum {
  DSA_TOPK_AUTO = 0,      /* the library's choice (today: two passes) */
  DSA_TOPK_TWO_PASS = 1,  /* the logits into the workspace, then a selection kernel */
  DSA_TOPK_FUSED = 2      /* selection in the decode epilogue, then a merge kernel */
} dsa_topk_form_t;

/*
 * Decode with top-k selection: for every request b, the k_top positions
 * t < seqlens[b] with the largest logits (the positions sparse attention
 * then reads), instead of the [B, W*64] logits.  topk_idx: int32, row b at
 * topk_idx + b * topk_stride (topk_stride >= k_top), the selected positions
 * in increasing order; a row with L <= k_top valid positions takes all of
 * them and pads with -1.  topk_val (nullable): their logits, same layout,
 * -inf for the padding.  Equal logits at the k-th place are taken in
 * position order.  workspace: device fp32 buffer of at least
 * B * W * 64 entries (16-byte aligned), owned by the caller; no -inf fill
 * is written anywhere.  Two kernel launches on `stream`, in one of two
 * forms (this entry point takes the two-pass one; the caller chooses with
 * dsa_indexer_topk_decode_form):
 *   two passes: the decode kernel writes the logits of the valid positions
 *     into the workspace, then the selection kernel (a cluster of two CTAs
 *     per request while 2 * B CTAs fit in one wave of one CTA per SM, else
 *     one CTA per request: a histogram pass, the k-th value's bin collected
 *     and ranked, an in-order write) reads them;
 *   fused: the decode kernel keeps the logits in shared memory, chunk by
 *     chunk of up to 32 pages of a row, and writes each chunk's best
 *     min(k_top, n) positions with their logits to the workspace; a merge
 *     kernel then selects each request's best among them.  No logit of the
 *     call is written to global memory.  It applies when k_top <= 2048 (a
 *     chunk: for k_top >= 2048 every chunk keeps all its positions and the
 *     merge does all the selecting), the
 *     decode takes its balanced form (W > 64 and B <= 384) and the
 *     workspace holds 4 * ceil((B + 1) / 4) + (C + B + ceil(B * W / 32)) *
 *     (4 + 2 * k_top) floats, C being the decode's persistent CTAs (two per
 *     SM).
 * Both forms take the same positions and return the same logits, bit for
 * bit: the logits come from the same arithmetic and the order is total.
 * Other arguments, checks and data errors as for dsa_indexer_logits_decode;
 * an over-long row selects nothing (all -1) and reports DSA_ERR_BAD_SEQLEN.
 */
int dsa_indexer_topk_decode(const void* q, const float* w, const void* kcache,
                            const void* kscale, long long page_stride_bytes, int num_pages,
                            int kv_dtype, const int* block_table, long long bt_stride,
                            const int* seqlens, int B, int H, int D, int page_size, int W,
                            int k_top, int* topk_idx, float* topk_val, long long topk_stride,
                            float* workspace, long long workspace_floats, int* dev_status,
                            void* stream);

/*
 * dsa_indexer_topk_decode with the form chosen by the caller (a
 * dsa_topk_form_t; DSA_ERR_INVALID_ARG for another value).  DSA_TOPK_FUSED
 * where the fused form does not apply returns DSA_ERR_UNSUPPORTED before
 * any launch.  The top-k is the logits' consumer: "The Dispatch Decision
 * ...", section "The Problem That Led Here".
 */
int dsa_indexer_topk_decode_form(const void* q, const float* w, const void* kcache,
                                 const void* kscale, long long page_stride_bytes, int num_pages,
                                 int kv_dtype, const int* block_table, long long bt_stride,
                                 const int* seqlens, int B, int H, int D, int page_size, int W,
                                 int k_top, int* topk_idx, float* topk_val, long long topk_stride,
                                 float* workspace, long long workspace_floats, int* dev_status,
                                 int form, void* stream);

/*
 * dsa_indexer_topk_decode without a caller workspace, for callers that
 * cannot allocate device memory for it (an allocator that is not theirs to
 * call, a memory pool fixed at start-up, code running inside another
 * library's allocation-free hot path).  The logits go to a fixed device
 * array of the library (24 Mi floats, 96 MiB per device); the call itself
 * allocates nothing.  With lazy module loading (the CUDA default) the array
 * is reserved on a device when this entry point is first used there; under
 * CUDA_MODULE_LOADING=EAGER every process that loads the library reserves
 * it on every device it creates a context on, whether or not it calls this.
 * B * W * 64 must not exceed 24 Mi (DSA_ERR_UNSUPPORTED otherwise, checked
 * before any device work).  The array is shared: calls on one device must
 * not overlap (use one stream, or order the streams), or they race.  The
 * first call with B > 0 on a device looks up the array's address (which may
 * load its module), so make one such call before capturing one in a CUDA
 * graph.  The pages have no counterpart: this is a convenience of the
 * library.  Every other argument is checked, and every result written, as
 * by dsa_indexer_topk_decode.
 */
int dsa_indexer_topk_decode_static(const void* q, const float* w, const void* kcache,
                                   const void* kscale, long long page_stride_bytes,
                                   int num_pages, int kv_dtype, const int* block_table,
                                   long long bt_stride, const int* seqlens, int B, int H, int D,
                                   int page_size, int W, int k_top, int* topk_idx,
                                   float* topk_val, long long topk_stride, int* dev_status,
                                   void* stream);

/*
 * Key-cache store: writes n new key rows into their cache slots, in the
 * page layouts above (the step before the indexer: its keys come from this
 * cache).  k: bf16 [n, 128], 16-byte aligned.  slot_mapping: int32 [n],
 * entry i = page * 64 + slot of row i; a negative entry skips the row.
 * kcache: the pool, page p at (char*)kcache + p * page_stride_bytes.
 *   DSA_KV_FP8_E4M3  page_stride_bytes >= 8448: the slot's 128 e4m3 codes
 *                    at page + slot * 128 and its fp32 scale s at
 *                    page + 8192 + slot * 4, with s = max_d |k[i, d]| / 448
 *                    (1 for an all-zero row) and code_d = e4m3(k[i, d] / s)
 *                    rounded to nearest even and saturated to +-448, every
 *                    step in fp32.  The pages give no quantisation rule; this
 *                    one maps the row's largest |k| to e4m3's largest finite
 *                    value, so k ~ code * s.
 *   DSA_KV_BF16      page_stride_bytes >= 16384: the row's 256 bytes at
 *                    page + slot * 256.
 * Host errors as for the indexer calls (D = 128, page_size = 64; k and
 * kcache 16-byte aligned, page_stride_bytes a multiple of 16).  A slot at or
 * past num_pages * 64 is skipped and DSA_ERR_BAD_PAGE stored into
 * *dev_status.  One kernel launch on `stream`; nothing is allocated.  Rows
 * with the same slot race (the last writer is unspecified).
 */
int dsa_kcache_store(const void* k, const int* slot_mapping, int n, void* kcache,
                     long long page_stride_bytes, int num_pages, int kv_dtype,
                     int D, int page_size, int* dev_status, void* stream);

/* A static, human-readable name for a status code. */
const char* dsa_status_string(int status);

/* DSA_INDEXER_ABI_VERSION of the loaded library. */
int dsa_indexer_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H */
