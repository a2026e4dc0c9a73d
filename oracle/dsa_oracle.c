/*
 * dsa_oracle.c -- CPU fp64 oracle of the DSA indexer paged MQA-logits.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it reads the same raw input bytes and decodes them with
 * its own bit decoders.
 *
 * What it computes (the plain definition, written out):
 *
 *   out[r, t] = -inf                                      if t >= L_r
 *   out[r, t] = s(t) * sum_h w[r,h] * max(0, sum_d q[r,h,d] * k(t)[d])
 *                                                         otherwise
 *
 * with k(t) the key of cached position t of row r, found through the row's
 * block table: physical page  phys = block_table[r][t / P],  slot j = t % P.
 * The per-position weighting, the ReLU, the per-head weights and the
 * position-specific scale are the ingredients named on
 *   "The Dispatch Wire: Connecting a Triton Indexer Kernel to Production
 *    Inference", section "The Road to This Message"
 * (a batched q.k product, ReLU, weight scaling and a reduction over heads).
 * The -inf rule for positions at or past the row's length follows
 *   "The Final Gate: Validating a Custom Triton Indexer Kernel Before
 *    Production Deployment", sections "What the Test Output Reveals" and
 *    "The Thinking Process Behind the Message".
 * The key-cache layouts follow
 *   - fp8: "The Dispatch Wire ...", section "The Reasoning and
 *     Decision-Making" and "The Final Gate ...", section "Assumptions and
 *     Knowledge Required": a page of P positions holds P*D e4m3 bytes
 *     (D bytes per position) followed by P fp32 scales;
 *   - bf16: "The Dispatch Decision: Wiring a Triton Kernel into Production",
 *     section "The Problem That Led Here": D bf16 values per position
 *     (256 bytes for D = 128) and no quantisation, so the scale is 1.
 * In prefill a row is one query token and L_r is its causal limit + 1; the
 * formula is the same.
 *
 * Error rows (a reading of the pages, which are silent here):
 *   - L_r > W*P: the whole row is NaN and the call reports ORACLE_BAD_SEQLEN;
 *   - a page id outside [0, num_pages) that a valid position needs: the valid
 *     positions of that page are NaN and the call reports ORACLE_BAD_PAGE;
 *   - L_r <= 0: every position is -inf.
 *
 * Accumulation is in double; each product of a bf16 and an e4m3/bf16 value is
 * exact in double, so the result is the exact value up to the rounding of the
 * final few additions.  No blocking, fusion or reordering beyond the
 * definition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_PAGE 6
#define ORACLE_BAD_SEQLEN 7

#define ORACLE_KV_E4M3 0
#define ORACLE_KV_BF16 1

/* OCP FP8 E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, exponent field 0 is subnormal
 * (value m * 2^-9). */
double dsa_oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int expo = (code >> 3) & 0xF;
  int man = code & 0x7;
  double mag;
  if (expo == 0xF && man == 0x7) return NAN;
  if (expo == 0)
    mag = ldexp((double)man, -9);
  else
    mag = ldexp((double)(8 + man), expo - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
double dsa_oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t* q;
  const float* w;
  const uint8_t* kcache;
  const uint8_t* kscale;
  long long page_stride;
  int num_pages;
  int kv_dtype;
  const int32_t* block_table;
  long long bt_stride;
  const int32_t* seqlens;
  int R, H, D, P, W;
  double* out;
  long long out_stride;
  int row_begin, row_end;
  int status;
} oracle_job;

/* Key value d of slot j on physical page phys, decoded to double. */
static double key_value(const oracle_job* J, int phys, int j, int d) {
  const uint8_t* page = J->kcache + (long long)phys * J->page_stride;
  if (J->kv_dtype == ORACLE_KV_E4M3) {
    return dsa_oracle_e4m3_to_double(page[(long long)j * J->D + d]);
  } else {
    const uint8_t* p = page + ((long long)j * J->D + d) * 2;
    uint16_t bits = (uint16_t)(p[0] | (p[1] << 8)); /* little-endian bytes */
    return dsa_oracle_bf16_to_double(bits);
  }
}

/* Per-position scale s(t): fp32 at kscale + phys*page_stride + 4*j, or 1. */
static double key_scale(const oracle_job* J, int phys, int j) {
  float s;
  if (J->kscale == NULL) return 1.0;
  memcpy(&s, J->kscale + (long long)phys * J->page_stride + 4LL * j, sizeof s);
  return (double)s;
}

static void run_rows(oracle_job* J) {
  const long long T = (long long)J->W * J->P;
  for (int r = J->row_begin; r < J->row_end; ++r) {
    double* o = J->out + (long long)r * J->out_stride;
    const int32_t* bt = J->block_table + (long long)r * J->bt_stride;
    long long L = J->seqlens[r];
    if (L > T) {
      for (long long t = 0; t < T; ++t) o[t] = NAN;
      J->status = ORACLE_BAD_SEQLEN;
      continue;
    }
    for (long long t = 0; t < T; ++t) {
      if (t >= L) {
        o[t] = -INFINITY;
        continue;
      }
      int page = (int)(t / J->P);
      int j = (int)(t % J->P);
      int phys = bt[page];
      if (phys < 0 || phys >= J->num_pages) {
        o[t] = NAN;
        J->status = ORACLE_BAD_PAGE;
        continue;
      }
      double acc = 0.0;
      for (int h = 0; h < J->H; ++h) {
        const uint16_t* qh = J->q + ((long long)r * J->H + h) * J->D;
        double dot = 0.0;
        for (int d = 0; d < J->D; ++d)
          dot += dsa_oracle_bf16_to_double(qh[d]) * key_value(J, phys, j, d);
        double relu = dot > 0.0 ? dot : 0.0;
        acc += (double)J->w[(long long)r * J->H + h] * relu;
      }
      o[t] = key_scale(J, phys, j) * acc;
    }
  }
}

static void* thread_main(void* arg) {
  run_rows((oracle_job*)arg);
  return NULL;
}

/* Number of CPUs this process may run on. */
int dsa_oracle_cpu_count(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Logits for R rows.  q: bf16 bits [R, H, D]; w: fp32 [R, H]; kcache: page
 * pool bytes, page p at kcache + p*page_stride; kscale: NULL (scale 1) or the
 * byte address of page 0's scale section, page p's P fp32 scales at
 * kscale + p*page_stride; block_table: int32, row r at block_table +
 * r*bt_stride (bt_stride 0 = all rows share one row); seqlens: int32 [R];
 * out: double [R, out_stride >= W*P].  Rows are split over nthreads threads
 * (<= 0: all online CPUs).  Returns ORACLE_OK or the last error code seen.
 */
int dsa_oracle_logits(const uint16_t* q, const float* w, const uint8_t* kcache,
                      const uint8_t* kscale, long long page_stride,
                      int num_pages, int kv_dtype, const int32_t* block_table,
                      long long bt_stride, const int32_t* seqlens, int R,
                      int H, int D, int P, int W, double* out,
                      long long out_stride, int nthreads) {
  if (R < 0 || H <= 0 || D <= 0 || P <= 0 || W <= 0) return ORACLE_BAD_ARG;
  if (kv_dtype != ORACLE_KV_E4M3 && kv_dtype != ORACLE_KV_BF16)
    return ORACLE_BAD_ARG;
  if (out_stride < (long long)W * P) return ORACLE_BAD_ARG;
  if (R == 0) return ORACLE_OK;
  if (nthreads <= 0) nthreads = dsa_oracle_cpu_count();
  if (nthreads > R) nthreads = R;

  oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return ORACLE_BAD_ARG;
  }
  for (int i = 0; i < nthreads; ++i) {
    oracle_job* J = &jobs[i];
    J->q = q;
    J->w = w;
    J->kcache = kcache;
    J->kscale = kscale;
    J->page_stride = page_stride;
    J->num_pages = num_pages;
    J->kv_dtype = kv_dtype;
    J->block_table = block_table;
    J->bt_stride = bt_stride;
    J->seqlens = seqlens;
    J->R = R;
    J->H = H;
    J->D = D;
    J->P = P;
    J->W = W;
    J->out = out;
    J->out_stride = out_stride;
    /* interleave-free contiguous split of rows */
    J->row_begin = (int)((long long)R * i / nthreads);
    J->row_end = (int)((long long)R * (i + 1) / nthreads);
    J->status = ORACLE_OK;
  }
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&tids[i], NULL, thread_main, &jobs[i]) != 0) break;
    started = i;
  }
  /* rows of threads that failed to start run here */
  run_rows(&jobs[0]);
  for (int i = started + 1; i < nthreads; ++i) run_rows(&jobs[i]);
  for (int i = 1; i <= started; ++i) pthread_join(tids[i], NULL);

  int status = ORACLE_OK;
  for (int i = 0; i < nthreads; ++i)
    if (jobs[i].status != ORACLE_OK) status = jobs[i].status;
  free(jobs);
  free(tids);
  return status;
}

/* ---------------------------------------------------------------------------
 * Key-cache store (the step before the indexer): new key rows k[i] (bf16,
 * D values) go to slot slot_mapping[i] = page * P + slot of the pool.
 *
 * The page layouts are the ones the indexer reads (see the header of this
 * file).  The pages give no quantisation rule for the fp8 cache; the reading
 * used here maps a row's largest |k| to e4m3's largest finite value 448:
 *
 *   s = max_d |k_d| / 448      (s = 1 when the row is all zero)
 *   code_d = nearest e4m3 value to k_d / s, ties to the even code,
 *            magnitudes above 448 saturated to 448
 *
 * The scale and the quotients are rounded to fp32, as in the kernel: they
 * decide integer codes, so both sides take that decision in the same
 * precision.  The encoder below is the definition itself: it searches the
 * 127 non-negative finite e4m3 values for the nearest one.
 * ------------------------------------------------------------------------- */

/* Nearest e4m3 code to x (round to nearest, ties to even mantissa,
 * saturating to +-448); x is not NaN.  The sign is kept, as in IEEE
 * rounding: a negative value that rounds to zero gives -0 (0x80). */
uint8_t dsa_oracle_e4m3_encode(float x) {
  const double a = fabs((double)x);
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* largest finite: S.1111.110 */
  int best = 0;
  double best_d = a; /* distance to code 0 (value 0) */
  for (int c = 1; c <= 0x7E; ++c) {
    const double v = dsa_oracle_e4m3_to_double((uint8_t)c);
    const double d = fabs(a - v);
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

int dsa_oracle_kcache_store(const uint16_t* k, const int32_t* slots, int n, int D, int P,
                            uint8_t* kcache, long long page_stride, int num_pages,
                            int kv_dtype) {
  int status = ORACLE_OK;
  if (n < 0 || D <= 0 || P <= 0 || num_pages <= 0) return ORACLE_BAD_ARG;
  for (int i = 0; i < n; ++i) {
    const int sl = slots[i];
    if (sl < 0) continue;
    const int page = sl / P, slot = sl % P;
    if (page >= num_pages) {
      status = ORACLE_BAD_PAGE;
      continue;
    }
    uint8_t* pg = kcache + (long long)page * page_stride;
    const uint16_t* row = k + (long long)i * D;
    if (kv_dtype == ORACLE_KV_BF16) {
      memcpy(pg + (long long)slot * D * 2, row, (size_t)D * 2);
      continue;
    }
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
      const float v = (float)dsa_oracle_bf16_to_double(row[d]); /* exact */
      const float av = v < 0.0f ? -v : v;
      if (av > amax) amax = av;
    }
    volatile float s = amax > 0.0f ? amax / 448.0f : 1.0f; /* fp32 division */
    for (int d = 0; d < D; ++d) {
      const float v = (float)dsa_oracle_bf16_to_double(row[d]);
      volatile float x = v / s; /* fp32 division */
      pg[(long long)slot * D + d] = dsa_oracle_e4m3_encode(x);
    }
    float sv = s;
    memcpy(pg + (long long)P * D + (long long)slot * 4, &sv, 4);
  }
  return status;
}
