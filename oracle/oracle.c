/*
 * oracle.c -- plain, slow CPU reference for paged GQA decode over a block-table
 * KV cache and for the GrowPage-style page budgeting step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
 * baseline load this file's library.  It shares no code, header, table or
 * helper with the CUDA library; the only thing both sides consume is the
 * seeded inputs built by the workload generator.
 *
 * Sources (web pages this build follows):
 *  [PKV]  aissential.tech, "PersistentKV: Page-Aware Decode Scheduling for
 *         Long-Context LLM Serving on Commodity GPUs" -- Summary and Method:
 *         block-table decode attention for grouped-query attention, K/V tiles
 *         reused across the grouped query heads, a compact workqueue of
 *         non-empty (sequence, KV-head, split) tasks.
 *  [GP]   mlsanity.com, "GrowPage: On-Demand KV Budgeting for Efficient LLM
 *         Reasoning Serving" -- Abstract: query summaries kept at a short
 *         and a long time scale, their attention working sets compared to
 *         track demand, compress-or-grow at each capacity boundary, on top
 *         of PagedAttention pages.
 *  [GP1]  aitrending.vip GrowPage summary -- Technical Details (same method).
 *  [EKV]  paperlayer.ai, "Elastic KV Cache for LLM Serving" -- section 2:
 *         fixed-size KV blocks handed out from an integer free list.
 *
 * Precision.  Attention (decode, split, merge) is computed in fp64 from the
 * exact fp16/bf16 input values.  The budgeting chain (query EMAs, page key
 * summaries, page scores) feeds integer decisions (top-k, grow/compact); the
 * pages fix no precision for it, so those decisions are taken in the CUDA
 * kernels' precision: fp32 with every operation rounded to nearest and the
 * summation order written out below (or_*_f32).  fp64 versions of the same
 * quantities (or_*_f64) exist to pin the fp32 ones within rounding bounds.
 *
 * Status codes returned here mirror the library's documented codes:
 *   0 ok, -1 invalid argument, -2 bad page id, -3 free list exhausted,
 *   -6 block-table row full.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_EBADPAGE (-2)
#define OR_ENOSPACE (-3)
#define OR_EFULL (-6)

#define OR_F16 0
#define OR_BF16 1

/* ------------------------------------------------------------------------ */
/* 16-bit float formats, decoded from their definitions.                     */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double or_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);              /* subnormal: m * 2^(1-15-10) */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/2^10) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double or_bf16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int m = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133);             /* subnormal: m * 2^(1-127-7) */
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(128 + m), e - 134);  /* (1 + m/2^7) * 2^(e-127) */
  return sign ? -v : v;
}

static double cv(uint16_t h, int dtype) {
  return dtype == OR_BF16 ? or_bf16_to_f64(h) : or_f16_to_f64(h);
}

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* ------------------------------------------------------------------------ */
/* Decode: one query token per sequence, GQA over a paged cache [PKV].       */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t *q, *k_pool, *v_pool;
  const int32_t *table, *seq_lens;
  int max_pages, num_pages, B, ps, Hq, Hkv, d, dtype;
  double scale;
  size_t q_seq_stride; /* elements between two sequences' q (0 = Hq * d) */
} DecodeArgs;

/* Attention of query head hq of sequence b over its tokens [t0, t1).
 * Query head hq reads KV head hq / G (contiguous grouping, G = Hq / Hkv).
 * Token t lives in pool page block_table[b][t / ps], slot t % ps.
 *   s_t = scale * <q, k_t>;  lse = ln sum_t exp(s_t) (as m + ln sum exp(s_t - m));
 *   out = sum_t exp(s_t - lse) v_t.
 * An empty range gives out = 0 and lse = -inf.                               */
static int decode_range(const DecodeArgs *a, int b, int hq, int64_t t0, int64_t t1,
                        double *out, double *lse) {
  int G = a->Hq / a->Hkv;
  int h = hq / G;
  int d = a->d;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (t1 <= t0) {
    *lse = -INFINITY;
    return OR_OK;
  }
  const size_t qs = a->q_seq_stride ? a->q_seq_stride : (size_t)a->Hq * d;
  const uint16_t *qv = a->q + (size_t)b * qs + (size_t)hq * d;
  double *qd = (double *)malloc(sizeof(double) * d);
  double *s = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
  for (int c = 0; c < d; ++c) qd[c] = cv(qv[c], a->dtype);
  int rc = OR_OK;
  for (int64_t t = t0; t < t1; ++t) {
    int32_t page = a->table[(size_t)b * a->max_pages + t / a->ps];
    if (page < 0 || page >= a->num_pages) { rc = OR_EBADPAGE; goto done; }
    const uint16_t *kt = a->k_pool + (((size_t)page * a->Hkv + h) * a->ps + t % a->ps) * d;
    double dot = 0.0;
    for (int c = 0; c < d; ++c) dot += qd[c] * cv(kt[c], a->dtype);
    s[t - t0] = a->scale * dot;
  }
  double m = -INFINITY;
  for (int64_t t = t0; t < t1; ++t) if (s[t - t0] > m) m = s[t - t0];
  double sum = 0.0;
  for (int64_t t = t0; t < t1; ++t) sum += exp(s[t - t0] - m);
  *lse = m + log(sum);
  for (int64_t t = t0; t < t1; ++t) {
    int32_t page = a->table[(size_t)b * a->max_pages + t / a->ps];
    const uint16_t *vt = a->v_pool + (((size_t)page * a->Hkv + h) * a->ps + t % a->ps) * d;
    double w = exp(s[t - t0] - *lse);
    for (int c = 0; c < d; ++c) out[c] += w * cv(vt[c], a->dtype);
  }
done:
  free(qd);
  free(s);
  return rc;
}

static int check_decode_args(const DecodeArgs *a) {
  if (a->B < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->d <= 0 || a->ps <= 0) return OR_EINVAL;
  if (a->Hq % a->Hkv) return OR_EINVAL;
  for (int b = 0; b < a->B; ++b) {
    if (a->seq_lens[b] < 0) return OR_EINVAL;
    if (ceil_div64(a->seq_lens[b], a->ps) > a->max_pages) return OR_EINVAL;
  }
  return OR_OK;
}

typedef struct {
  const DecodeArgs *a;
  double *out, *lse;
  int next_row, nrows, rc;
  pthread_mutex_t mu;
} DecodePool;

static void *decode_worker(void *p) {
  DecodePool *pool = (DecodePool *)p;
  const DecodeArgs *a = pool->a;
  for (;;) {
    pthread_mutex_lock(&pool->mu);
    int r = pool->next_row++;
    pthread_mutex_unlock(&pool->mu);
    if (r >= pool->nrows) break;
    /* one work item = one (sequence, KV head): its G query heads */
    int b = r / a->Hkv, h = r % a->Hkv, G = a->Hq / a->Hkv;
    for (int g = 0; g < G; ++g) {
      int hq = h * G + g;
      int rc = decode_range(a, b, hq, 0, a->seq_lens[b], pool->out + ((size_t)b * a->Hq + hq) * a->d,
                            pool->lse + (size_t)b * a->Hq + hq);
      if (rc) {
        pthread_mutex_lock(&pool->mu);
        pool->rc = rc;
        pthread_mutex_unlock(&pool->mu);
      }
    }
  }
  return NULL;
}

/* Full decode step: out [B][Hq][d], lse [B][Hq] (natural log, scale included). */
int or_decode(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
              const int32_t *block_table, int max_pages, int num_pages, const int32_t *seq_lens,
              int B, int page_size, int Hq, int Hkv, int d, int dtype, double scale,
              double *out, double *lse, int nthreads) {
  DecodeArgs a = {q, k_pool, v_pool, block_table, seq_lens, max_pages, num_pages,
                  B, page_size, Hq, Hkv, d, dtype, scale, 0};
  int rc = check_decode_args(&a);
  if (rc) return rc;
  DecodePool pool;
  pool.a = &a;
  pool.out = out;
  pool.lse = lse;
  pool.next_row = 0;
  pool.nrows = B * Hkv;
  pool.rc = OR_OK;
  pthread_mutex_init(&pool.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, decode_worker, &pool);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&pool.mu);
  return pool.rc;
}

/* Decode for a list of (b, hq) pairs only -- used to check sampled outputs of
 * full-size workloads.  rows: [nrows][2]; out [nrows][d]; lse [nrows].       */
int or_decode_rows(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                   const int32_t *block_table, int max_pages, int num_pages, const int32_t *seq_lens,
                   int B, int page_size, int Hq, int Hkv, int d, int dtype, double scale,
                   const int32_t *rows, int nrows, double *out, double *lse) {
  DecodeArgs a = {q, k_pool, v_pool, block_table, seq_lens, max_pages, num_pages,
                  B, page_size, Hq, Hkv, d, dtype, scale, 0};
  int rc = check_decode_args(&a);
  if (rc) return rc;
  for (int r = 0; r < nrows; ++r) {
    int b = rows[2 * r], hq = rows[2 * r + 1];
    if (b < 0 || b >= B || hq < 0 || hq >= Hq) return OR_EINVAL;
    rc = decode_range(&a, b, hq, 0, seq_lens[b], out + (size_t)r * d, lse + r);
    if (rc) return rc;
  }
  return OR_OK;
}

/* Attention of (b, hq) restricted to tokens [t0, t1): the partial result one
 * KV split produces (out normalised over its own tokens, lse over them).     */
int or_decode_range(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                    const int32_t *block_table, int max_pages, int num_pages, const int32_t *seq_lens,
                    int B, int page_size, int Hq, int Hkv, int d, int dtype, double scale,
                    int b, int hq, int64_t t0, int64_t t1, double *out, double *lse) {
  DecodeArgs a = {q, k_pool, v_pool, block_table, seq_lens, max_pages, num_pages,
                  B, page_size, Hq, Hkv, d, dtype, scale, 0};
  if (t0 < 0 || t1 > seq_lens[b]) return OR_EINVAL;
  return decode_range(&a, b, hq, t0, t1, out, lse);
}

/* Several query tokens per sequence -- the step before decode (a prefill
 * chunk, or drafted tokens being verified) over the same pool and table.
 * The T queries of sequence b are its last T tokens; query i attends to the
 * tokens [0, L_b - T + 1 + i) (causal), with the attention of decode_range.
 * q, out: [B][T][Hq][d]; lse: [B][T][Hq].                                   */
typedef struct {
  const DecodeArgs *a;
  const uint16_t *q;
  int T;
  double *out, *lse;
  int next, n, rc;
  pthread_mutex_t mu;
} MultiPool;

static void *multi_worker(void *p) {
  MultiPool *pool = (MultiPool *)p;
  for (;;) {
    pthread_mutex_lock(&pool->mu);
    int r = pool->next++;
    pthread_mutex_unlock(&pool->mu);
    if (r >= pool->n) break;
    /* one work item = one (query token i, sequence b, KV head h) */
    DecodeArgs a = *pool->a;
    const int T = pool->T, Hq = a.Hq, d = a.d, G = a.Hq / a.Hkv;
    const int h = r % a.Hkv, b = (r / a.Hkv) % a.B, i = r / (a.Hkv * a.B);
    a.q = pool->q + (size_t)i * Hq * d;  /* query token i of every sequence */
    int64_t lim = (int64_t)a.seq_lens[b] - T + 1 + i;
    if (lim < 0) lim = 0;
    for (int g = 0; g < G; ++g) {
      const int hq = h * G + g;
      const size_t row = ((size_t)b * T + i) * Hq + hq;
      int rc = decode_range(&a, b, hq, 0, lim, pool->out + row * d, pool->lse + row);
      if (rc) {
        pthread_mutex_lock(&pool->mu);
        pool->rc = rc;
        pthread_mutex_unlock(&pool->mu);
      }
    }
  }
  return NULL;
}

int or_attend_multi(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                    const int32_t *block_table, int max_pages, int num_pages,
                    const int32_t *seq_lens, int B, int T, int page_size, int Hq, int Hkv, int d,
                    int dtype, double scale, double *out, double *lse, int nthreads) {
  if (T < 1) return OR_EINVAL;
  DecodeArgs a = {q, k_pool, v_pool, block_table, seq_lens, max_pages, num_pages,
                  B, page_size, Hq, Hkv, d, dtype, scale, (size_t)T * Hq * d};
  int rc = check_decode_args(&a);
  if (rc) return rc;
  MultiPool pool;
  pool.a = &a;
  pool.q = q;
  pool.T = T;
  pool.out = out;
  pool.lse = lse;
  pool.next = 0;
  pool.n = T * B * Hkv;
  pool.rc = OR_OK;
  pthread_mutex_init(&pool.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
  for (int k = 0; k < nthreads; ++k) pthread_create(&th[k], NULL, multi_worker, &pool);
  for (int k = 0; k < nthreads; ++k) pthread_join(th[k], NULL);
  free(th);
  pthread_mutex_destroy(&pool.mu);
  return pool.rc;
}

/* Log-sum-exp merge of split partials (the exact recombination of softmax
 * pieces; the pages' "sequence-split" tasks [PKV, Method] need it):
 *   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) out_s.
 * Parts with lse_s = -inf (empty) contribute nothing.                        */
void or_merge(const double *lse_parts, const double *out_parts, int nparts, int d,
              double *lse, double *out) {
  double m = -INFINITY;
  for (int s = 0; s < nparts; ++s) if (lse_parts[s] > m) m = lse_parts[s];
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  double sum = 0.0;
  for (int s = 0; s < nparts; ++s) sum += exp(lse_parts[s] - m);
  *lse = m + log(sum);
  for (int s = 0; s < nparts; ++s) {
    double w = exp(lse_parts[s] - *lse);
    for (int c = 0; c < d; ++c) out[c] += w * out_parts[(size_t)s * d + c];
  }
}

/* ------------------------------------------------------------------------ */
/* Workqueue of non-empty (sequence, KV-head, split) tasks [PKV].            */
/* ------------------------------------------------------------------------ */

/* Split size rule when the caller passes 0: spread the W non-empty pages of
 * the batch evenly over the decode workers, never below min_chunk pages.    */
int64_t or_chunk_auto(int64_t W, int64_t n_workers, int64_t min_chunk) {
  int64_t c = n_workers > 0 ? ceil_div64(W, n_workers) : W;
  if (c < min_chunk) c = min_chunk;
  if (c < 1) c = 1;
  return c;
}

/* Definition.  Sequence b holds np_b = ceil(L_b / ps) pages; laying the
 * sequences' pages end to end gives offsets O_b = sum_{b'<b} np_b' and a total
 * W.  The flattened range is cut into chunks of `chunk` pages; each chunk is
 * one decode worker's share.  A split of sequence b is the non-empty
 * intersection of [O_b, O_b + np_b) with one chunk; every split yields one
 * task per KV head.  Task record (8 int32):
 *   b, h, split, nsplit_b, page_begin, page_end (pages of b), chunk, L_b.
 * Order: by (b, split, h).  chunk_begin[c] (c = 0..nchunks) is the index of
 * the first (b, split) group whose chunk is >= c; seq_group_begin[b] the index
 * of b's first group; seq_nsplit[b] its split count (0 when L_b = 0).
 * meta[0..4] = number of tasks, number of groups, chunk, nchunks, W.          */
int or_workqueue(const int32_t *seq_lens, int B, int Hkv, int page_size, int64_t chunk,
                 int32_t *tasks, int64_t max_tasks, int32_t *chunk_begin, int64_t max_chunks,
                 int32_t *seq_group_begin, int32_t *seq_nsplit, int64_t *meta) {
  if (B < 0 || Hkv <= 0 || page_size <= 0 || chunk <= 0) return OR_EINVAL;
  int64_t W = 0;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) return OR_EINVAL;
    W += ceil_div64(seq_lens[b], page_size);
  }
  int64_t nchunks = W > 0 ? ceil_div64(W, chunk) : 0;
  if (nchunks + 1 > max_chunks) return OR_EINVAL;
  int64_t ntask = 0, ngroup = 0, O = 0;
  int64_t next_chunk = 0; /* chunk_begin entries written so far */
  for (int b = 0; b < B; ++b) {
    int64_t np = ceil_div64(seq_lens[b], page_size);
    seq_group_begin[b] = (int32_t)ngroup;
    seq_nsplit[b] = 0;
    if (np == 0) continue;
    int64_t c_first = O / chunk, c_last = (O + np - 1) / chunk;
    seq_nsplit[b] = (int32_t)(c_last - c_first + 1);
    for (int64_t c = c_first; c <= c_last; ++c) {
      int64_t lo = c * chunk > O ? c * chunk : O;
      int64_t hi = (c + 1) * chunk < O + np ? (c + 1) * chunk : O + np;
      while (next_chunk <= c) chunk_begin[next_chunk++] = (int32_t)ngroup;
      for (int h = 0; h < Hkv; ++h) {
        if (ntask >= max_tasks) return OR_EINVAL;
        int32_t *r = tasks + 8 * ntask;
        r[0] = b;
        r[1] = h;
        r[2] = (int32_t)(c - c_first);
        r[3] = seq_nsplit[b];
        r[4] = (int32_t)(lo - O);
        r[5] = (int32_t)(hi - O);
        r[6] = (int32_t)c;
        r[7] = seq_lens[b];
        ++ntask;
      }
      ++ngroup;
    }
    O += np;
  }
  while (next_chunk <= nchunks) chunk_begin[next_chunk++] = (int32_t)ngroup;
  meta[0] = ntask;
  meta[1] = ngroup;
  meta[2] = chunk;
  meta[3] = nchunks;
  meta[4] = W;
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Dual-timescale query summaries [GP, Abstract; GP1, Technical Details].    */
/* The pages give no formula.  This build's instantiation: per KV head h the */
/* group-mean query g_t[h] = mean over the G query heads of h; a fast and a  */
/* slow exponential moving average with decays a_fast, a_slow:               */
/*   ema <- a * ema + (1 - a) * g_t,   initialised to g_t on the first step. */
/* State layout: ema [B][2][Hkv][d] (index 0 fast, 1 slow).                  */
/* ------------------------------------------------------------------------ */

/* fp32, operation by operation: acc = 0; acc = acc + q_g (g ascending);
 * g = acc / G; ema = (a * ema) + ((1 - a) * g), each op rounded to fp32.     */
void or_ema_f32(const uint16_t *q, int B, int Hq, int Hkv, int d, int dtype,
                float a_fast, float a_slow, int first, float *ema) {
  int G = Hq / Hkv;
  float a[2] = {a_fast, a_slow};
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int c = 0; c < d; ++c) {
        float acc = 0.0f;
        for (int g = 0; g < G; ++g) {
          float x = (float)cv(q[((size_t)b * Hq + h * G + g) * d + c], dtype);
          acc = acc + x;
        }
        float gm = acc / (float)G;
        for (int u = 0; u < 2; ++u) {
          float *e = &ema[(((size_t)b * 2 + u) * Hkv + h) * d + c];
          if (first) {
            *e = gm;
          } else {
            float t1 = a[u] * *e;
            float om = 1.0f - a[u];
            float t2 = om * gm;
            *e = t1 + t2;
          }
        }
      }
}

void or_ema_f64(const uint16_t *q, int B, int Hq, int Hkv, int d, int dtype,
                double a_fast, double a_slow, int first, double *ema) {
  int G = Hq / Hkv;
  double a[2] = {a_fast, a_slow};
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h)
      for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int g = 0; g < G; ++g) acc += cv(q[((size_t)b * Hq + h * G + g) * d + c], dtype);
        double gm = acc / G;
        for (int u = 0; u < 2; ++u) {
          double *e = &ema[(((size_t)b * 2 + u) * Hkv + h) * d + c];
          *e = first ? gm : a[u] * *e + (1.0 - a[u]) * gm;
        }
      }
}

/* ------------------------------------------------------------------------ */
/* Page key summaries: per (page, KV head, channel) the mean, minimum and     */
/* maximum key over the page's ps slots.  Layout summ [P][Hkv][3][d]:         */
/* index 0 mean, 1 min, 2 max.  Only the listed pages are written.           */
/* fp32 mean: acc = 0; acc = acc + k_t (t ascending); mean = acc / ps.       */
/* ------------------------------------------------------------------------ */

int or_page_summaries_f32(const uint16_t *k_pool, int num_pages, const int32_t *page_ids, int n,
                          int Hkv, int ps, int d, int dtype, float *summ) {
  for (int i = 0; i < n; ++i) {
    int32_t p = page_ids[i];
    if (p < 0 || p >= num_pages) return OR_EBADPAGE;
    for (int h = 0; h < Hkv; ++h)
      for (int c = 0; c < d; ++c) {
        float acc = 0.0f, mn = INFINITY, mx = -INFINITY;
        for (int t = 0; t < ps; ++t) {
          float x = (float)cv(k_pool[(((size_t)p * Hkv + h) * ps + t) * d + c], dtype);
          acc = acc + x;
          if (x < mn) mn = x;
          if (x > mx) mx = x;
        }
        float *s = summ + ((size_t)p * Hkv + h) * 3 * d;
        s[c] = acc / (float)ps;
        s[d + c] = mn;
        s[2 * d + c] = mx;
      }
  }
  return OR_OK;
}

int or_page_summaries_f64(const uint16_t *k_pool, int num_pages, const int32_t *page_ids, int n,
                          int Hkv, int ps, int d, int dtype, double *summ) {
  for (int i = 0; i < n; ++i) {
    int32_t p = page_ids[i];
    if (p < 0 || p >= num_pages) return OR_EBADPAGE;
    for (int h = 0; h < Hkv; ++h)
      for (int c = 0; c < d; ++c) {
        double acc = 0.0, mn = INFINITY, mx = -INFINITY;
        for (int t = 0; t < ps; ++t) {
          double x = cv(k_pool[(((size_t)p * Hkv + h) * ps + t) * d + c], dtype);
          acc += x;
          if (x < mn) mn = x;
          if (x > mx) mx = x;
        }
        double *s = summ + ((size_t)p * Hkv + h) * 3 * d;
        s[c] = acc / ps;
        s[d + c] = mn;
        s[2 * d + c] = mx;
      }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Page scores.  For summary u (fast, slow) and logical page j of b:         */
/*   S_u(j) = sum_h sum_c [ u_hc * mean_jhc + max(u_hc * min_jhc, u_hc * max_jhc) ]
 * -- the mean-key dot product plus the channel-wise min/max bound on the    */
/* largest logit in the page.  scores [B][max_pages][2]; entries j >= np_b    */
/* are -inf; rows of inactive sequences are left untouched.                  */
/* ------------------------------------------------------------------------ */

/* fp32 order, stated as 32 lanes: lane l owns channels l*CPL .. l*CPL+CPL-1
 * (CPL = d/32).  acc_l = 0; for h ascending, for i ascending:
 *   term = (u*mean) + max(u*min, u*max)   [three rounded products, one sum]
 *   acc_l = acc_l + term.
 * Then for s = 16, 8, 4, 2, 1: acc_l <- acc_l + acc_{l xor s} for every l at
 * once; the score is acc_0.                                                 */
int or_score_pages_f32(const float *ema, const float *summ, int num_pages, const int32_t *table,
                       int max_pages, const int32_t *seq_lens, const uint8_t *active, int B,
                       int Hkv, int d, int ps, float *scores) {
  if (d % 32) return OR_EINVAL;
  int CPL = d / 32;
  for (int b = 0; b < B; ++b) {
    if (active && !active[b]) continue;
    int64_t np = ceil_div64(seq_lens[b], ps);
    for (int j = 0; j < max_pages; ++j) {
      for (int u = 0; u < 2; ++u) {
        float *out = &scores[((size_t)b * max_pages + j) * 2 + u];
        if (j >= np) {
          *out = -INFINITY;
          continue;
        }
        int32_t p = table[(size_t)b * max_pages + j];
        if (p < 0 || p >= num_pages) return OR_EBADPAGE;
        float acc[32], nxt[32];
        for (int l = 0; l < 32; ++l) {
          acc[l] = 0.0f;
          for (int h = 0; h < Hkv; ++h)
            for (int i = 0; i < CPL; ++i) {
              int c = l * CPL + i;
              float uu = ema[(((size_t)b * 2 + u) * Hkv + h) * d + c];
              const float *s = summ + ((size_t)p * Hkv + h) * 3 * d;
              float tm = uu * s[c];
              float ta = uu * s[d + c];
              float tb = uu * s[2 * d + c];
              float term = tm + (ta > tb ? ta : tb);
              acc[l] = acc[l] + term;
            }
        }
        for (int sft = 16; sft >= 1; sft >>= 1) {
          for (int l = 0; l < 32; ++l) nxt[l] = acc[l] + acc[l ^ sft];
          memcpy(acc, nxt, sizeof(acc));
        }
        *out = acc[0];
      }
    }
  }
  return OR_OK;
}

int or_score_pages_f64(const double *ema, const double *summ, int num_pages, const int32_t *table,
                       int max_pages, const int32_t *seq_lens, const uint8_t *active, int B,
                       int Hkv, int d, int ps, double *scores) {
  for (int b = 0; b < B; ++b) {
    if (active && !active[b]) continue;
    int64_t np = ceil_div64(seq_lens[b], ps);
    for (int j = 0; j < max_pages; ++j)
      for (int u = 0; u < 2; ++u) {
        double *out = &scores[((size_t)b * max_pages + j) * 2 + u];
        if (j >= np) {
          *out = -INFINITY;
          continue;
        }
        int32_t p = table[(size_t)b * max_pages + j];
        if (p < 0 || p >= num_pages) return OR_EBADPAGE;
        double acc = 0.0;
        for (int h = 0; h < Hkv; ++h)
          for (int c = 0; c < d; ++c) {
            double uu = ema[(((size_t)b * 2 + u) * Hkv + h) * d + c];
            const double *s = summ + ((size_t)p * Hkv + h) * 3 * d;
            double ta = uu * s[d + c], tb = uu * s[2 * d + c];
            acc += uu * s[c] + (ta > tb ? ta : tb);
          }
        *out = acc;
      }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Page selection: top-k retention, forced pages, compress-or-grow [GP].     */
/* ------------------------------------------------------------------------ */

typedef struct {
  int j;
  float key;
} Cand;

/* Order for "top": larger key first; equal keys -> lower logical page first. */
static int cand_cmp(const void *x, const void *y) {
  const Cand *a = (const Cand *)x, *b = (const Cand *)y;
  if (a->key > b->key) return -1;
  if (a->key < b->key) return 1;
  return a->j < b->j ? -1 : (a->j > b->j ? 1 : 0);
}

/* Marks sel[j] = 1 for the k best of the candidates (k clipped to [0, n]). */
static void top_k(const int *cands, int n, const float *key, int k, uint8_t *sel) {
  Cand *v = (Cand *)malloc(sizeof(Cand) * (n > 0 ? n : 1));
  for (int i = 0; i < n; ++i) {
    v[i].j = cands[i];
    v[i].key = key[cands[i]];
  }
  qsort(v, n, sizeof(Cand), cand_cmp);
  if (k > n) k = n;
  for (int i = 0; i < k; ++i) sel[v[i].j] = 1;
  free(v);
}

#define OR_SELECT_TOPK 0
#define OR_SELECT_BOUNDARY 1

/* For every sequence b (n = ceil(L_b/ps) resident pages):
 *   F = {j < n_first} U {j >= n - n_last} (forced), C = the other pages.
 *   R(j) = S_fast(j) + S_slow(j) (one fp32 add).
 * mode TOPK (inactive rows: keep everything):
 *   keep = F U top_k(C, R) with k = budget[b] - |F|.
 * mode BOUNDARY (active rows are at a capacity boundary):
 *   each summary's attention working set is its top w pages of C, with
 *   w = ceil(ws_frac * |C|) (fp32, clipped to [1, |C|]);
 *   W_f = top_w(C, S_fast), W_s = top_w(C, S_slow), drift D = |W_f \ W_s|;
 *   wants_grow = D > delta * w (fp32) -- the recent working set has moved
 *   beyond the long-term one (demand is widening); with C empty nothing can be
 *   evicted and the sequence always wants to grow.
 *   Grows are granted in ascending b while granted < free_count; a granted
 *   sequence keeps every page, grow[b] = 1 and budget[b] += 1.  Otherwise
 *   keep = F U top_k(C, R) with k = n - 1 - |F| (one page evicted).
 * keep_mask [B][max_pages] (1 = keep; 0 for j >= n); grow [B]; drift [B]. */
int or_select_pages(const float *scores, const int32_t *seq_lens, const uint8_t *active,
                    int32_t *budget, int B, int max_pages, int ps, int n_first, int n_last,
                    float delta, float ws_frac, int mode, int free_count, uint8_t *keep_mask,
                    uint8_t *grow, int32_t *drift) {
  if (mode != OR_SELECT_TOPK && mode != OR_SELECT_BOUNDARY) return OR_EINVAL;
  float *sf = (float *)malloc(sizeof(float) * max_pages);
  float *ss = (float *)malloc(sizeof(float) * max_pages);
  float *rr = (float *)malloc(sizeof(float) * max_pages);
  int *cands = (int *)malloc(sizeof(int) * max_pages);
  uint8_t *wf = (uint8_t *)malloc(max_pages);
  uint8_t *ws = (uint8_t *)malloc(max_pages);
  int granted = 0;
  for (int b = 0; b < B; ++b) {
    int n = (int)ceil_div64(seq_lens[b], ps);
    uint8_t *keep = keep_mask + (size_t)b * max_pages;
    memset(keep, 0, max_pages);
    grow[b] = 0;
    if (drift) drift[b] = 0;
    int is_active = active ? active[b] : 1;
    if (!is_active) {
      for (int j = 0; j < n; ++j) keep[j] = 1;
      continue;
    }
    int nc = 0, nf = 0;
    for (int j = 0; j < n; ++j) {
      const float *sc = scores + ((size_t)b * max_pages + j) * 2;
      sf[j] = sc[0];
      ss[j] = sc[1];
      rr[j] = sc[0] + sc[1];
      int forced = (j < n_first) || (j >= n - n_last);
      if (forced) {
        keep[j] = 1;
        ++nf;
      } else {
        cands[nc++] = j;
      }
    }
    if (mode == OR_SELECT_TOPK) {
      int k = budget[b] - nf;
      if (k < 0) k = 0;
      top_k(cands, nc, rr, k, keep);
      continue;
    }
    int k = n - 1 - nf;
    if (k < 0) k = 0;
    int wants;
    if (nc == 0) {
      wants = 1;
    } else {
      int w = (int)ceilf(ws_frac * (float)nc);
      if (w < 1) w = 1;
      if (w > nc) w = nc;
      memset(wf, 0, max_pages);
      memset(ws, 0, max_pages);
      top_k(cands, nc, sf, w, wf);
      top_k(cands, nc, ss, w, ws);
      int D = 0;
      for (int i = 0; i < nc; ++i) D += wf[cands[i]] && !ws[cands[i]];
      if (drift) drift[b] = D;
      float thr = delta * (float)w;
      wants = (float)D > thr;
    }
    if (wants && granted < free_count) {
      ++granted;
      grow[b] = 1;
      budget[b] += 1;
      for (int j = 0; j < n; ++j) keep[j] = 1;
    } else {
      top_k(cands, nc, rr, k, keep);
    }
  }
  free(sf);
  free(ss);
  free(rr);
  free(cands);
  free(wf);
  free(ws);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Compaction: stable gather of kept tokens into fewer pages [GP]; the free  */
/* list is the integer stack of fixed-size blocks [EKV, section 2].          */
/* ------------------------------------------------------------------------ */

/* Definition.  For each b the kept tokens (t < L_b with keep bit set; with a
 * page mask the bit of page t/ps) in ascending order fill new logical slots
 * 0, 1, 2, ...; new page m holds slots [m*ps, (m+1)*ps).  New page m reuses
 * old page j (no copy) when each of its cnt_m tokens is token j*ps + s at the
 * same slot s; otherwise it takes a fresh page.  Fresh pages are popped from
 * the free-list top in (b, m) order (the i-th pop reads
 * free_list[top - 1 - i]); if the pops exceed the stack nothing changes and
 * -3 is returned.  The K/V of every token placed in a fresh page is copied
 * there (all KV heads).  Old pages that are not reused are then pushed in
 * (b, j) order.  The row is rewritten (-1 padded) and L_b = kept count.
 * free_list has room for num_pages entries.
 * Shared pages (prefix caching, GrowPage Abstract): when refcnt is not NULL
 * it holds each pool page's number of block-table references.  A fresh page
 * gets count 1; each old page that is not reused loses one reference, in
 * (b, j) order, and is pushed when its count reaches 0.  Kept pages are never
 * written, so a page another sequence still uses is never modified.          */
int or_compact(int32_t *table, int max_pages, int32_t *seq_lens, const uint8_t *keep,
               int token_granular, uint16_t *k_pool, uint16_t *v_pool, int num_pages,
               int32_t *free_list, int32_t *free_top, int32_t *refcnt, int B, int Hkv, int d,
               int ps) {
  int64_t mask_w = token_granular ? (int64_t)max_pages * ps : max_pages;
  int64_t total_fresh = 0;
  /* pass 1: count fresh pages */
  int64_t **kept = (int64_t **)calloc(B, sizeof(int64_t *));
  int64_t *nkept = (int64_t *)calloc(B, sizeof(int64_t));
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b];
    kept[b] = (int64_t *)malloc(sizeof(int64_t) * (L > 0 ? L : 1));
    for (int64_t t = 0; t < L; ++t) {
      int64_t bit = token_granular ? t : t / ps;
      if (keep[(size_t)b * mask_w + bit]) kept[b][nkept[b]++] = t;
    }
    int64_t nnew = ceil_div64(nkept[b], ps);
    for (int64_t m = 0; m < nnew; ++m) {
      int64_t cnt = nkept[b] - m * ps < ps ? nkept[b] - m * ps : ps;
      int64_t t0 = kept[b][m * ps];
      int reuse = (t0 % ps) == 0;
      for (int64_t s = 0; s < cnt && reuse; ++s) reuse = kept[b][m * ps + s] == t0 + s;
      if (!reuse) ++total_fresh;
    }
  }
  int rc = OR_OK;
  if (total_fresh > *free_top) {
    rc = OR_ENOSPACE;
    goto out;
  }
  {
    int64_t top = *free_top, pops = 0;
    int64_t row_elems = (int64_t)Hkv * ps * d; /* elements of one pool page */
    int32_t *newrow = (int32_t *)malloc(sizeof(int32_t) * max_pages);
    uint8_t *reused = (uint8_t *)malloc(max_pages);
    int32_t *freed = (int32_t *)malloc(sizeof(int32_t) * ((size_t)B * max_pages + 1));
    int64_t nfreed = 0;
    for (int b = 0; b < B; ++b) {
      int64_t L = seq_lens[b];
      int64_t np_old = ceil_div64(L, ps);
      int64_t nnew = ceil_div64(nkept[b], ps);
      memset(reused, 0, max_pages);
      for (int j = 0; j < max_pages; ++j) newrow[j] = -1;
      for (int64_t m = 0; m < nnew; ++m) {
        int64_t cnt = nkept[b] - m * ps < ps ? nkept[b] - m * ps : ps;
        int64_t t0 = kept[b][m * ps];
        int reuse = (t0 % ps) == 0;
        for (int64_t s = 0; s < cnt && reuse; ++s) reuse = kept[b][m * ps + s] == t0 + s;
        if (reuse) {
          newrow[m] = table[(size_t)b * max_pages + t0 / ps];
          reused[t0 / ps] = 1;
        } else {
          int32_t fresh = free_list[top - 1 - pops];
          ++pops;
          newrow[m] = fresh;
          if (refcnt) refcnt[fresh] = 1;
          for (int64_t s = 0; s < cnt; ++s) {
            int64_t t = kept[b][m * ps + s];
            int32_t src = table[(size_t)b * max_pages + t / ps];
            for (int h = 0; h < Hkv; ++h) {
              size_t so = ((size_t)src * Hkv + h) * ps * d + (size_t)(t % ps) * d;
              size_t dst = ((size_t)fresh * Hkv + h) * ps * d + (size_t)s * d;
              memcpy(k_pool + dst, k_pool + so, sizeof(uint16_t) * d);
              memcpy(v_pool + dst, v_pool + so, sizeof(uint16_t) * d);
            }
          }
        }
      }
      (void)row_elems;
      for (int64_t j = 0; j < np_old; ++j)
        if (!reused[j]) freed[nfreed++] = table[(size_t)b * max_pages + j];
      memcpy(table + (size_t)b * max_pages, newrow, sizeof(int32_t) * max_pages);
      seq_lens[b] = (int32_t)nkept[b];
    }
    top -= pops;
    /* With shared pages, a freed reference only drops the page's count; the
     * page returns to the free list when its last reference goes. */
    for (int64_t i = 0; i < nfreed; ++i) {
      if (refcnt) {
        refcnt[freed[i]] -= 1;
        if (refcnt[freed[i]] != 0) continue;
      }
      free_list[top++] = freed[i];
    }
    *free_top = (int32_t)top;
    free(newrow);
    free(reused);
    free(freed);
  }
out:
  for (int b = 0; b < B; ++b) free(kept[b]);
  free(kept);
  free(nkept);
  (void)num_pages;
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Append: write the new token's K/V at slot L_b % ps of page             */
/* block_table[b][L_b / ps]; when L_b % ps == 0 the page is first popped     */
/* from the free list (pops in ascending b).  Then L_b += 1.  Nothing        */
/* changes on an error: a full row (-6), else a bad page id in use or about  */
/* to be popped (-2), else too few free pages (-3).                          */
/* k_new, v_new: [B][Hkv][d].                                                 */
/* Shared pages: with refcnt (not NULL), a sequence whose last page is       */
/* partly filled and shared (count > 1) first copies it (copy-on-write): it  */
/* pops a fresh page in the same ascending-b order, copies the page's first  */
/* L_b % ps slots (K and V, all heads) there, points its table entry at it,  */
/* drops one reference from the shared page; popped pages get count 1.      */
int or_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool, uint16_t *v_pool,
              int num_pages, int32_t *table, int max_pages, int32_t *seq_lens, int32_t *free_list,
              int32_t *free_top, int32_t *refcnt, int B, int Hkv, int d, int ps) {
  /* checks first, in this order of precedence: a full row, a bad page id (one
   * in use, or one that would be popped), too few free pages */
  int64_t need = 0;
  int full = 0, bad = 0;
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b];
    if (L < 0) {
      bad = 1;
    } else if (L % ps == 0) {
      if (L / ps >= max_pages) full = 1;
      ++need;
    } else {
      int32_t p = table[(size_t)b * max_pages + L / ps];
      if (p < 0 || p >= num_pages) bad = 1;
      else if (refcnt && refcnt[p] > 1) ++need;
    }
  }
  if (need <= *free_top)
    for (int64_t i = 0; i < need; ++i) {
      int32_t p = free_list[*free_top - 1 - i];
      if (p < 0 || p >= num_pages) bad = 1;
    }
  if (full) return OR_EFULL;
  if (bad) return OR_EBADPAGE;
  if (need > *free_top) return OR_ENOSPACE;
  int64_t top = *free_top;
  size_t tile = (size_t)ps * d; /* elements of one (page, head) tile */
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b];
    int32_t *slot = &table[(size_t)b * max_pages + L / ps];
    if (L % ps == 0) {
      *slot = free_list[--top];
      if (refcnt) refcnt[*slot] = 1;
    } else if (refcnt && refcnt[*slot] > 1) {
      int32_t old = *slot, fresh = free_list[--top];
      for (int h = 0; h < Hkv; ++h) {
        size_t so = ((size_t)old * Hkv + h) * tile, dst = ((size_t)fresh * Hkv + h) * tile;
        memcpy(k_pool + dst, k_pool + so, sizeof(uint16_t) * (size_t)(L % ps) * d);
        memcpy(v_pool + dst, v_pool + so, sizeof(uint16_t) * (size_t)(L % ps) * d);
      }
      refcnt[old] -= 1;
      refcnt[fresh] = 1;
      *slot = fresh;
    }
    int32_t p = *slot;
    for (int h = 0; h < Hkv; ++h) {
      size_t dst = (((size_t)p * Hkv + h) * ps + (size_t)(L % ps)) * d;
      memcpy(k_pool + dst, k_new + ((size_t)b * Hkv + h) * d, sizeof(uint16_t) * d);
      memcpy(v_pool + dst, v_new + ((size_t)b * Hkv + h) * d, sizeof(uint16_t) * d);
    }
    seq_lens[b] = (int32_t)(L + 1);
  }
  *free_top = (int32_t)top;
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Which sequences take part in a budgeting pass.                            */
/*   mode 0 (initial fit): active iff ceil(L_b/ps) > budget[b];              */
/*   mode 1 (capacity boundary): active iff L_b > 0, L_b % ps == 0 and       */
/*           L_b / ps >= budget[b] -- the last page is full, the next token  */
/*           needs a page, and the sequence already holds its budget [GP].   */
/* ------------------------------------------------------------------------ */
int or_mark_active(const int32_t *seq_lens, const int32_t *budget, int B, int ps, int mode,
                   uint8_t *active) {
  if (mode != 0 && mode != 1) return OR_EINVAL;
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b];
    if (mode == 0)
      active[b] = ceil_div64(L, ps) > budget[b];
    else
      active[b] = L > 0 && L % ps == 0 && L / ps >= budget[b];
  }
  return OR_OK;
}
