/*
 * msa_oracle.c -- plain, slow, fp64 CPU oracle for the block-sparse paged
 * decode path.  TEST INFRASTRUCTURE ONLY (see msa_oracle.h).
 *
 * Every function follows a stated definition, step by step, with no tiling,
 * fusion or reordering.  Rows are shared out across plain pthreads; each row
 * is computed by the same sequential loop whatever the thread count.
 *
 * Sources of the definitions (page titles of the MiniMax-M3 sparse-attention
 * pages, then the section):
 *   - 128-token index blocks, CPU-side block count ceil(len/128):
 *       vLLM PR 56170 page, "Key source snippets" (metadata build).
 *   - row position = context_len + j, cu_seqlens_k prefix with [0] = 0:
 *       vLLM PR 56170 page, "Implementation breakdown" items 1 and 3.
 *   - index scoring + top-k writing the page-16 sparse table and the
 *       per-row context length:  vLLM PR 54682 page, "Implementation
 *       breakdown" items 1 and 4.
 *   - page-16 view of the page-128 cache, sparse-table build with bounded
 *       zero fill:  vLLM PR 47287 page, "Implementation breakdown" item 3
 *       and "Review highlights" (out-of-bounds zero-fill fix).
 *   - FP8 k_scale / v_scale, scalar or per_token_head:  vLLM PR 47287 page,
 *       "Implementation breakdown" item 2 and "Key files" (fp8 scale test).
 *   - learnable per-head sink, natural-log LSE, fp32 [num_heads] sinks:
 *       vLLM PR 54404 page, "Features and motivation", "Key source
 *       snippets" (LSE op docstring, sink validation).
 *   - KV insert with skip_index (the step before the path): vLLM PR 47287
 *       page, "Implementation breakdown" item 1 (index-reuse layers skip the
 *       index-cache write) and item 5 (separate K/V page layout).
 *   - where the pages are silent (block score = max over the block's valid
 *       tokens of the raw index dot product, ties to the lower block index,
 *       ascending table order, sink in the denominator, empty row -> O = 0):
 *       the readings listed in the design notes of this repository.
 *
 * FP8: OCP 8-bit floating point specification, E4M3 ("fn") encoding.
 */
#include "msa_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK 128
#define PAGE16 16

/* ---------------------------------------------------------------- values */

double orc_bf16_value(uint16_t bits) {
  /* bf16 is the top half of an IEEE binary32 */
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double orc_fp8_e4m3_value(uint8_t code) {
  /* OCP E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
   * Exponent field 0 encodes subnormals 2^(1-7) * m/8; the single pattern
   * S.1111.111 is NaN; there is no infinity. */
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

static double kv_value(const void* cache, int32_t kv_dtype, int64_t index) {
  if (kv_dtype == 1) return orc_fp8_e4m3_value(((const uint8_t*)cache)[index]);
  return orc_bf16_value(((const uint16_t*)cache)[index]);
}

/* ------------------------------------------------------------- threading */

typedef void (*row_fn)(void* ctx, int32_t r);
typedef struct {
  row_fn fn;
  void* ctx;
  int32_t r0, r1;
} span_t;

static void* run_span(void* arg) {
  span_t* s = (span_t*)arg;
  for (int32_t r = s->r0; r < s->r1; ++r) s->fn(s->ctx, r);
  return NULL;
}

static void for_each_row(int32_t n, int32_t nthreads, row_fn fn, void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n) nthreads = n > 0 ? n : 1;
  if (nthreads == 1) {
    for (int32_t r = 0; r < n; ++r) fn(ctx, r);
    return;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  span_t* sp = (span_t*)malloc(sizeof(span_t) * (size_t)nthreads);
  for (int32_t i = 0; i < nthreads; ++i) {
    sp[i].fn = fn;
    sp[i].ctx = ctx;
    sp[i].r0 = (int32_t)((int64_t)n * i / nthreads);
    sp[i].r1 = (int32_t)((int64_t)n * (i + 1) / nthreads);
    pthread_create(&th[i], NULL, run_span, &sp[i]);
  }
  for (int32_t i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  free(sp);
}

/* ------------------------------------------------------------- geometry */

/* ok codes: 0 = row not scored (uncovered or its request is malformed or
 * has inconsistent lengths); 1 = valid; 2 = scored but its request holds an
 * out-of-range page id, so nothing is selected for it. */
uint32_t orc_row_geometry(const orc_batch* b, int32_t* req, int32_t* pos, int32_t* nb,
                          int32_t* ok) {
  const int32_t R = b->num_reqs, N = b->num_rows;
  const int32_t* cq = b->cu_seqlens_q;
  const int32_t* ck = b->cu_seqlens_k;
  uint32_t st = 0;
  for (int32_t r = 0; r < N; ++r) {
    req[r] = -1;
    pos[r] = -1;
    nb[r] = 0;
    ok[r] = 0;
  }
  /* rows of request q are [cu_q[q], cu_q[q+1]); they must tile [0, N) */
  int monotone = (cq[0] == 0) && (cq[R] == N);
  for (int32_t q = 0; q < R; ++q)
    if (cq[q + 1] < cq[q]) monotone = 0;
  if (!monotone) return ORC_MALFORMED;

  for (int32_t q = 0; q < R; ++q) {
    const int32_t qlen = cq[q + 1] - cq[q];
    const int32_t slen = ck[q + 1] - ck[q];
    const int32_t ctx = b->context_lens[q];
    uint32_t bad = 0;
    if (slen < qlen || ctx < 0 || (int64_t)slen > (int64_t)BLOCK * b->bt_stride) {
      bad = ORC_MALFORMED;
    } else if (ctx + qlen != slen) {
      bad = ORC_BAD_LEN;
    } else {
      const int32_t nbq = (slen + BLOCK - 1) / BLOCK;
      for (int32_t blk = 0; blk < nbq; ++blk) {
        const int32_t page = b->block_table[(int64_t)q * b->bt_stride + blk];
        if (page < 0 || page >= b->num_pages) bad |= ORC_BAD_PAGE;
      }
    }
    st |= bad;
    for (int32_t j = 0; j < qlen; ++j) {
      const int32_t r = cq[q] + j;
      req[r] = q;
      if (bad & (ORC_MALFORMED | ORC_BAD_LEN)) continue;
      pos[r] = ctx + j;
      nb[r] = (pos[r] + 1 + BLOCK - 1) / BLOCK;
      ok[r] = bad ? 2 : 1;
    }
  }
  return st;
}

typedef struct {
  int32_t *req, *pos, *nb, *ok;
} geom_t;

static uint32_t geometry_alloc(const orc_batch* b, geom_t* g) {
  size_t n = (size_t)(b->num_rows > 0 ? b->num_rows : 1);
  g->req = (int32_t*)malloc(n * sizeof(int32_t));
  g->pos = (int32_t*)malloc(n * sizeof(int32_t));
  g->nb = (int32_t*)malloc(n * sizeof(int32_t));
  g->ok = (int32_t*)malloc(n * sizeof(int32_t));
  return orc_row_geometry(b, g->req, g->pos, g->nb, g->ok);
}

static void geometry_free(geom_t* g) {
  free(g->req);
  free(g->pos);
  free(g->nb);
  free(g->ok);
}

/* ---------------------------------------------------------- index score */

typedef struct {
  const orc_batch* b;
  const geom_t* g;
  const uint16_t* idx_q;
  const void* idx_k;      /* bf16 bits, or e4m3 codes when fp8 */
  const float* k_scale;   /* fp8 only: [P, 128, hi] per-token scale, or NULL (1) */
  int32_t fp8;
  int32_t hi, di;
  float* scores;
  int32_t score_stride;
} score_ctx;

/* Value of index-K element d of (page, token tl, head h). */
static double index_k_value(const score_ctx* c, int64_t base, int32_t d) {
  if (c->fp8) return orc_fp8_e4m3_value(((const uint8_t*)c->idx_k)[base + d]);
  return orc_bf16_value(((const uint16_t*)c->idx_k)[base + d]);
}

static void score_row(void* vctx, int32_t r) {
  const score_ctx* c = (const score_ctx*)vctx;
  float* out = c->scores + (int64_t)r * c->score_stride;
  for (int32_t blk = 0; blk < c->score_stride; ++blk) out[blk] = -INFINITY;
  if (c->g->ok[r] == 0) return;
  const int32_t q = c->g->req[r];
  const int32_t pos = c->g->pos[r];
  for (int32_t blk = 0; blk < c->g->nb[r] && blk < c->score_stride; ++blk) {
    const int32_t page = c->b->block_table[(int64_t)q * c->b->bt_stride + blk];
    if (page < 0 || page >= c->b->num_pages) continue; /* unreadable: stays -inf */
    double best = -INFINITY;
    for (int32_t tl = 0; tl < BLOCK; ++tl) {
      const int32_t t = blk * BLOCK + tl;
      if (t > pos) break; /* causal: only tokens at or before the row's position */
      for (int32_t h = 0; h < c->hi; ++h) {
        const uint16_t* qv = c->idx_q + ((int64_t)r * c->hi + h) * c->di;
        const int64_t slot = ((int64_t)page * BLOCK + tl) * c->hi + h;
        double dot = 0.0;
        for (int32_t d = 0; d < c->di; ++d)
          dot += orc_bf16_value(qv[d]) * index_k_value(c, slot * c->di, d);
        if (c->fp8 && c->k_scale) dot *= (double)c->k_scale[slot]; /* dequantised key */
        if (dot > best) best = dot; /* NaN dots never win */
      }
    }
    out[blk] = (float)best;
  }
}

uint32_t orc_index_score(const orc_batch* b, const uint16_t* idx_q, const uint16_t* idx_k,
                         int32_t index_heads, int32_t index_dim, float* scores,
                         int32_t score_stride, int32_t nthreads) {
  geom_t g;
  uint32_t st = geometry_alloc(b, &g);
  score_ctx c = {b, &g, idx_q, idx_k, NULL, 0, index_heads, index_dim, scores, score_stride};
  for_each_row(b->num_rows, nthreads, score_row, &c);
  geometry_free(&g);
  return st;
}

uint32_t orc_index_score_fp8(const orc_batch* b, const uint16_t* idx_q, const uint8_t* idx_k,
                             const float* k_scale, int32_t index_heads, int32_t index_dim,
                             float* scores, int32_t score_stride, int32_t nthreads) {
  geom_t g;
  uint32_t st = geometry_alloc(b, &g);
  score_ctx c = {b, &g, idx_q, idx_k, k_scale, 1, index_heads, index_dim, scores, score_stride};
  for_each_row(b->num_rows, nthreads, score_row, &c);
  geometry_free(&g);
  return st;
}

/* --------------------------------------------------- top-k + table build */

typedef struct {
  float score;
  int32_t block;
} cand_t;

/* Total order used for selection: higher score first; a NaN score ranks
 * below every number; equal scores go to the lower block index. */
static int cand_cmp(const void* pa, const void* pb) {
  const cand_t* a = (const cand_t*)pa;
  const cand_t* b = (const cand_t*)pb;
  const int an = isnan(a->score), bn = isnan(b->score);
  if (an != bn) return an ? 1 : -1;
  if (!an && a->score != b->score) return a->score > b->score ? -1 : 1;
  return (a->block > b->block) - (a->block < b->block);
}

static int int_cmp(const void* pa, const void* pb) {
  const int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

typedef struct {
  const orc_batch* b;
  const geom_t* g;
  const float* scores;
  int32_t score_stride, topk;
  int32_t *topk_idx, *tbl;
  int32_t tbl_stride;
  int32_t* sparse_len;
} topk_ctx;

static void topk_row(void* vctx, int32_t r) {
  const topk_ctx* c = (const topk_ctx*)vctx;
  int32_t* sel = c->topk_idx + (int64_t)r * c->topk;
  int32_t* row = c->tbl + (int64_t)r * c->tbl_stride;
  for (int32_t i = 0; i < c->topk; ++i) sel[i] = -1;
  for (int32_t i = 0; i < c->tbl_stride; ++i) row[i] = 0;
  c->sparse_len[r] = 0;
  if (c->g->ok[r] != 1) return;
  const int32_t q = c->g->req[r];
  const int32_t L = c->g->pos[r] + 1; /* visible tokens */
  const int32_t n = c->g->nb[r];
  const int32_t m = n < c->topk ? n : c->topk;

  /* 1. rank every candidate block by (score desc, block asc); keep the first m */
  cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
  for (int32_t blk = 0; blk < n; ++blk) {
    cand[blk].score = c->scores[(int64_t)r * c->score_stride + blk];
    cand[blk].block = blk;
  }
  qsort(cand, (size_t)n, sizeof(cand_t), cand_cmp);
  for (int32_t i = 0; i < m; ++i) sel[i] = cand[i].block;
  free(cand);
  /* 2. the selected blocks go out in ascending block order */
  qsort(sel, (size_t)m, sizeof(int32_t), int_cmp);

  /* 3. expand each selected page-128 block into its page-16 pages; only
   *    pages holding at least one visible token are written */
  int32_t total = 0;
  for (int32_t i = 0; i < m; ++i) {
    const int32_t blk = sel[i];
    const int32_t page = c->b->block_table[(int64_t)q * c->b->bt_stride + blk];
    int32_t valid = L - blk * BLOCK;
    if (valid > BLOCK) valid = BLOCK;
    const int32_t sub = (valid + PAGE16 - 1) / PAGE16;
    for (int32_t j = 0; j < sub; ++j) row[8 * i + j] = 8 * page + j;
    total += valid;
  }
  c->sparse_len[r] = total;
}

uint32_t orc_topk_build_table(const orc_batch* b, const float* scores, int32_t score_stride,
                              int32_t topk, int32_t* topk_idx, int32_t* sparse_tbl,
                              int32_t tbl_stride, int32_t* sparse_len, int32_t nthreads) {
  geom_t g;
  uint32_t st = geometry_alloc(b, &g);
  topk_ctx c = {b, &g, scores, score_stride, topk, topk_idx, sparse_tbl, tbl_stride, sparse_len};
  for_each_row(b->num_rows, nthreads, topk_row, &c);
  geometry_free(&g);
  return st;
}

/* ------------------------------------------------------------ attention */

/* One softmax-attention head over an explicit token list (flat token ids in
 * the [P*128] token space; token id x lives at page-16 x/16, slot x%16).
 *   s_t  = softmax_scale * k_scale_t * (q . k_t)
 *   m    = max(max_t s_t, sink)
 *   den  = sum_t exp(s_t - m) + exp(sink - m)
 *   O    = sum_t exp(s_t - m) * v_scale_t * v_t / den
 *   LSE  = m + ln(den)
 * With no sink the sink terms are absent; with no token and no sink the row
 * is empty: O = 0, LSE = -inf. */
typedef struct {
  int32_t hq, hkv, d;
  const uint16_t* q;
  const void *k, *v;
  int32_t kv_dtype, scale_mode;
  const float *k_scale, *v_scale, *sinks;
  double softmax_scale;
} attn_common;

static double token_scale(const float* scale, int32_t mode, int64_t token, int32_t hkv,
                          int32_t kvh) {
  if (mode == 1) return (double)scale[0];
  if (mode == 2) return (double)scale[token * hkv + kvh];
  return 1.0;
}

static void attend_head(const attn_common* a, int32_t r, int32_t h, const int64_t* tokens,
                        int32_t n, double* s, double* out, double* lse) {
  const int32_t group = a->hq / a->hkv;
  const int32_t kvh = h / group;
  const uint16_t* qh = a->q + ((int64_t)r * a->hq + h) * a->d;
  const int has_sink = a->sinks != NULL;
  const double sink = has_sink ? (double)a->sinks[h] : -INFINITY;
  double m = -INFINITY;
  for (int32_t t = 0; t < n; ++t) {
    const int64_t base = (tokens[t] * a->hkv + kvh) * a->d;
    double dot = 0.0;
    for (int32_t d = 0; d < a->d; ++d)
      dot += orc_bf16_value(qh[d]) * kv_value(a->k, a->kv_dtype, base + d);
    s[t] = a->softmax_scale * token_scale(a->k_scale, a->scale_mode, tokens[t], a->hkv, kvh) * dot;
    if (s[t] > m) m = s[t];
  }
  if (has_sink && sink > m) m = sink;
  for (int32_t d = 0; d < a->d; ++d) out[d] = 0.0;
  if (m == -INFINITY) { /* empty row */
    *lse = -INFINITY;
    return;
  }
  double den = has_sink ? exp(sink - m) : 0.0;
  for (int32_t t = 0; t < n; ++t) {
    const double p = exp(s[t] - m);
    den += p;
    const double pv = p * token_scale(a->v_scale, a->scale_mode, tokens[t], a->hkv, kvh);
    const int64_t base = (tokens[t] * a->hkv + kvh) * a->d;
    for (int32_t d = 0; d < a->d; ++d) out[d] += pv * kv_value(a->v, a->kv_dtype, base + d);
  }
  for (int32_t d = 0; d < a->d; ++d) out[d] /= den;
  *lse = m + log(den);
}

typedef struct {
  attn_common a;
  const int32_t *tbl, *len;
  int32_t tbl_stride, num_pages16;
  double *out, *lse;
  uint32_t* row_status;
} sparse_ctx;

static void sparse_row(void* vctx, int32_t r) {
  const sparse_ctx* c = (const sparse_ctx*)vctx;
  int32_t n = c->len[r];
  int poisoned = (n < 0) || ((int64_t)n > (int64_t)PAGE16 * c->tbl_stride);
  if (!poisoned) {
    for (int32_t t = 0; t < n; t += PAGE16) {
      const int32_t e = c->tbl[(int64_t)r * c->tbl_stride + t / PAGE16];
      if (e < 0 || e >= c->num_pages16) poisoned = 1;
    }
  }
  c->row_status[r] = poisoned ? ORC_BAD_TABLE : 0u;
  if (poisoned) n = 0; /* a poisoned row is computed as an empty row */
  int64_t* tokens = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int32_t t = 0; t < n; ++t) {
    const int32_t e = c->tbl[(int64_t)r * c->tbl_stride + t / PAGE16];
    tokens[t] = (int64_t)e * PAGE16 + t % PAGE16;
  }
  for (int32_t h = 0; h < c->a.hq; ++h)
    attend_head(&c->a, r, h, tokens, n, s, c->out + ((int64_t)r * c->a.hq + h) * c->a.d,
                c->lse + (int64_t)r * c->a.hq + h);
  free(tokens);
  free(s);
}

uint32_t orc_sparse_attn(int32_t num_rows, int32_t hq, int32_t hkv, int32_t head_dim,
                         const uint16_t* q, const void* k_cache, const void* v_cache,
                         int32_t kv_dtype, int32_t num_pages16, int32_t scale_mode,
                         const float* k_scale, const float* v_scale, const int32_t* sparse_tbl,
                         int32_t tbl_stride, const int32_t* sparse_len, const float* sinks,
                         double softmax_scale, double* out, double* lse, int32_t nthreads) {
  sparse_ctx c;
  c.a.hq = hq;
  c.a.hkv = hkv;
  c.a.d = head_dim;
  c.a.q = q;
  c.a.k = k_cache;
  c.a.v = v_cache;
  c.a.kv_dtype = kv_dtype;
  c.a.scale_mode = scale_mode;
  c.a.k_scale = k_scale;
  c.a.v_scale = v_scale;
  c.a.sinks = sinks;
  c.a.softmax_scale = softmax_scale;
  c.tbl = sparse_tbl;
  c.len = sparse_len;
  c.tbl_stride = tbl_stride;
  c.num_pages16 = num_pages16;
  c.out = out;
  c.lse = lse;
  c.row_status = (uint32_t*)calloc((size_t)(num_rows > 0 ? num_rows : 1), sizeof(uint32_t));
  for_each_row(num_rows, nthreads, sparse_row, &c);
  uint32_t st = 0;
  for (int32_t r = 0; r < num_rows; ++r) st |= c.row_status[r];
  free(c.row_status);
  return st;
}

typedef struct {
  attn_common a;
  const orc_batch* b;
  const geom_t* g;
  double *out, *lse;
} dense_ctx;

static void dense_row(void* vctx, int32_t r) {
  const dense_ctx* c = (const dense_ctx*)vctx;
  const int32_t n = (c->g->ok[r] == 1) ? c->g->pos[r] + 1 : 0;
  const int32_t q = c->g->req[r];
  int64_t* tokens = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int32_t t = 0; t < n; ++t) {
    const int32_t page = c->b->block_table[(int64_t)q * c->b->bt_stride + t / BLOCK];
    tokens[t] = (int64_t)page * BLOCK + t % BLOCK;
  }
  for (int32_t h = 0; h < c->a.hq; ++h)
    attend_head(&c->a, r, h, tokens, n, s, c->out + ((int64_t)r * c->a.hq + h) * c->a.d,
                c->lse + (int64_t)r * c->a.hq + h);
  free(tokens);
  free(s);
}

uint32_t orc_dense_attn(const orc_batch* b, int32_t hq, int32_t hkv, int32_t head_dim,
                        const uint16_t* q, const void* k_cache, const void* v_cache,
                        int32_t kv_dtype, int32_t scale_mode, const float* k_scale,
                        const float* v_scale, const float* sinks, double softmax_scale,
                        double* out, double* lse, int32_t nthreads) {
  geom_t g;
  uint32_t st = geometry_alloc(b, &g);
  dense_ctx c;
  c.a.hq = hq;
  c.a.hkv = hkv;
  c.a.d = head_dim;
  c.a.q = q;
  c.a.k = k_cache;
  c.a.v = v_cache;
  c.a.kv_dtype = kv_dtype;
  c.a.scale_mode = scale_mode;
  c.a.k_scale = k_scale;
  c.a.v_scale = v_scale;
  c.a.sinks = sinks;
  c.a.softmax_scale = softmax_scale;
  c.b = b;
  c.g = &g;
  c.out = out;
  c.lse = lse;
  for_each_row(b->num_rows, nthreads, dense_row, &c);
  geometry_free(&g);
  return st;
}

/* ------------------------------------------------------------ KV insert */

uint8_t orc_fp8_e4m3_encode(float x) {
  /* Brute force over the 127 finite magnitudes of the format: the nearest
   * value wins; on a tie the even code (mantissa LSB 0) wins; anything at or
   * beyond the largest finite magnitude saturates to it. */
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  uint8_t best = 0;
  double best_diff = INFINITY;
  for (int code = 0; code <= 0x7E; ++code) {
    const double d = fabs(a - orc_fp8_e4m3_value((uint8_t)code));
    if (d < best_diff || (d == best_diff && (code & 1) == 0)) {
      best = (uint8_t)code;
      best_diff = d;
    }
  }
  return (uint8_t)(sign | best);
}

static void quantize_row(const uint16_t* src, int32_t d, uint8_t* dst, float* scale_out,
                         int32_t scale_mode, float given_scale) {
  float s = 1.0f;
  if (scale_mode == 2) {
    float amax = 0.0f;
    for (int32_t i = 0; i < d; ++i) {
      const float v = fabsf((float)orc_bf16_value(src[i]));
      if (v > amax) amax = v;
    }
    s = amax > 0.0f ? amax / 448.0f : 1.0f;
    *scale_out = s;
  } else if (scale_mode == 1) {
    s = given_scale;
  }
  for (int32_t i = 0; i < d; ++i) {
    const float q = (float)orc_bf16_value(src[i]) / s; /* fp32 division */
    dst[i] = orc_fp8_e4m3_encode(q);
  }
}

uint32_t orc_kv_insert(const orc_batch* b, int32_t hkv, int32_t head_dim, const uint16_t* k_new,
                       const uint16_t* v_new, int32_t index_heads, int32_t index_dim,
                       const uint16_t* idx_new, void* k_cache, void* v_cache,
                       void* idx_k_cache, int32_t kv_dtype, int32_t scale_mode,
                       float* k_scale, float* v_scale, int32_t skip_index, int32_t idx_dtype,
                       float* idx_scale) {
  geom_t g;
  const uint32_t st = geometry_alloc(b, &g);
  for (int32_t r = 0; r < b->num_rows; ++r) {
    if (g.ok[r] != 1) continue;
    const int32_t q = g.req[r];
    const int32_t pos = g.pos[r];
    const int32_t page = b->block_table[(int64_t)q * b->bt_stride + pos / BLOCK];
    const int64_t token = (int64_t)page * BLOCK + pos % BLOCK; /* flat slot in [P*128] */
    for (int32_t h = 0; h < hkv; ++h) {
      const int64_t src = ((int64_t)r * hkv + h) * head_dim;
      const int64_t dst = (token * hkv + h) * head_dim;
      if (kv_dtype == 1) {
        float ks = 1.0f, vs = 1.0f;
        quantize_row(k_new + src, head_dim, (uint8_t*)k_cache + dst, &ks, scale_mode,
                     scale_mode == 1 ? k_scale[0] : 1.0f);
        quantize_row(v_new + src, head_dim, (uint8_t*)v_cache + dst, &vs, scale_mode,
                     scale_mode == 1 ? v_scale[0] : 1.0f);
        if (scale_mode == 2) {
          k_scale[token * hkv + h] = ks;
          v_scale[token * hkv + h] = vs;
        }
      } else {
        memcpy((uint16_t*)k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)head_dim);
        memcpy((uint16_t*)v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)head_dim);
      }
    }
    if (!skip_index && idx_dtype == 1) {
      /* e4m3 index keys, per token and index head: the per-token-head rule
       * when scales are kept, else scale 1 */
      for (int32_t h = 0; h < index_heads; ++h) {
        const int64_t src = ((int64_t)r * index_heads + h) * index_dim;
        const int64_t dst = (token * index_heads + h) * index_dim;
        float s = 1.0f;
        quantize_row(idx_new + src, index_dim, (uint8_t*)idx_k_cache + dst, &s,
                     idx_scale ? 2 : 0, 1.0f);
        if (idx_scale) idx_scale[token * index_heads + h] = s;
      }
    } else if (!skip_index) {
      const int64_t n = (int64_t)index_heads * index_dim;
      memcpy((uint16_t*)idx_k_cache + token * n, idx_new + (int64_t)r * n,
             sizeof(uint16_t) * (size_t)n);
    }
  }
  geometry_free(&g);
  return st;
}

/* ------------------------------------------------------ sparse MLA decode */

/* One latent KV row per token: kv[t, 0:dqk] is the key (latent part + rope
 * part), kv[t, 0:dv] the value.  Row r attends over the token ids
 * kv_indices[kv_indptr[r] .. kv_indptr[r+1]) with the same softmax, sink and
 * natural-log LSE as attend_head.  FP8 operands ("Attention sinks for ROCm
 * AITER sparse MLA", "Key source snippets": the decode op's q_scale and
 * kv_scale): an e4m3 query element is q_scale * code, an e4m3 cache element
 * kv_scale * code, for the key and the value alike. */
typedef struct {
  int32_t heads, dqk, dv;
  const void *q, *kv;
  int32_t q_fp8, kv_fp8;
  double q_scale, kv_scale;
  int64_t num_tokens;
  const int32_t *indptr, *indices;
  const float* sinks;
  double scale;
  double *out, *lse;
  uint32_t* row_status;
} mla_ctx;

static double mla_q(const mla_ctx* c, int64_t index) {
  if (c->q_fp8) return c->q_scale * orc_fp8_e4m3_value(((const uint8_t*)c->q)[index]);
  return orc_bf16_value(((const uint16_t*)c->q)[index]);
}

static double mla_kv(const mla_ctx* c, int64_t index) {
  if (c->kv_fp8) return c->kv_scale * orc_fp8_e4m3_value(((const uint8_t*)c->kv)[index]);
  return orc_bf16_value(((const uint16_t*)c->kv)[index]);
}

static void mla_row(void* vctx, int32_t r) {
  const mla_ctx* c = (const mla_ctx*)vctx;
  const int64_t b0 = c->indptr[r], b1 = c->indptr[r + 1];
  int64_t n = b1 - b0;
  int poisoned = n < 0;
  for (int64_t i = 0; !poisoned && i < n; ++i) {
    const int32_t t = c->indices[b0 + i];
    if (t < 0 || (int64_t)t >= c->num_tokens) poisoned = 1;
  }
  c->row_status[r] = poisoned ? ORC_BAD_TABLE : 0u;
  if (poisoned) n = 0; /* a poisoned row is computed as an empty row */
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int32_t h = 0; h < c->heads; ++h) {
    const int64_t qh = ((int64_t)r * c->heads + h) * c->dqk;
    double* o = c->out + ((int64_t)r * c->heads + h) * c->dv;
    const int has_sink = c->sinks != NULL;
    const double sink = has_sink ? (double)c->sinks[h] : -INFINITY;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
      const int64_t k = (int64_t)c->indices[b0 + i] * c->dqk;
      double dot = 0.0;
      for (int32_t d = 0; d < c->dqk; ++d) dot += mla_q(c, qh + d) * mla_kv(c, k + d);
      s[i] = c->scale * dot;
      if (s[i] > m) m = s[i];
    }
    if (has_sink && sink > m) m = sink;
    for (int32_t d = 0; d < c->dv; ++d) o[d] = 0.0;
    if (m == -INFINITY) {
      c->lse[(int64_t)r * c->heads + h] = -INFINITY;
      continue;
    }
    double den = has_sink ? exp(sink - m) : 0.0;
    for (int64_t i = 0; i < n; ++i) {
      const double p = exp(s[i] - m);
      den += p;
      const int64_t v = (int64_t)c->indices[b0 + i] * c->dqk; /* value = latent part */
      for (int32_t d = 0; d < c->dv; ++d) o[d] += p * mla_kv(c, v + d);
    }
    for (int32_t d = 0; d < c->dv; ++d) o[d] /= den;
    c->lse[(int64_t)r * c->heads + h] = m + log(den);
  }
  free(s);
}

uint32_t orc_sparse_mla_ex(int32_t num_rows, int32_t heads, int32_t dqk, int32_t dv,
                           const void* q, int32_t q_fp8, double q_scale, const void* kv_cache,
                           int32_t kv_fp8, double kv_scale, int64_t num_tokens,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           const float* sinks, double softmax_scale, double* out, double* lse,
                           int32_t nthreads) {
  mla_ctx c = {heads,    dqk,        dv,         q,          kv_cache, q_fp8, kv_fp8,
               q_scale,  kv_scale,   num_tokens, kv_indptr,  kv_indices, sinks,
               softmax_scale, out,   lse,        NULL};
  c.row_status = (uint32_t*)calloc((size_t)(num_rows > 0 ? num_rows : 1), sizeof(uint32_t));
  for_each_row(num_rows, nthreads, mla_row, &c);
  uint32_t st = 0;
  for (int32_t r = 0; r < num_rows; ++r) st |= c.row_status[r];
  free(c.row_status);
  return st;
}

uint32_t orc_sparse_mla(int32_t num_rows, int32_t heads, int32_t dqk, int32_t dv,
                        const uint16_t* q, const uint16_t* kv_cache, int64_t num_tokens,
                        const int32_t* kv_indptr, const int32_t* kv_indices, const float* sinks,
                        double softmax_scale, double* out, double* lse, int32_t nthreads) {
  return orc_sparse_mla_ex(num_rows, heads, dqk, dv, q, 0, 1.0, kv_cache, 0, 1.0, num_tokens,
                           kv_indptr, kv_indices, sinks, softmax_scale, out, lse, nthreads);
}
