/*
 * msa_oracle.h -- plain fp64 CPU oracle for the block-sparse paged decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code, header, table or helper with the CUDA library: it is written
 * straight from the definitions on the MiniMax-M3 sparse-attention pages
 * (vLLM PR 47287 "Add ROCm AITER sparse paged attention for MiniMax-M3",
 * PR 54682 "Optimise MiniMax-M3 decode index and top-k on gfx950",
 * PR 54404 "Attention sinks for ROCm AITER sparse MLA", PR 56170 "device
 * zeroing of cu_seqlens_k[0]") and the OCP FP8 format definition.
 *
 * All arrays are host memory, row-major, owned by the caller.
 *   bf16 tensors : uint16_t bit patterns
 *   fp8 tensors  : uint8_t OCP e4m3fn codes
 */
#ifndef MSA_ORACLE_H
#define MSA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status bits (the same meaning as the library's device status word) */
#define ORC_BAD_PAGE 1u    /* block-table page id outside [0, P) */
#define ORC_BAD_LEN 2u     /* context_len + q_len != seq_len */
#define ORC_MALFORMED 4u   /* malformed cu_seqlens / lengths beyond the table */
#define ORC_BAD_TABLE 8u   /* sparse-table entry outside the page-16 pool */

typedef struct {
  int32_t num_reqs;             /* R */
  int32_t num_rows;             /* N */
  const int32_t* cu_seqlens_q;  /* [R+1] */
  const int32_t* cu_seqlens_k;  /* [R+1] */
  const int32_t* context_lens;  /* [R] */
  const int32_t* block_table;   /* [R, bt_stride] page-128 ids */
  int32_t bt_stride;
  int32_t num_pages;            /* P */
} orc_batch;

/* Value of one OCP e4m3fn code (bias 7, no infinities, S.1111.111 = NaN). */
double orc_fp8_e4m3_value(uint8_t code);
/* Value of one bf16 bit pattern. */
double orc_bf16_value(uint16_t bits);

/* Per-row geometry.  req[r] = owning request or -1, pos[r] = absolute
 * position, nb[r] = ceil((pos+1)/128), ok[r] = 1 unless the row is poisoned.
 * Returns the status bits the batch raises. */
uint32_t orc_row_geometry(const orc_batch* b, int32_t* req, int32_t* pos, int32_t* nb,
                          int32_t* ok);

/* Step 1: block scores.  scores[r, b] for b < nb[r] = max over index heads and
 * over tokens t of block b with t <= pos[r] of sum_d qidx[r,h,d]*kidx[t,h,d],
 * accumulated in fp64 and rounded to fp32; -inf for b >= nb[r], for blocks
 * whose page id is out of range and for every block of a poisoned row. */
uint32_t orc_index_score(const orc_batch* b, const uint16_t* idx_q, const uint16_t* idx_k,
                         int32_t index_heads, int32_t index_dim, float* scores,
                         int32_t score_stride, int32_t nthreads);

/* Step 1 with an FP8 index-K cache (OCP e4m3 codes [P,128,Hi,Di]; optional
 * fp32 per-token scales k_scale [P,128,Hi], NULL meaning 1): the dot product
 * with the decoded codes, times the token's scale, then the same maximum and
 * fp32 rounding as orc_index_score. */
uint32_t orc_index_score_fp8(const orc_batch* b, const uint16_t* idx_q, const uint8_t* idx_k,
                             const float* k_scale, int32_t index_heads, int32_t index_dim,
                             float* scores, int32_t score_stride, int32_t nthreads);

/* Steps 2+3: top-k (ties to the lower block, output ascending by block) and
 * page-16 table expansion with the context-length clamp. */
uint32_t orc_topk_build_table(const orc_batch* b, const float* scores, int32_t score_stride,
                              int32_t topk, int32_t* topk_idx, int32_t* sparse_tbl,
                              int32_t tbl_stride, int32_t* sparse_len, int32_t nthreads);

/* Step 4: GQA attention over the tokens the page-16 table addresses, with
 * optional dequant scales and sink.  out [N,Hq,D] and lse [N,Hq] in fp64. */
uint32_t orc_sparse_attn(int32_t num_rows, int32_t hq, int32_t hkv, int32_t head_dim,
                         const uint16_t* q, const void* k_cache, const void* v_cache,
                         int32_t kv_dtype, int32_t num_pages16, int32_t scale_mode,
                         const float* k_scale, const float* v_scale, const int32_t* sparse_tbl,
                         int32_t tbl_stride, const int32_t* sparse_len, const float* sinks,
                         double softmax_scale, double* out, double* lse, int32_t nthreads);

/* Dense attention over every visible token t < pos[r]+1 through the page-128
 * block table (no index, no selection); the identity the sparse path reduces
 * to when top-k covers every block. */
uint32_t orc_dense_attn(const orc_batch* b, int32_t hq, int32_t hkv, int32_t head_dim,
                        const uint16_t* q, const void* k_cache, const void* v_cache,
                        int32_t kv_dtype, int32_t scale_mode, const float* k_scale,
                        const float* v_scale, const float* sinks, double softmax_scale,
                        double* out, double* lse, int32_t nthreads);

/* OCP e4m3fn code of a float: round to nearest, ties to the even code,
 * saturating to +-448 (infinities included); NaN gives 0x7F. */
uint8_t orc_fp8_e4m3_encode(float x);

/* The step before the path: write every row's new K, V (and index-K unless
 * skip_index) into the paged pools at the row's own position (page
 * block_table[q, pos/128], slot pos%128).  FP8 caches: SCALAR divides by the
 * given k_scale[0] / v_scale[0]; PER_TOKEN_HEAD computes s = max_d |x_d| / 448
 * per token and KV head (s = 1 when all zero), stores it in k_scale/v_scale
 * at the slot and divides by it.  The division is fp32 and the code is
 * orc_fp8_e4m3_encode of the quotient.  An FP8 index cache (idx_dtype 1:
 * e4m3 codes) is written the same way per token and index head, with the
 * PER_TOKEN_HEAD rule into idx_scale [P,128,Hi] when idx_scale is given and
 * scale 1 when it is NULL; a bf16 one (idx_dtype 0) takes a copy.  Rows of
 * requests that do not pass the geometry checks are not written. */
uint32_t orc_kv_insert(const orc_batch* b, int32_t hkv, int32_t head_dim, const uint16_t* k_new,
                       const uint16_t* v_new, int32_t index_heads, int32_t index_dim,
                       const uint16_t* idx_new, void* k_cache, void* v_cache,
                       void* idx_k_cache, int32_t kv_dtype, int32_t scale_mode,
                       float* k_scale, float* v_scale, int32_t skip_index, int32_t idx_dtype,
                       float* idx_scale);

/* Sparse MLA decode (the sparse-MLA-with-sinks page): one latent KV head,
 * kv_cache [num_tokens, dqk] bf16 whose first dv columns are the value; row r
 * attends over token ids kv_indices[kv_indptr[r] .. kv_indptr[r+1]) with
 *   s_t = softmax_scale * (q_h . kv_t[0:dqk]),  m = max(max_t s_t, sink_h),
 *   den = sum_t exp(s_t - m) + exp(sink_h - m),
 *   out = sum_t exp(s_t - m) kv_t[0:dv] / den,  lse = m + ln(den)
 * in fp64 (no sink: its terms are absent).  A row with a negative count or a
 * token id outside [0, num_tokens) is an empty row and raises ORC_BAD_TABLE.
 * q [num_rows, heads, dqk] bf16; out [num_rows, heads, dv], lse [num_rows, heads]. */
uint32_t orc_sparse_mla(int32_t num_rows, int32_t heads, int32_t dqk, int32_t dv,
                        const uint16_t* q, const uint16_t* kv_cache, int64_t num_tokens,
                        const int32_t* kv_indptr, const int32_t* kv_indices, const float* sinks,
                        double softmax_scale, double* out, double* lse, int32_t nthreads);

/* The same with FP8 operands ("Attention sinks for ROCm AITER sparse MLA",
 * "Key source snippets": q_scale, kv_scale of the decode op): q (q_fp8 = 1)
 * holds e4m3 codes, an element being q_scale * code; kv_cache (kv_fp8 = 1)
 * holds e4m3 codes, an element of the key and of the value being
 * kv_scale * code; a bf16 operand ignores its scale. */
uint32_t orc_sparse_mla_ex(int32_t num_rows, int32_t heads, int32_t dqk, int32_t dv,
                           const void* q, int32_t q_fp8, double q_scale, const void* kv_cache,
                           int32_t kv_fp8, double kv_scale, int64_t num_tokens,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           const float* sinks, double softmax_scale, double* out, double* lse,
                           int32_t nthreads);

#ifdef __cplusplus
}
#endif
#endif
