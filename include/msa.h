/*
 * msa.h -- C ABI of libmsa: block-sparse paged decode for MiniMax-M3-style
 * sparse attention on one GB300 (sm_103a).
 *
 * Per query row the path scores every cached 128-token block with an index
 * query, keeps the top-k blocks, expands them into a page-16 sparse block
 * table, and runs GQA attention over only those tokens (bf16 or FP8-e4m3
 * KV with optional dequant scales, optional per-head sink, natural-log LSE).
 *
 * Definitions come from the MiniMax-M3 sparse-attention pages:
 *   [P47287] "Add ROCm AITER sparse paged attention for MiniMax-M3"
 *            (vLLM PR 47287)
 *   [P54682] "Optimise MiniMax-M3 decode index and top-k on gfx950"
 *            (vLLM PR 54682)
 *   [P54404] "Attention sinks for ROCm AITER sparse MLA" (vLLM PR 54404)
 *   [P56170] "Device-side zeroing of cu_seqlens_k[0] for MiniMax M3"
 *            (vLLM PR 56170)
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller; the library keeps no
 *     reference after the call returns and never allocates, frees or copies
 *     between host and device.
 *   - Work is enqueued on `stream` and is asynchronous.  No entry point
 *     synchronises the host (no blocking copy, no stream sync), so a
 *     sequence of calls can be captured into a CUDA graph.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned as an msa_status.  Errors in device-side data (page ids,
 *     lengths) cannot be seen on the host without a sync; kernels set bits
 *     in the caller's `dev_status` word (atomicOr, never cleared by the
 *     library), give the affected rows defined "empty" outputs and never
 *     trap.  Clear the word before a call if you want per-call bits.
 *   - Arrays are row-major and densely packed unless a stride is given.
 *     Device pointers must be 16-byte aligned.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_NULL = 1,        /* a required pointer is NULL */
  MSA_ERR_SHAPE = 2,       /* inconsistent sizes or strides, misaligned pointer */
  MSA_ERR_DTYPE = 3,       /* unknown kv dtype or scale mode */
  MSA_ERR_UNSUPPORTED = 4, /* valid but not built: see each entry point */
  MSA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than msa_workspace_size() */
  MSA_ERR_CUDA = 6         /* a CUDA launch failed (cudaGetLastError after launch) */
} msa_status;

/* KV cache element types */
enum { MSA_KV_BF16 = 0, MSA_KV_FP8_E4M3 = 1 };
/* KV dequant scale modes [P47287 "Implementation breakdown" item 2] */
enum { MSA_SCALE_NONE = 0, MSA_SCALE_SCALAR = 1, MSA_SCALE_PER_TOKEN_HEAD = 2 };

/* Device status bits (atomicOr into *dev_status).  A "poisoned" row gets
 * the outputs of an empty row: scores not written, topk_idx = -1, table =
 * 0, sparse_len = 0, O = 0, LSE = sink (or -inf without a sink). */
#define MSA_DEV_BAD_PAGE 1u  /* a request's block table holds a page id outside [0, num_pages)
                                for one of its ceil(seq_len/128) blocks: its rows are poisoned */
#define MSA_DEV_BAD_LEN 2u   /* context_lens[q] + q_len != seq_len: the request is poisoned
                                [P56170 "Implementation breakdown" item 3] */
#define MSA_DEV_MALFORMED 4u /* cu_seqlens_q does not tile [0, num_rows), seq_len < q_len,
                                context_len < 0, seq_len > 128 * bt_stride, or q_len below
                                a non-zero min_q_len: the request is poisoned */
#define MSA_DEV_BAD_TABLE 8u /* sparse table entry outside the page-16 pool, or sparse_len
                                < 0 or > 16 * tbl_stride: the row is poisoned */
#define MSA_DEV_TIMEOUT 16u  /* a bounded wait inside a kernel gave up (hardware stall);
                                outputs of that call are unspecified */

/* Batch geometry: the attention-metadata inputs of [P56170 "Key source
 * snippets"] (the prefill metadata record) and [P54682 "Implementation
 * breakdown" item 2].  All arrays are device int32.
 *   cu_seqlens_q [R+1]  rows of request q are [cu_q[q], cu_q[q+1]); must be
 *                       non-decreasing with cu_q[0] = 0, cu_q[R] = num_rows
 *   cu_seqlens_k [R+1]  seq_len of request q = cu_k[q+1] - cu_k[q] (the
 *                       pages keep cu_k[0] = 0; only differences are used)
 *   context_lens [R]    tokens cached before this step; row j of request q
 *                       sits at absolute position context_lens[q] + j and
 *                       sees tokens 0..position (causal)
 *   block_table  [R, bt_stride]  page-128 physical page of each logical
 *                       128-token block; only the first ceil(seq_len/128)
 *                       entries of a row are read
 *   num_pages    P, the number of page-128 pages in the pools (bounds check)
 *   max_q_len    host-side upper bound of any request's q_len (the metadata's
 *                max_query_len); only a launch hint: when it is >= 64, requests
 *                with >= 64 rows are scored by the tensor-core kernel.  Results
 *                do not depend on it.
 *   min_q_len    host-side lower bound of every request's q_len, 0 when not
 *                known.  When it is >= 64 (and the block-major prefill
 *                attention serves the call, see msa_decode) msa_decode
 *                launches no split-K decode attention.  A request with fewer
 *                rows than a non-zero bound is poisoned (MSA_DEV_MALFORMED). */
typedef struct msa_batch {
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* context_lens;
  const int32_t* block_table;
  int32_t bt_stride;
  int32_t num_reqs;
  int32_t num_rows;
  int32_t num_pages;
  int32_t max_q_len;
  int32_t min_q_len;
} msa_batch;

/* Attention operands [P47287 "Implementation breakdown" items 2-3],
 * [P54404 "Key source snippets"].
 *   q        [num_rows, num_heads, head_dim] bf16
 *   k_cache, v_cache  page-128 pools [P, 128, num_kv_heads, head_dim] of
 *            kv_dtype; the page-16 view [8P, 16, num_kv_heads, head_dim] is
 *            the same bytes (page-16 id e = 8 * page128 + j)
 *   scale_mode NONE: k_scale/v_scale ignored (may be NULL)
 *            SCALAR: k_scale, v_scale each fp32 [1]
 *            PER_TOKEN_HEAD: fp32 [P, 128, num_kv_heads], paged like K/V
 *            The dequantised key is k_scale * k, the value v_scale * v.
 *   sinks    fp32 [num_heads] learnable sink logits, or NULL for none; a
 *            sink adds exp(sink_h) to head h's softmax denominator
 *   softmax_scale  logit = softmax_scale * (q . k_dequantised)
 *   out      [num_rows, num_heads, head_dim] bf16
 *   lse      [num_rows, num_heads] fp32, natural log of the denominator
 *            out was normalised by (sink term included)
 * Supported: num_kv_heads == 1 (one KV head per rank, as on [P47287 "Risks
 * and impact" item 4]), head_dim == 128, 1 <= num_heads <= 16.  Others
 * return MSA_ERR_UNSUPPORTED.  With FP8 KV the query is converted to fp16
 * for the tensor-core products, so |q| must stay below 65504. */
typedef struct msa_attn_args {
  const void* q;
  int32_t num_rows;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  const void* k_cache;
  const void* v_cache;
  int32_t kv_dtype;
  int32_t num_pages; /* P, page-128 pages in the pools */
  int32_t scale_mode;
  const float* k_scale;
  const float* v_scale;
  const float* sinks;
  float softmax_scale;
  void* out;
  float* lse;
} msa_attn_args;

/* Optional CUDA events msa_decode records on `stream` after each stage (for
 * timing; any may be NULL).  msa_decode writes `kernels`: the number of
 * kernels the call launched. */
typedef struct msa_trace {
  cudaEvent_t after_score;
  cudaEvent_t after_topk;
  cudaEvent_t after_attn;
  int32_t kernels;
} msa_trace;

/* The paged index-K cache, the keys of step 1 [P54682 "Implementation
 * breakdown" item 1; the optional FP8 index storage and FP8 index scoring of
 * its "Related context"].
 *   k_cache  [P, 128, heads, dim], paged like the KV pools (token t of a
 *            request at page block_table[q, t/128], slot t%128):
 *            dtype MSA_KV_BF16: bf16 values;
 *            dtype MSA_KV_FP8_E4M3: OCP e4m3 codes, the key being
 *            k_scale[page, slot, h] * code (k_scale may be NULL: scale 1)
 *   k_scale  fp32 [P, 128, heads] (FP8 only)
 *   heads, dim  supported: (1, 64), (2, 64), (1, 128)
 * Score and decode only read the cache; msa_kv_insert writes it. */
typedef struct msa_index_cache {
  void* k_cache;
  float* k_scale;
  int32_t dtype;
  int32_t heads;
  int32_t dim;
} msa_index_cache;

/* Step 1, index scoring [P54682 "Implementation breakdown" item 1; the
 * balanced scorer of "Key files" that maps work by each request's actual
 * block count and shares index-K tiles across a request's query rows].
 * For each row r (request q, position pos) and block b < nb_r =
 * ceil((pos+1)/128):
 *     scores[r*score_stride + b] = max over index heads h and tokens
 *         t in [128b, min(128b+127, pos)] of  sum_d idx_q[r,h,d]*key[t,h,d]
 * with key[t,h,d] from the index cache (FP8: scale[t,h] * code), the sum in
 * fp32 (FP8: the products of the exact fp16 images of q and the code, then
 * times the scale).
 *   idx_q    [num_rows, heads, dim] bf16 (FP8 cache: converted to fp16 for
 *            the tensor-core products, so |idx_q| must stay below 65504)
 *   scores   [num_rows, score_stride] fp32; score_stride >= bt_stride.
 *            Entries b >= nb_r, and rows of poisoned requests, are not
 *            written; a block whose page id is out of range scores -inf.
 * Supported: the index shapes above; num_reqs <= 4096. */
msa_status msa_index_score(const msa_batch* batch, const void* idx_q,
                           const msa_index_cache* index, float* scores, int32_t score_stride,
                           uint32_t* dev_status, cudaStream_t stream);

/* Steps 2+3, top-k selection fused with the page-16 table build and the
 * context-length clamp [P54682 "Implementation breakdown" items 1 and 4;
 * P47287 "Implementation breakdown" item 3 and "Review highlights"].
 * For each row r with nb_r candidate blocks:
 *   - select m = min(topk, nb_r) blocks with the highest scores; equal scores
 *     go to the lower block index; NaN ranks below every number;
 *   - topk_idx[r, 0..m) = the selected blocks in ASCENDING block order,
 *     topk_idx[r, m..topk) = -1;
 *   - for the i-th selected block b with page p = block_table[q, b] and
 *     valid = min(128, pos+1 - 128b):
 *       sparse_tbl[r, 8i + j] = 8p + j   for j < ceil(valid/16)
 *     every other entry of the row up to tbl_stride is 0;
 *   - sparse_len[r] = sum of valid over the selected blocks, so token n of
 *     the row lives at page-16 sparse_tbl[r, n/16], slot n%16.
 *   scores   [num_rows, score_stride] fp32 (only b < nb_r is read)
 *   topk_idx [num_rows, topk] int32
 *   sparse_tbl [num_rows, tbl_stride] int32, tbl_stride >= 8*topk
 *   sparse_len [num_rows] int32
 * Supported: bt_stride <= 16384, topk <= 2048. */
msa_status msa_topk_build_table(const msa_batch* batch, const float* scores,
                                int32_t score_stride, int32_t topk, int32_t* topk_idx,
                                int32_t* sparse_tbl, int32_t tbl_stride, int32_t* sparse_len,
                                uint32_t* dev_status, cudaStream_t stream);

/* Step 4, sparse paged GQA attention [P47287 "Implementation breakdown"
 * items 2-3; P54404 "Features and motivation", "Key source snippets"].
 * For row r and head h (KV head h / (num_heads/num_kv_heads)) over the
 * n = sparse_len[r] tokens the table addresses:
 *   s_t = softmax_scale * k_scale_t * (q_h . k_t),  m = max(max_t s_t, sink_h)
 *   den = sum_t exp(s_t - m) + exp(sink_h - m)
 *   out = sum_t exp(s_t - m) * v_scale_t * v_t / den,  lse = m + ln(den)
 * (no sink: the sink terms are absent).  An empty row gives out = 0 and
 * lse = sink_h (or -inf).  The work is split along the tokens; partial
 * results are merged through their LSE inside the call.
 *   sparse_tbl [num_rows, tbl_stride] int32 page-16 ids, sparse_len [num_rows]
 *   workspace  device scratch of msa_workspace_size(...) bytes; its first
 *              use must find it zero-filled (cudaMemset once); every call
 *              leaves the counters it uses back at zero.  Calls that share a
 *              workspace must be ordered on one stream. */
msa_status msa_sparse_paged_attn(const msa_attn_args* attn, const int32_t* sparse_tbl,
                                 int32_t tbl_stride, const int32_t* sparse_len, void* workspace,
                                 size_t workspace_bytes, uint32_t* dev_status,
                                 cudaStream_t stream);

/* Size of the device array msa_sparse_paged_attn_static draws its scratch
 * from (8 MiB per GPU that loads the library, held until the process exits). */
#define MSA_STATIC_SCRATCH_BYTES (8u << 20)

/* msa_sparse_paged_attn without a workspace, for callers that cannot
 * allocate device memory: code where cudaMalloc is off limits because it
 * synchronises the device and would stall a serving loop, plug-ins whose
 * host framework owns all device memory and offers no allocator, runtimes
 * that forbid allocation after start-up.  (The pages have no counterpart;
 * it is an addition of this library.)
 * Same arguments, semantics, argument checks and results as
 * msa_sparse_paged_attn, minus the workspace: the split-merge scratch comes
 * from one static device array of MSA_STATIC_SCRATCH_BYTES.  Argument errors
 * are returned before anything touches the array or the stream.
 *   - Scratch use: rows are split along their tokens (at most 128 page-16
 *     entries per split).  Rows of 1 to 8 splits (tbl_stride <= 1024, i.e.
 *     top-k <= 128 blocks) merge inside a thread-block cluster and use only
 *     4 bytes per row (rounded up to 256).  Rows of more splits merge
 *     through partials: 4 + 8320 * splits bytes per row, splits =
 *     ceil(tbl_stride / 128).  A call needing more than
 *     MSA_STATIC_SCRATCH_BYTES returns MSA_ERR_WORKSPACE (e.g. more than
 *     ~100 rows at tbl_stride 1280).
 *   - Allocates nothing and calls no allocating routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - A call of more than 8 splits clears the array's counters on `stream`
 *     (cudaMemsetAsync) before the kernel; the rest of the array keeps the
 *     last call's data.
 *   - The array is shared by all calls in the process: calls whose kernels
 *     overlap on the GPU race on it (order them on one stream). */
msa_status msa_sparse_paged_attn_static(const msa_attn_args* attn, const int32_t* sparse_tbl,
                                        int32_t tbl_stride, const int32_t* sparse_len,
                                        uint32_t* dev_status, cudaStream_t stream);

/* The whole path: msa_index_score -> msa_topk_build_table ->
 * msa_sparse_paged_attn in stream order, with the intermediates held in the
 * workspace [P54682 "Implementation breakdown" items 1-3: the decode index
 * scoring fused with the top-k, the indexer writing the sparse table the
 * attention consumes].  topk_idx, sparse_tbl and sparse_len may be NULL
 * (held in the workspace) or device arrays that receive them; tbl_stride is
 * the width of the caller's sparse_tbl (>= 8*topk, ignored when NULL).
 * trace may be NULL.  Calls sharing a workspace must be ordered on one
 * stream.  Selection, table and lengths are bit-identical to the three
 * separate calls, and so are O / LSE except on the rows of requests with
 * >= 64 rows when max_q_len >= 64, the KV is bf16 without per-token scales
 * and topk <= 128: those rows take a block-major tensor-core attention,
 * whose O / LSE agree with the other path within the attention tolerance,
 * not bit for bit.  When min_q_len >= 64 as well, every row takes that path
 * and the split-K decode attention is not launched (a poisoned row is then
 * written as an empty row by the block-major path's merge). */
msa_status msa_decode(const msa_batch* batch, const void* idx_q, const msa_index_cache* index,
                      int32_t topk, const msa_attn_args* attn, int32_t* topk_idx, int32_t* sparse_tbl,
                      int32_t tbl_stride, int32_t* sparse_len, void* workspace,
                      size_t workspace_bytes, uint32_t* dev_status, msa_trace* trace,
                      cudaStream_t stream);

/* The step before the path: write the new tokens' K, V and index-K into
 * the paged pools [P47287 "Implementation breakdown" item 1: the fused
 * q/k-norm + RoPE + KV insert with skip_index, so index-reuse layers skip the
 * index-cache write; item 5: separate K and V pools].  Every query row of the
 * batch is a new token at its own position pos = context_lens[q] + j; its
 * vectors go to page block_table[q, pos/128], slot pos%128 (the q/k norm and
 * RoPE need model weights and stay with the caller).
 *   k_new, v_new [num_rows, num_kv_heads, head_dim] bf16
 *   k_cache, v_cache  pools [P, 128, num_kv_heads, head_dim] of kv_dtype
 *   idx_new      [num_rows, index->heads, index->dim] bf16
 *   index        the index cache (may be NULL when skip_index)
 * FP8 pools store OCP e4m3 codes of x / s (IEEE fp32 division, round to
 * nearest even, saturating to +-448): SCALAR takes s = k_scale[0] (v_scale[0])
 * as input; PER_TOKEN_HEAD sets s = max_d |x_d| / 448 per token and KV head
 * (1 for an all-zero vector) and writes it to k_scale / v_scale [P, 128,
 * num_kv_heads] at the slot; NONE takes s = 1.  bf16 pools take a copy.  An
 * FP8 index cache is written the same way, per token and index head, with
 * the PER_TOKEN_HEAD rule when index->k_scale is given and s = 1 when it is
 * NULL.  Rows of requests that fail the device checks (MSA_DEV_BAD_PAGE,
 * _BAD_LEN, _MALFORMED) are not written.  Supported: head_dim == 128. */
msa_status msa_kv_insert(const msa_batch* batch, const void* k_new, const void* v_new,
                         int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                         int32_t kv_dtype, int32_t scale_mode, float* k_scale, float* v_scale,
                         const void* idx_new, const msa_index_cache* index, int32_t skip_index,
                         uint32_t* dev_status, cudaStream_t stream);

/* Sparse MLA decode operands ["Attention sinks for ROCm AITER sparse MLA"
 * (vLLM PR 54404), "Implementation breakdown" items 1-2, "Key source
 * snippets": one latent KV head, the indptr / indices token convention].
 *   q          [num_rows, num_heads, dqk] bf16
 *   kv_cache   [num_tokens, dqk] bf16: one latent row per cached token; the
 *              key is the whole row, the value its first dv values
 *   kv_indptr  [num_rows + 1] int32, kv_indices [kv_indptr[num_rows]] int32:
 *              row r attends over token ids kv_indices[kv_indptr[r] ..
 *              kv_indptr[r+1]) (repeats count as often as they appear)
 *   max_tokens bound on every row's count; it sizes the work split, and a
 *              longer row (or an id outside [0, num_tokens)) makes that row
 *              an empty row and raises MSA_DEV_BAD_TABLE
 *   sinks      fp32 [num_heads] or NULL;  softmax_scale as for attention
 *   out        [num_rows, num_heads, dv] bf16;  lse [num_rows, num_heads] fp32
 *   kv_dtype   MSA_KV_BF16, or MSA_KV_FP8_E4M3: kv_cache holds OCP e4m3
 *              codes [num_tokens, dqk] and an element (of the key and of the
 *              value) is kv_scale[0] * code (kv_scale: device fp32 [1])
 *   q_dtype    MSA_KV_BF16, or MSA_KV_FP8_E4M3 (only with an FP8 cache): q
 *              holds e4m3 codes and an element is q_scale[0] * code
 *              [the decode op's q_scale / kv_scale, "Key source snippets"]
 * For head h: s_t = softmax_scale * (q_h . kv_t[0:dqk]),
 * m = max(max_t s_t, sink_h), den = sum_t exp(s_t - m) + exp(sink_h - m),
 * out = sum_t exp(s_t - m) kv_t[0:dv] / den, lse = m + ln(den).
 * With an FP8 cache the products run in f16 on the tensor cores (e4m3 codes
 * convert exactly; a bf16 query converts to f16, so |q| must stay below
 * 65504).  Supported: dqk == 576, dv == 512 (512 latent + 64 rope),
 * 1 <= num_heads <= 128, num_rows <= 65535; an FP8 query with a bf16 cache
 * returns MSA_ERR_UNSUPPORTED. */
typedef struct msa_mla_args {
  const void* q;
  int32_t num_rows;
  int32_t num_heads;
  int32_t dqk;
  int32_t dv;
  const void* kv_cache;
  int64_t num_tokens;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  int32_t max_tokens;
  const float* sinks;
  float softmax_scale;
  void* out;
  float* lse;
  int32_t q_dtype;
  int32_t kv_dtype;
  const float* q_scale;
  const float* kv_scale;
} msa_mla_args;

/* Bytes of workspace msa_sparse_mla_decode needs (zero-filled before its
 * first use; every call leaves its counters back at zero). */
size_t msa_sparse_mla_workspace_size(int32_t num_rows, int32_t num_heads, int32_t max_tokens);

/* Sparse MLA decode with sinks and a natural-log LSE, as defined above. */
msa_status msa_sparse_mla_decode(const msa_mla_args* mla, void* workspace,
                                 size_t workspace_bytes, uint32_t* dev_status,
                                 cudaStream_t stream);

/* Bytes of workspace msa_decode (bt_stride > 0) or msa_sparse_paged_attn
 * (bt_stride = 0, topk = 0) needs for these sizes. */
size_t msa_workspace_size(int32_t num_rows, int32_t bt_stride, int32_t topk, int32_t num_heads,
                          int32_t head_dim, int32_t tbl_stride);

/* Check of the bounded waits (failure detection without a GPU fault).
 * Every kernel of the library gives up a wait that has not completed after
 * a time limit (2 s), records MSA_DEV_TIMEOUT and returns, freeing what it
 * holds, instead of hanging [P54404 "Key source snippets": a missing result
 * must raise, not hang].  This entry point exercises that machinery on
 * purpose: one CTA waits, with the library's own bounded wait and a limit
 * of limit_us microseconds (1 .. 1e6), on an mbarrier armed for transaction
 * bytes that nothing delivers, and on expiry sets MSA_DEV_TIMEOUT in
 * *dev_status.  flags:
 *   MSA_CHECK_WAIT_TMEM  the CTA holds tensor memory during the wait and
 *                        frees it on the way out;
 *   MSA_CHECK_WAIT_COPY  a real 16-byte bulk copy from copy_src (device,
 *                        16-byte aligned) is in flight and is drained
 *                        before the CTA leaves (a drain that itself gave up
 *                        would set MSA_DEV_TIMEOUT << 1).
 * The context stays usable: later calls on the stream run normally.
 * Argument errors: dev_status NULL or a copy without copy_src -> NULL;
 * limit_us out of range -> SHAPE; unknown flags -> UNSUPPORTED. */
#define MSA_CHECK_WAIT_TMEM 1
#define MSA_CHECK_WAIT_COPY 2
msa_status msa_check_bounded_wait(uint32_t* dev_status, uint32_t limit_us, int32_t flags,
                                  const void* copy_src, cudaStream_t stream);

/* Static description of a status code. */
const char* msa_status_string(msa_status status);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H */
