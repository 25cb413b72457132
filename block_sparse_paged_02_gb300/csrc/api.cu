// api.cu -- the C ABI of libmsa: argument validation, workspace layout and
// kernel launches.  Nothing here touches device data or synchronises: every
// check is on host-visible arguments, and data errors are left to the
// kernels' device status word (see msa.h).
#include <cstring>
#include <mutex>

#include "msa_internal.cuh"

namespace msa {

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Attention work split: page-16 entries per split and the split count.  The
// grid (splits x rows) is sized to fill the GPU once: as many splits per row
// as fit in ctas_per_sm resident CTAs on every SM, each split a multiple of 4
// entries (one per warp) and at most kMaxSplitEntries.  Workspaces are sized
// with the largest residency of any variant (3), launches use their own.
constexpr int kMaxAttnCtasPerSm =
    MSA_ATTN_CTAS_FP8 > MSA_ATTN_CTAS_BF16 ? MSA_ATTN_CTAS_FP8 : MSA_ATTN_CTAS_BF16;

void attn_split(int num_rows, int max_entries, int ctas_per_sm, int* pps, int* splits) {
  const int capacity = device_sm_count() * ctas_per_sm;
  int target = num_rows > 0 ? capacity / num_rows : 1;
  if (target < 1) target = 1;
  int per = (max_entries + target - 1) / target;
  per = per < 4 ? 4 : (per + 3) / 4 * 4;
  // at most 8 splits (one thread-block cluster merges them) whenever the
  // entries fit: the cluster merge is much cheaper than the workspace one
  if ((max_entries + per - 1) / per > 8 && max_entries <= 8 * kMaxSplitEntries)
    per = ((max_entries + 7) / 8 + 3) / 4 * 4;
  if (per > kMaxSplitEntries) per = kMaxSplitEntries;
  *pps = per;
  *splits = max_entries > 0 ? (max_entries + per - 1) / per : 1;
}

int attn_ctas_per_sm(const msa_attn_args* a) {
  return a->kv_dtype == MSA_KV_FP8_E4M3 ? MSA_ATTN_CTAS_FP8 : MSA_ATTN_CTAS_BF16;
}

struct DecodeWs {
  size_t counters, scores, topk, tbl, len, partials;
  // prefill path (present when topk <= kPrefillMaxTopk): route [N], list
  // counts and lists, the plan, the per-(row, slot) partials
  bool prefill;
  size_t route, pf_counts, pf_lists, plan_hdr, plan_req_q, plan_req_item, item_rec, item_kv,
      item_chunk, item_cost, part_o, part_ml;
  long long max_routed_reqs, max_items;
  size_t total;
};

DecodeWs decode_layout(int num_rows, int bt_stride, int topk, int splits) {
  DecodeWs w;
  const size_t n = (size_t)(num_rows > 0 ? num_rows : 1);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  w.counters = take(n * 4);
  w.scores = take(n * (size_t)bt_stride * 4);
  w.topk = take(n * (size_t)topk * 4);
  w.tbl = take(n * (size_t)topk * 8 * 4);
  w.len = take(n * 4);
  w.partials = take(n * (size_t)splits * kPartFloats * 4);
  w.prefill = topk >= 1 && topk <= kPrefillMaxTopk;
  if (w.prefill) {
    // a routed request has >= kPrefillMinRows rows, so at most n / 64 of them,
    // each with at most bt_stride blocks; list counts sit at q0 * bt / 64
    const size_t bt = (size_t)bt_stride;
    w.max_routed_reqs = (long long)(n / kPrefillMinRows + 1);
    w.max_items = (long long)(n * bt / kPrefillMinRows + bt);
    w.route = take(n * 4);
    w.pf_counts = take((size_t)w.max_items * 4);
    w.pf_lists = take(n * bt * 4);
    w.plan_hdr = take(64);
    w.plan_req_q = take((size_t)w.max_routed_reqs * 4);
    w.plan_req_item = take((size_t)w.max_routed_reqs * 4);
    w.item_rec = take((size_t)w.max_items * 16);
    w.item_kv = take((size_t)w.max_items * 8);
    w.item_chunk = take((size_t)w.max_items * 4);  // (max_items > items: room for the totals)
    w.item_cost = take((size_t)w.max_items * 4);
    w.part_o = take(n * (size_t)topk * 16 * kHeadDim * 2);
    w.part_ml = take(n * (size_t)topk * 16 * 8);
  }
  w.total = off;
  return w;
}

msa_status check_batch(const msa_batch* b) {
  if (!b) return MSA_ERR_NULL;
  if (b->num_reqs < 0 || b->num_rows < 0 || b->num_pages < 0 || b->bt_stride < 1)
    return MSA_ERR_SHAPE;
  if (b->num_reqs > 0 &&
      (!b->cu_seqlens_q || !b->cu_seqlens_k || !b->context_lens || !b->block_table))
    return MSA_ERR_NULL;
  if (b->num_reqs == 0 && !b->cu_seqlens_q) return MSA_ERR_NULL;
  if (b->num_reqs > kMaxReqs || b->bt_stride > kMaxBlocksPerRow) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

msa_status check_attn(const msa_attn_args* a) {
  if (!a) return MSA_ERR_NULL;
  if (a->kv_dtype != MSA_KV_BF16 && a->kv_dtype != MSA_KV_FP8_E4M3) return MSA_ERR_DTYPE;
  if (a->scale_mode < MSA_SCALE_NONE || a->scale_mode > MSA_SCALE_PER_TOKEN_HEAD)
    return MSA_ERR_DTYPE;
  if (a->num_rows < 0 || a->num_heads < 1 || a->num_kv_heads < 1 || a->num_pages < 0)
    return MSA_ERR_SHAPE;
  if (a->num_heads % a->num_kv_heads != 0) return MSA_ERR_SHAPE;
  if (a->num_kv_heads != 1 || a->head_dim != kHeadDim || a->num_heads > kMaxHeads)
    return MSA_ERR_UNSUPPORTED;
  if (a->num_rows > 0 && (!a->q || !a->k_cache || !a->v_cache || !a->out || !a->lse))
    return MSA_ERR_NULL;
  if (a->scale_mode != MSA_SCALE_NONE && (!a->k_scale || !a->v_scale)) return MSA_ERR_NULL;
  if (!aligned16(a->q) || !aligned16(a->k_cache) || !aligned16(a->v_cache) ||
      !aligned16(a->out) || !aligned16(a->lse))
    return MSA_ERR_SHAPE;
  if (a->scale_mode == MSA_SCALE_PER_TOKEN_HEAD && (!aligned16(a->k_scale) || !aligned16(a->v_scale)))
    return MSA_ERR_SHAPE;
  return MSA_OK;
}

msa_status check_index(const msa_index_cache* x) {
  if (!x) return MSA_ERR_NULL;
  if (x->dtype != MSA_KV_BF16 && x->dtype != MSA_KV_FP8_E4M3) return MSA_ERR_DTYPE;
  if (!((x->heads == 1 && (x->dim == 64 || x->dim == 128)) || (x->heads == 2 && x->dim == 64)))
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

AttnLaunch make_attn(const msa_attn_args* a, const int32_t* tbl, int tbl_stride,
                     const int32_t* len, float* partials, uint32_t* counters, int pps,
                     int splits, uint32_t* status) {
  AttnLaunch L;
  L.q = static_cast<const uint16_t*>(a->q);
  L.num_rows = a->num_rows;
  L.num_heads = a->num_heads;
  L.k = static_cast<const uint8_t*>(a->k_cache);
  L.v = static_cast<const uint8_t*>(a->v_cache);
  L.kv_fp8 = a->kv_dtype == MSA_KV_FP8_E4M3;
  L.num_pages16 = 8ll * a->num_pages;
  L.scale_mode = a->scale_mode;
  L.k_scale = a->k_scale;
  L.v_scale = a->v_scale;
  L.sinks = a->sinks;
  L.softmax_scale = a->softmax_scale;
  L.tbl = tbl;
  L.tbl_stride = tbl_stride;
  L.sparse_len = len;
  L.out = static_cast<uint16_t*>(a->out);
  L.lse = a->lse;
  L.partials = partials;
  L.counters = counters;
  L.splits = splits;
  L.pages_per_split = pps;
  L.status = status;
  L.route = nullptr;
  return L;
}

msa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

// Sparse MLA work split: splits of each (row, 16-head group) so that the
// grid fills MSA_MLA_CTAS CTAs per SM, each split at least 64 and at most
// mla_max_tokens_per_split() token ids, a multiple of 16, and at most 8
// splits (one cluster) when that bound allows.
void mla_split(int num_rows, int num_heads, int max_tokens, int* splits, int* per) {
  const int groups = (num_heads + 15) / 16;
  const long long base = (long long)num_rows * groups;
  const int capacity = device_sm_count() * MSA_MLA_CTAS;
  int s = base > 0 ? (int)max(1ll, capacity / base) : 1;
  const int lim = mla_max_tokens_per_split();
  s = max(s, (max_tokens + lim - 1) / lim);
  s = min(s, max(1, (max_tokens + 63) / 64));
  // at most 8 splits (one thread-block cluster merges them) whenever a
  // split can hold the rest
  if (s > 8 && (max_tokens + 7) / 8 <= lim) s = 8;
  int t = (max_tokens + s - 1) / s;
  t = (t + 15) / 16 * 16;
  if (t > lim) t = lim;
  *per = t;
  *splits = max(1, (max_tokens + t - 1) / t);
}

struct MlaWs {
  size_t counters, partials, total;
};

MlaWs mla_layout(int num_rows, int num_heads, int max_tokens) {
  int splits, per;
  mla_split(num_rows, num_heads, max_tokens, &splits, &per);
  const size_t rg = (size_t)(num_rows > 0 ? num_rows : 1) * (size_t)((num_heads + 15) / 16);
  MlaWs w;
  w.counters = 0;
  w.partials = round_up(rg * 4, 256);
  // partials only for more splits than one cluster holds
  w.total = w.partials + (splits > 8 ? rg * (size_t)splits * 16 * 516 * 4 : 0);
  return w;
}

// Step 1: the streaming CUDA-core kernel, plus the tensor-core kernel for
// requests with many rows when the batch may hold any (max_q_len hint).
cudaError_t launch_scores(ScoreLaunch p, cudaStream_t stream, int* kernels = nullptr) {
  // (bf16 keys only: an FP8 cache would need FP8 queries for the f8 MMA kinds)
  const bool tc = !p.idx_fp8 && p.batch.max_q_len >= kTcMinRows &&
                  tc_score_supported(p.index_heads, p.index_dim);
  p.tc_min_rows = tc ? kTcMinRows : 0;
  // every request known to have tensor-core rows (min_q_len hint): the
  // CUDA-core kernel would score nothing; the tensor-core one then reports
  // the batch's status bits
  const bool cuda_core = !(tc && p.batch.min_q_len >= kTcMinRows);
  p.report_status = cuda_core ? 0 : 1;
  if (kernels) *kernels = (cuda_core ? 1 : 0) + (tc ? 1 : 0);
  if (cuda_core) {
    cudaError_t e = launch_index_score(p, stream);
    if (e != cudaSuccess || !tc) return e;
  }
  return launch_index_score_tc(p, stream);
}

}  // namespace

msa_status attn_prepare(const msa_attn_args* attn, const int32_t* sparse_tbl, int tbl_stride,
                        const int32_t* sparse_len, const uint32_t* dev_status, int* pps,
                        int* splits) {
  msa_status st = check_attn(attn);
  if (st != MSA_OK) return st;
  if (!dev_status) return MSA_ERR_NULL;
  if (tbl_stride < 1) return MSA_ERR_SHAPE;
  *pps = 0;
  *splits = 0;
  if (attn->num_rows == 0) return MSA_OK;
  if (!sparse_tbl || !sparse_len) return MSA_ERR_NULL;
  attn_split(attn->num_rows, tbl_stride, attn_ctas_per_sm(attn), pps, splits);
  return MSA_OK;
}

size_t attn_scratch_offset_partials(int num_rows) {
  return round_up((size_t)(num_rows > 0 ? num_rows : 1) * 4, 256);
}

size_t attn_scratch_need(int num_rows, int splits) {
  const size_t counters = attn_scratch_offset_partials(num_rows);
  if (splits <= kMaxClusterSplits) return counters;
  return counters + round_up((size_t)num_rows * (size_t)splits * kPartFloats * 4, 256);
}

msa_status attn_run(const msa_attn_args* attn, const int32_t* sparse_tbl, int tbl_stride,
                    const int32_t* sparse_len, void* scratch, int pps, int splits,
                    uint32_t* dev_status, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws);
  float* partials = reinterpret_cast<float*>(ws + attn_scratch_offset_partials(attn->num_rows));
  AttnLaunch p = make_attn(attn, sparse_tbl, tbl_stride, sparse_len, partials, counters, pps,
                           splits, dev_status);
  return cuda_status(launch_sparse_attn(p, stream, false));
}

}  // namespace msa

using namespace msa;

extern "C" {

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_NULL: return "a required pointer is NULL";
    case MSA_ERR_SHAPE: return "inconsistent sizes, strides or alignment";
    case MSA_ERR_DTYPE: return "unknown kv dtype or scale mode";
    case MSA_ERR_UNSUPPORTED: return "configuration not supported by this build";
    case MSA_ERR_WORKSPACE: return "workspace missing or too small";
    case MSA_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

size_t msa_workspace_size(int32_t num_rows, int32_t bt_stride, int32_t topk, int32_t num_heads,
                          int32_t head_dim, int32_t tbl_stride) {
  (void)num_heads;
  (void)head_dim;
  if (num_rows < 0 || bt_stride < 0 || topk < 0 || tbl_stride < 0) return 0;
  int pps, splits;
  const int max_entries = topk > 0 ? 8 * topk : tbl_stride;
  attn_split(num_rows, max_entries, kMaxAttnCtasPerSm, &pps, &splits);
  if (bt_stride == 0) {  // attention only: counters + partials
    const size_t n = (size_t)(num_rows > 0 ? num_rows : 1);
    return round_up(n * 4, 256) + round_up(n * (size_t)splits * kPartFloats * 4, 256);
  }
  return decode_layout(num_rows, bt_stride, topk, splits).total;
}

msa_status msa_index_score(const msa_batch* batch, const void* idx_q,
                           const msa_index_cache* index, float* scores, int32_t score_stride,
                           uint32_t* dev_status, cudaStream_t stream) {
  msa_status st = check_batch(batch);
  if (st != MSA_OK) return st;
  st = check_index(index);
  if (st != MSA_OK) return st;
  if (!dev_status || (batch->num_rows > 0 && (!idx_q || !index->k_cache || !scores)))
    return MSA_ERR_NULL;
  if (score_stride < batch->bt_stride) return MSA_ERR_SHAPE;
  if (!aligned16(idx_q) || !aligned16(index->k_cache) ||
      (index->k_scale && !aligned16(index->k_scale)))
    return MSA_ERR_SHAPE;
  if (batch->num_rows == 0 || batch->num_reqs == 0) return MSA_OK;
  ScoreLaunch p{*batch, static_cast<const uint16_t*>(idx_q),
                static_cast<const uint8_t*>(index->k_cache), index->heads, index->dim, scores,
                score_stride, dev_status, 0, index->dtype == MSA_KV_FP8_E4M3,
                index->dtype == MSA_KV_FP8_E4M3 ? index->k_scale : nullptr};
  return cuda_status(launch_scores(p, stream));
}

msa_status msa_topk_build_table(const msa_batch* batch, const float* scores,
                                int32_t score_stride, int32_t topk, int32_t* topk_idx,
                                int32_t* sparse_tbl, int32_t tbl_stride, int32_t* sparse_len,
                                uint32_t* dev_status, cudaStream_t stream) {
  msa_status st = check_batch(batch);
  if (st != MSA_OK) return st;
  if (!dev_status) return MSA_ERR_NULL;
  if (topk < 1) return MSA_ERR_SHAPE;
  if (topk > kMaxTopk) return MSA_ERR_UNSUPPORTED;
  if (tbl_stride < 8 * topk || score_stride < batch->bt_stride) return MSA_ERR_SHAPE;
  if (batch->num_rows > 0 && (!scores || !topk_idx || !sparse_tbl || !sparse_len))
    return MSA_ERR_NULL;
  if (batch->num_rows == 0) return MSA_OK;
  if (batch->num_reqs == 0) return MSA_ERR_SHAPE;  // rows without any request
  TopkLaunch p{*batch,     scores,     score_stride, topk,    topk_idx, sparse_tbl, tbl_stride,
               sparse_len, nullptr,    dev_status,   nullptr, nullptr,  nullptr};
  return cuda_status(launch_topk_table(p, stream, false));
}

msa_status msa_sparse_paged_attn(const msa_attn_args* attn, const int32_t* sparse_tbl,
                                 int32_t tbl_stride, const int32_t* sparse_len, void* workspace,
                                 size_t workspace_bytes, uint32_t* dev_status,
                                 cudaStream_t stream) {
  int pps, splits;
  const msa_status st =
      attn_prepare(attn, sparse_tbl, tbl_stride, sparse_len, dev_status, &pps, &splits);
  if (st != MSA_OK || attn->num_rows == 0) return st;
  const size_t need = msa_workspace_size(attn->num_rows, 0, 0, attn->num_heads, attn->head_dim,
                                         tbl_stride);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return MSA_ERR_WORKSPACE;
  return attn_run(attn, sparse_tbl, tbl_stride, sparse_len, workspace, pps, splits, dev_status,
                  stream);
}

msa_status msa_decode(const msa_batch* batch, const void* idx_q, const msa_index_cache* index,
                      int32_t topk, const msa_attn_args* attn, int32_t* topk_idx, int32_t* sparse_tbl,
                      int32_t tbl_stride, int32_t* sparse_len, void* workspace,
                      size_t workspace_bytes, uint32_t* dev_status, msa_trace* trace,
                      cudaStream_t stream) {
  msa_status st = check_batch(batch);
  if (st != MSA_OK) return st;
  st = check_attn(attn);
  if (st != MSA_OK) return st;
  if (!dev_status) return MSA_ERR_NULL;
  if (topk < 1) return MSA_ERR_SHAPE;
  if (topk > kMaxTopk) return MSA_ERR_UNSUPPORTED;
  if (attn->num_rows != batch->num_rows) return MSA_ERR_SHAPE;
  if (attn->num_pages != batch->num_pages) return MSA_ERR_SHAPE;
  st = check_index(index);
  if (st != MSA_OK) return st;
  if (sparse_tbl && tbl_stride < 8 * topk) return MSA_ERR_SHAPE;
  if (batch->num_rows == 0) return MSA_OK;
  if (batch->num_reqs == 0) return MSA_ERR_SHAPE;
  if (!idx_q || !index->k_cache) return MSA_ERR_NULL;
  if (!aligned16(idx_q) || !aligned16(index->k_cache) ||
      (index->k_scale && !aligned16(index->k_scale)))
    return MSA_ERR_SHAPE;
  const size_t need = msa_workspace_size(batch->num_rows, batch->bt_stride, topk,
                                         attn->num_heads, attn->head_dim, 8 * topk);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return MSA_ERR_WORKSPACE;

  int pps, splits, ws_pps, ws_splits;
  attn_split(batch->num_rows, 8 * topk, attn_ctas_per_sm(attn), &pps, &splits);
  attn_split(batch->num_rows, 8 * topk, kMaxAttnCtasPerSm, &ws_pps, &ws_splits);
  const DecodeWs L = decode_layout(batch->num_rows, batch->bt_stride, topk, ws_splits);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  float* scores = reinterpret_cast<float*>(ws + L.scores);
  int32_t* k_idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(ws + L.topk);
  int32_t* tbl = sparse_tbl ? sparse_tbl : reinterpret_cast<int32_t*>(ws + L.tbl);
  const int tstride = sparse_tbl ? tbl_stride : 8 * topk;
  int32_t* len = sparse_len ? sparse_len : reinterpret_cast<int32_t*>(ws + L.len);

  // Rows of requests with >= kPrefillMinRows rows take the block-major
  // tensor-core attention when the batch may hold any (the max_q_len hint),
  // the KV is bf16 without per-token scales and the selection fits a list
  // entry; every other row takes the split-K decode attention.
  const bool prefill = L.prefill && batch->max_q_len >= kPrefillMinRows &&
                       attn->kv_dtype == MSA_KV_BF16 &&
                       attn->scale_mode != MSA_SCALE_PER_TOKEN_HEAD &&
                       batch->num_rows < (1 << 23) &&
                       (long long)batch->num_rows * batch->bt_stride < (1ll << 31) &&
                       prefill_attn_available();
  // every request known to bring >= kPrefillMinRows rows: no decode attention
  const bool prefill_only = prefill && batch->min_q_len >= kPrefillMinRows;
  int32_t* route = prefill ? reinterpret_cast<int32_t*>(ws + L.route) : nullptr;
  int32_t* pf_counts = prefill ? reinterpret_cast<int32_t*>(ws + L.pf_counts) : nullptr;
  int32_t* pf_lists = prefill ? reinterpret_cast<int32_t*>(ws + L.pf_lists) : nullptr;

  ScoreLaunch sp{*batch, static_cast<const uint16_t*>(idx_q),
                 static_cast<const uint8_t*>(index->k_cache), index->heads, index->dim, scores,
                 batch->bt_stride, dev_status, 0, index->dtype == MSA_KV_FP8_E4M3,
                 index->dtype == MSA_KV_FP8_E4M3 ? index->k_scale : nullptr};
  int score_kernels = 0;
  cudaError_t e = launch_scores(sp, stream, &score_kernels);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  if (trace && trace->after_score) cudaEventRecord(trace->after_score, stream);

  if (prefill) {
    // the list counters start at zero on every call, whatever another call
    // (of another shape) left in this workspace
    if (cudaMemsetAsync(pf_counts, 0, (size_t)L.max_items * 4, stream) != cudaSuccess)
      return MSA_ERR_CUDA;
  }
  TopkLaunch tp{*batch, scores,     batch->bt_stride, topk,  k_idx,   tbl, tstride,
                len,    counters,   dev_status,       route, pf_counts, pf_lists};
  e = launch_topk_table(tp, stream, true);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  if (trace && trace->after_topk) cudaEventRecord(trace->after_topk, stream);

  if (prefill) {
    PrefillLaunch pl;
    pl.batch = *batch;
    pl.q = static_cast<const uint16_t*>(attn->q);
    pl.num_heads = attn->num_heads;
    pl.k = static_cast<const uint16_t*>(attn->k_cache);
    pl.v = static_cast<const uint16_t*>(attn->v_cache);
    pl.k_scale = attn->scale_mode == MSA_SCALE_SCALAR ? attn->k_scale : nullptr;
    pl.v_scale = attn->scale_mode == MSA_SCALE_SCALAR ? attn->v_scale : nullptr;
    pl.sinks = attn->sinks;
    pl.softmax_scale = attn->softmax_scale;
    pl.topk = topk;
    pl.topk_idx = k_idx;
    pl.route = route;
    pl.pf_counts = pf_counts;
    pl.pf_lists = pf_lists;
    pl.plan_hdr = reinterpret_cast<int32_t*>(ws + L.plan_hdr);
    pl.plan_req_q = reinterpret_cast<int32_t*>(ws + L.plan_req_q);
    pl.plan_req_item = reinterpret_cast<int32_t*>(ws + L.plan_req_item);
    pl.item_rec = reinterpret_cast<int4*>(ws + L.item_rec);
    pl.item_kv = reinterpret_cast<int2*>(ws + L.item_kv);
    pl.item_chunk = reinterpret_cast<int32_t*>(ws + L.item_chunk);
    pl.item_cost = reinterpret_cast<int32_t*>(ws + L.item_cost);
    pl.max_routed_reqs = (int)L.max_routed_reqs;
    pl.max_items = (int)L.max_items;
    pl.finish_unrouted = prefill_only ? 1 : 0;
    pl.part_o = reinterpret_cast<uint16_t*>(ws + L.part_o);
    pl.part_ml = reinterpret_cast<float2*>(ws + L.part_ml);
    pl.out = static_cast<uint16_t*>(attn->out);
    pl.lse = attn->lse;
    pl.status = dev_status;
    e = launch_prefill_attn(pl, stream);
    if (e != cudaSuccess) return MSA_ERR_CUDA;
  }

  if (!prefill_only) {
    AttnLaunch ap = make_attn(attn, tbl, tstride, len, reinterpret_cast<float*>(ws + L.partials),
                              counters, pps, splits, dev_status);
    ap.route = route;  // rows of the prefill path leave at once
    // the attention split depends only on the selected width (8*topk entries).
    // Programmatic launch (its CTAs waiting on SMs while the top-k runs) pays
    // off for a grid of more CTAs than SMs; a smaller one, in clusters of up
    // to 8, measured faster as a plain launch (batched decode 34.3 -> 31.9
    // us) and without the slow steps a programmatic one saw (speculative:
    // a third of the steps ~10 us slower)
    const bool programmatic = (long long)ap.num_rows * ap.splits > device_sm_count();
    e = launch_sparse_attn(ap, stream, programmatic);
    if (e != cudaSuccess) return MSA_ERR_CUDA;
  }
  if (trace && trace->after_attn) cudaEventRecord(trace->after_attn, stream);
  if (trace) trace->kernels = score_kernels + 1 + (prefill ? 3 : 0) + (prefill_only ? 0 : 1);
  return MSA_OK;
}

size_t msa_sparse_mla_workspace_size(int32_t num_rows, int32_t num_heads, int32_t max_tokens) {
  if (num_rows < 0 || num_heads < 1 || max_tokens < 1) return 0;
  return mla_layout(num_rows, num_heads, max_tokens).total;
}

msa_status msa_sparse_mla_decode(const msa_mla_args* a, void* workspace, size_t workspace_bytes,
                                 uint32_t* dev_status, cudaStream_t stream) {
  if (!a || !dev_status) return MSA_ERR_NULL;
  if (a->num_rows < 0 || a->num_heads < 1 || a->num_tokens < 0 || a->max_tokens < 1)
    return MSA_ERR_SHAPE;
  if (a->dqk != 576 || a->dv != 512 || a->num_heads > 128 || a->num_rows > 65535)
    return MSA_ERR_UNSUPPORTED;
  if ((a->q_dtype != MSA_KV_BF16 && a->q_dtype != MSA_KV_FP8_E4M3) ||
      (a->kv_dtype != MSA_KV_BF16 && a->kv_dtype != MSA_KV_FP8_E4M3))
    return MSA_ERR_DTYPE;
  if (a->q_dtype == MSA_KV_FP8_E4M3 && a->kv_dtype != MSA_KV_FP8_E4M3)
    return MSA_ERR_UNSUPPORTED;
  if (a->num_rows == 0) return MSA_OK;
  if (!a->q || !a->kv_cache || !a->kv_indptr || !a->kv_indices || !a->out || !a->lse)
    return MSA_ERR_NULL;
  if ((a->kv_dtype == MSA_KV_FP8_E4M3 && !a->kv_scale) ||
      (a->q_dtype == MSA_KV_FP8_E4M3 && !a->q_scale))
    return MSA_ERR_NULL;
  if (!aligned16(a->q) || !aligned16(a->kv_cache) || !aligned16(a->out)) return MSA_ERR_SHAPE;
  const MlaWs L = mla_layout(a->num_rows, a->num_heads, a->max_tokens);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return MSA_ERR_WORKSPACE;
  MlaLaunch p;
  p.q = static_cast<const uint16_t*>(a->q);
  p.kv = static_cast<const uint16_t*>(a->kv_cache);
  p.num_tokens = a->num_tokens;
  p.indptr = a->kv_indptr;
  p.indices = a->kv_indices;
  p.num_rows = a->num_rows;
  p.num_heads = a->num_heads;
  p.head_groups = (a->num_heads + 15) / 16;
  p.max_tokens = a->max_tokens;
  mla_split(a->num_rows, a->num_heads, a->max_tokens, &p.splits, &p.tokens_per_split);
  p.sinks = a->sinks;
  p.softmax_scale = a->softmax_scale;
  p.out = static_cast<uint16_t*>(a->out);
  p.lse = a->lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  p.partials = reinterpret_cast<float*>(ws + L.partials);
  p.status = dev_status;
  p.kv_fp8 = a->kv_dtype == MSA_KV_FP8_E4M3;
  p.q_fp8 = a->q_dtype == MSA_KV_FP8_E4M3;
  p.q_scale = p.q_fp8 ? a->q_scale : nullptr;
  p.kv_scale = p.kv_fp8 ? a->kv_scale : nullptr;
  return cuda_status(launch_sparse_mla(p, stream));
}

msa_status msa_kv_insert(const msa_batch* batch, const void* k_new, const void* v_new,
                         int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                         int32_t kv_dtype, int32_t scale_mode, float* k_scale, float* v_scale,
                         const void* idx_new, const msa_index_cache* index, int32_t skip_index,
                         uint32_t* dev_status, cudaStream_t stream) {
  msa_status st = check_batch(batch);
  if (st != MSA_OK) return st;
  if (!dev_status) return MSA_ERR_NULL;
  if (kv_dtype != MSA_KV_BF16 && kv_dtype != MSA_KV_FP8_E4M3) return MSA_ERR_DTYPE;
  if (scale_mode < MSA_SCALE_NONE || scale_mode > MSA_SCALE_PER_TOKEN_HEAD) return MSA_ERR_DTYPE;
  if (num_kv_heads < 1) return MSA_ERR_SHAPE;
  if (head_dim != kHeadDim) return MSA_ERR_UNSUPPORTED;
  if (!skip_index) {
    st = check_index(index);
    if (st != MSA_OK) return st;
  }
  if (batch->num_rows == 0) return MSA_OK;
  if (batch->num_reqs == 0) return MSA_ERR_SHAPE;
  if (!k_new || !v_new || !k_cache || !v_cache) return MSA_ERR_NULL;
  if (!skip_index && (!idx_new || !index->k_cache)) return MSA_ERR_NULL;
  const bool fp8 = kv_dtype == MSA_KV_FP8_E4M3;
  if (fp8 && scale_mode != MSA_SCALE_NONE && (!k_scale || !v_scale)) return MSA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return MSA_ERR_SHAPE;
  if (!skip_index && (!aligned16(idx_new) || !aligned16(index->k_cache))) return MSA_ERR_SHAPE;
  KvInsertLaunch p;
  p.batch = *batch;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.idx_new = static_cast<const uint16_t*>(idx_new);
  p.num_kv_heads = num_kv_heads;
  p.index_heads = skip_index ? 0 : index->heads;
  p.index_dim = skip_index ? 0 : index->dim;
  p.k_cache = static_cast<uint8_t*>(k_cache);
  p.v_cache = static_cast<uint8_t*>(v_cache);
  p.idx_k_cache = skip_index ? nullptr : static_cast<uint16_t*>(index->k_cache);
  p.kv_fp8 = fp8;
  p.scale_mode = fp8 ? scale_mode : MSA_SCALE_NONE;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.skip_index = skip_index != 0;
  p.idx_fp8 = !skip_index && index->dtype == MSA_KV_FP8_E4M3;
  p.idx_scale = p.idx_fp8 ? index->k_scale : nullptr;
  p.status = dev_status;
  return cuda_status(launch_kv_insert(p, stream));
}

}  // extern "C"
