// topk_table.cu -- steps 2+3: top-k block selection fused with the page-16
// sparse-table build and the context-length clamp.
//
// Definitions: "Optimise MiniMax-M3 decode index and top-k on gfx950" (vLLM
// PR 54682), "Implementation breakdown" items 1 and 4 (one kernel writes the
// top-k, the page-16 sparse table and the per-row context length), and "Add
// ROCm AITER sparse paged attention for MiniMax-M3" (vLLM PR 47287),
// "Implementation breakdown" item 3 (page-16 view of the page-128 cache) and
// "Review highlights" (the zero fill must stay inside the row width).
//
// One CTA per query row.  The row's nb (<= 16384) candidate scores become
// orderable 32-bit keys in shared memory; a 4-pass 8-bit radix select finds
// the k-th largest key T and how many keys equal to T are still needed; a
// stable ballot/popc compaction in block order then emits exactly the
// selected blocks in ascending order (keys > T, plus the lowest-indexed keys
// == T), which is the unique result under the lower-index tie rule.  The
// table expansion and length follow in the same CTA.
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Block-wide exclusive count of `flag` over the CTA in thread order, plus
// the total.  Uses `scratch[kWarps]`.
__device__ __forceinline__ int block_excl_count(bool flag, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) scratch[warp] = __popc(bal);
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = scratch[w];
    before += (w < warp) ? c : 0;
    all += c;
  }
  __syncthreads();
  *total = all;
  return before + in_warp;
}

// Block-wide inclusive scan of one value per thread.
__device__ __forceinline__ int block_incl_scan(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) before += (w < warp) ? scratch[w] : 0;
  __syncthreads();
  return before + v;
}

__global__ void __launch_bounds__(kThreads) topk_table_kernel(const TopkLaunch p) {
  extern __shared__ uint32_t keys[];  // [bt_stride] keys, then [topk] selected blocks
  __shared__ uint32_t hist[256];
  __shared__ int scratch[kWarps];
  __shared__ int s_req, s_digit, s_rem, s_bad;
  const msa_batch& b = p.batch;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int R = b.num_reqs;
  int* sel = reinterpret_cast<int*>(keys + b.bt_stride);

  // ---- which request owns the row, and is it usable?
  if (tid == 0) {
    s_bad = 0;
    s_req = -1;
    if (!(b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows)) s_bad = MSA_DEV_MALFORMED;
  }
  __syncthreads();
  for (int q = tid; q < R; q += kThreads)
    if (b.cu_seqlens_q[q + 1] < b.cu_seqlens_q[q]) s_bad = MSA_DEV_MALFORMED;
  __syncthreads();
  int q = -1, q0 = 0, qlen = 0, ctx = 0, nbq = 0;
  uint32_t bad = (uint32_t)s_bad;
  if (!bad) {
    if (tid == 0) {  // largest q with cu_q[q] <= r (rows are tiled, so r < cu_q[q+1])
      int lo = 0, hi = R;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (b.cu_seqlens_q[mid] <= r) lo = mid; else hi = mid;
      }
      while (lo < R - 1 && b.cu_seqlens_q[lo + 1] <= r) ++lo;  // skip empty requests
      s_req = lo;
    }
    __syncthreads();
    q = s_req;
    bad = request_lengths(b, q, &q0, &qlen, &ctx, &nbq);
    if (!bad) {
      int page_bad = 0;
      for (int blk = tid; blk < nbq; blk += kThreads) {
        const int page = b.block_table[(long long)q * b.bt_stride + blk];
        page_bad |= (page < 0 || page >= b.num_pages);
      }
      if (__syncthreads_or(page_bad)) bad = MSA_DEV_BAD_PAGE;
    }
  }
  const bool first_row_of_req = (q >= 0) && (r == q0);
  if (bad) {
    if (tid == 0 && (first_row_of_req || (bad == MSA_DEV_MALFORMED && r == 0)))
      atomicOr(p.status, bad);
    for (int i = tid; i < p.topk; i += kThreads) p.topk_idx[(long long)r * p.topk + i] = -1;
    for (int i = tid; i < p.tbl_stride; i += kThreads) p.tbl[(long long)r * p.tbl_stride + i] = 0;
    if (tid == 0) {
      p.sparse_len[r] = 0;
      if (p.attn_counters) p.attn_counters[r] = 0;
    }
    return;
  }

  const int pos = ctx + (r - q0);
  const int L = pos + 1;
  const int n = (L + kBlock - 1) / kBlock;
  const int k = p.topk;
  const int m = min(k, n);
  const float* srow = p.scores + (long long)r * p.score_stride;

  // ---- threshold key T and the number of keys == T to take
  uint32_t T = 0;
  int need_eq = 0;
  const bool take_all = n <= k;
  if (!take_all) {
    for (int i = tid; i < n; i += kThreads) keys[i] = score_key(srow[i]);
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    __syncthreads();
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      hist[tid] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      // suffix counts: thread t looks at digit 255 - t
      const int v = (int)hist[255 - tid];
      const int incl = block_incl_scan(v, scratch);  // keys with digit >= 255 - t
      if (incl >= remaining && incl - v < remaining) {
        s_digit = 255 - tid;
        s_rem = remaining - (incl - v);
      }
      __syncthreads();
      prefix |= (uint32_t)s_digit << shift;
      mask |= 255u << shift;
      remaining = s_rem;
      __syncthreads();
    }
    T = prefix;
    need_eq = remaining;
  }

  // ---- stable compaction in block order -> ascending selected blocks
  int eq_carry = 0, sel_carry = 0;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + tid;
    uint32_t key = 0;
    if (!take_all && i < n) key = keys[i];
    const bool is_eq = !take_all && i < n && key == T;
    int eq_total;
    const int eq_before = block_excl_count(is_eq, scratch, &eq_total);
    const bool take =
        i < n && (take_all || key > T || (is_eq && eq_carry + eq_before < need_eq));
    int sel_total;
    const int at = sel_carry + block_excl_count(take, scratch, &sel_total);
    if (take) {
      sel[at] = i;
      p.topk_idx[(long long)r * k + at] = i;
    }
    eq_carry += eq_total;
    sel_carry += sel_total;
  }
  for (int i = m + tid; i < k; i += kThreads) p.topk_idx[(long long)r * k + i] = -1;
  __syncthreads();

  // ---- page-16 expansion, zero fill bounded by the row width
  const int* bt_row = b.block_table + (long long)q * b.bt_stride;
  for (int i = tid; i < p.tbl_stride; i += kThreads) {
    const int e = i >> 3, j = i & 7;
    int v = 0;
    if (e < m) {
      const int blk = sel[e];
      const int valid = min(kBlock, L - kBlock * blk);
      if (j < (valid + kPage16 - 1) / kPage16) v = 8 * bt_row[blk] + j;
    }
    p.tbl[(long long)r * p.tbl_stride + i] = v;
  }
  if (tid == 0) {
    // only the block holding the row's last token can be partial, and it is
    // the highest selected block when selected
    p.sparse_len[r] = m > 0 ? kBlock * (m - 1) + min(kBlock, L - kBlock * sel[m - 1]) : 0;
    if (p.attn_counters) p.attn_counters[r] = 0;
  }
}

}  // namespace

cudaError_t launch_topk_table(const TopkLaunch& p, cudaStream_t stream) {
  if (p.batch.num_rows == 0) return cudaSuccess;
  const size_t smem = (size_t)(p.batch.bt_stride + p.topk) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_table_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_table_kernel<<<p.batch.num_rows, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace msa
