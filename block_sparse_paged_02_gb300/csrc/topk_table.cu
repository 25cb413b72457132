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
// One CTA per row; each thread holds KPT consecutive block scores as
// orderable 32-bit keys in registers (rows of up to 1024 blocks: 1024
// threads, one key each).  The k-th largest key T is found from the top: with
// one key per thread by a radix select over four 8-bit digits (a shared
// 256-bin histogram per digit, one warp locating the bin that holds the k-th
// largest); with several keys per thread bit by bit (T takes a bit whenever
// at least k keys are >= the candidate: a warp reduction plus one barrier
// per bit).  One
// block-wide exclusive scan of the packed (== T, > T) counts then places, in
// ascending block order, every key > T and the lowest-indexed keys == T until
// k are taken -- the unique result under the lower-index tie rule.  The
// row's block-table entries are read into shared memory while the score
// kernel still runs (they are checked there anyway), so the page-16
// expansion after the selection touches no global memory but its writes.
#include "msa_internal.cuh"

namespace msa {
namespace {

// One key per thread (rows of up to 1024 blocks): the radix select has the
// shorter chain, the counting-barrier bit search fewer instructions and 32
// registers (two CTAs per SM, and room beside a score CTA while the PDL
// prologue runs).  Measured steps (same box): 16 rows of up to 1024 blocks
// 46.0-46.3 us radix against 49.2-50.4 us bit search; 64 rows of up to 1024
// blocks 85.4-85.6 against 84.9-85.4 us; 8 rows of up to 256 blocks
// 35.7-35.9 against 34.6-34.7 us; 4096 rows 139 against 106 us of top-k.
// So the radix select runs for at most MSA_TOPK_RADIX_MAX_ROWS rows whose
// table rows exceed 512 blocks.
#ifndef MSA_TOPK_RADIX_MAX_ROWS
#define MSA_TOPK_RADIX_MAX_ROWS 32
#endif
// batches of at least this many rows (with at most 1024 blocks and top-k <=
// 128) run one warp per row
#ifndef MSA_TOPK_WARP_MIN_ROWS
#define MSA_TOPK_WARP_MIN_ROWS 512
#endif

// Exclusive scan of one int per thread over a CTA of THREADS threads (two
// barriers); *total receives the sum.  scratch holds THREADS/32 + 1 ints.
template <int THREADS>
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  constexpr int kWarps = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {  // scan of the warp totals
    const int t = lane < kWarps ? scratch[lane] : 0;
    int y = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += n;
    }
    if (lane < kWarps) scratch[lane] = y - t;
    if (lane == 31) scratch[kWarps] = y;
  }
  __syncthreads();
  const int before = scratch[warp];
  *total = scratch[kWarps];
  __syncthreads();  // scratch is reused by the next scan
  return before + x - v;
}

// Fused decode with a prefill path: the row's selected block `blk` (its
// slot-th selection) joins the request's list for that block (see
// TopkLaunch).  A block is selected at most once per row, so a list never
// holds more than q_len entries.
__device__ __forceinline__ void prefill_append(const TopkLaunch& p, int q0, int qlen, int r,
                                               int slot, int blk) {
  const long long bt = p.batch.bt_stride;
  const int pos = atomicAdd(p.pf_counts + (long long)q0 * bt / kPrefillMinRows + blk, 1);
  p.pf_lists[(long long)q0 * bt + (long long)blk * qlen + pos] = (r << 8) | slot;
}

template <int KPT, int THREADS, bool RADIX>
__device__ __forceinline__ void topk_table_body(const TopkLaunch& p) {
  constexpr int kWarps = THREADS / 32;
  // [topk] selected blocks (ascending), then the request's block-table row
  extern __shared__ int sel[];
  int* pages = sel + p.topk;
  __shared__ int s_cnt[2][kWarps];
  __shared__ int s_scan[kWarps + 1];
  __shared__ int s_bad;
  __shared__ int s_hist[KPT == 1 && RADIX ? 256 : 1];
  __shared__ int s_sel[2];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const msa_batch& b = p.batch;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = b.num_reqs;
  const int k = p.topk;
  const unsigned full = 0xffffffffu;

  // ---- tiling check and the row's request: count requests starting at or before r
  if (tid == 0)
    s_bad = (b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows) ? 0 : MSA_DEV_MALFORMED;
  int le = 0;
  bool mono = true;
  for (int q = tid; q < R; q += THREADS) {
    const int c0 = b.cu_seqlens_q[q], c1 = b.cu_seqlens_q[q + 1];
    mono &= c1 >= c0;
    le += c0 <= r;
  }
  le = __reduce_add_sync(full, le);
  if (lane == 0) s_cnt[0][warp] = le;
  const bool all_mono = __syncthreads_and(mono) != 0;
  if (!all_mono && tid == 0) s_bad = MSA_DEV_MALFORMED;
  __syncthreads();
  uint32_t bad = (uint32_t)s_bad;
  int count_le = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) count_le += s_cnt[0][w];
  __syncthreads();  // s_cnt is reused below

  int q = -1, q0 = 0, qlen = 0, ctx = 0, nbq = 0, L = 0, n = 0;
  uint32_t key[KPT];
  const float* srow = p.scores + (long long)r * p.score_stride;
  if (!bad) {
    q = count_le - 1;  // cu_q is sorted and r < cu_q[R]
    bad = request_lengths(b, q, &q0, &qlen, &ctx, &nbq);
  }
  if (!bad) {
    int page_bad = 0;
    for (int blk = tid; blk < nbq; blk += THREADS) {
      const int page = b.block_table[(long long)q * b.bt_stride + blk];
      page_bad |= (page < 0 || page >= b.num_pages);
      pages[blk] = page;
    }
    if (__syncthreads_or(page_bad)) bad = MSA_DEV_BAD_PAGE;
  }
  // everything above reads only the batch geometry; the scores come from the
  // previous kernel on the stream, which may still be running until here
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!bad) {
    L = ctx + (r - q0) + 1;  // visible tokens
    n = (L + kBlock - 1) / kBlock;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int blk = KPT * tid + i;
      key[i] = blk < n ? score_key(srow[blk]) : 0u;
    }
  }
  int32_t* out_idx = p.topk_idx + (long long)r * k;
  int32_t* out_tbl = p.tbl + (long long)r * p.tbl_stride;
  if (bad) {
    const bool report = (q >= 0) ? (r == q0) : (r == 0);
    if (tid == 0 && report) atomicOr(p.status, bad);
    for (int i = tid; i < k; i += THREADS) out_idx[i] = -1;
    for (int i = tid; i < p.tbl_stride; i += THREADS) out_tbl[i] = 0;
    if (tid == 0) {
      p.sparse_len[r] = 0;
      if (p.attn_counters) p.attn_counters[r] = 0;
      if (p.route) p.route[r] = 0;  // an empty row, left to the decode attention
    }
    return;
  }

  const int m = min(k, n);
  if (n <= k) {  // every candidate is selected
    for (int i = tid; i < n; i += THREADS) {
      sel[i] = i;
      out_idx[i] = i;
    }
  } else {
    // ---- the k-th largest key T (keys of blocks >= n are 0 < any candidate)
    uint32_t T = 0;
    if constexpr (KPT == 1 && RADIX) {
      // Radix select, 8 bits per round from the top: a 256-bin histogram of
      // the next digit over the keys that match the bits found so far
      // (lanes with equal digits add once, through __match_any_sync), then
      // one warp finds the bin holding the k-th largest from the top.  Four
      // rounds of three barriers replace 32 counting barriers; the result is
      // the same k-th largest key.
      int kk = k;
      uint32_t mask = 0;
#pragma unroll 1
      for (int shift = 24; shift >= 0; shift -= 8) {
        if (tid < 256) s_hist[tid] = 0;
        __syncthreads();
        const bool in = (key[0] & mask) == T;
        const uint32_t dig = in ? (key[0] >> shift) & 255u : 256u;
        const unsigned peers = __match_any_sync(full, dig);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&s_hist[dig], __popc(peers));
        __syncthreads();
        if (warp == 0) {
          // lane l holds bins 255-8l .. 248-8l (descending)
          int h[8], sum = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            h[i] = s_hist[255 - 8 * lane - i];
            sum += h[i];
          }
          int incl = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += v;
          }
          const unsigned hit = __ballot_sync(full, incl >= kk);
          if (lane == __ffs(hit) - 1) {
            int cum = incl - sum;  // keys in higher bins
            int b = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (cum + h[i] >= kk) {
                b = 255 - 8 * lane - i;
                break;
              }
              cum += h[i];
            }
            s_sel[0] = b;
            s_sel[1] = kk - cum;
          }
        }
        __syncthreads();
        T |= (uint32_t)s_sel[0] << shift;
        mask |= 255u << shift;
        kk = s_sel[1];
      }
    } else {
#pragma unroll 1
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = T | (1u << bit);
      int total;
      if constexpr (KPT == 1) {
        total = __syncthreads_count(key[0] >= cand);
      } else {
        int c = 0;
#pragma unroll
        for (int i = 0; i < KPT; ++i) c += key[i] >= cand;
        c = __reduce_add_sync(full, c);
        if (lane == 0) s_cnt[bit & 1][warp] = c;  // double-buffered: one barrier per bit
        __syncthreads();
        total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) total += s_cnt[bit & 1][w];
      }
      if (total >= k) T = cand;
    }
    }
    // ---- keys > T, then the lowest-indexed keys == T until k are taken:
    // one scan of (count == T) << 16 | (count > T) (both < 2^16)
    int my_gt = 0, my_eq = 0;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const bool live = KPT * tid + i < n;
      my_gt += live && key[i] > T;
      my_eq += live && key[i] == T;
    }
    int packed_total;
    const int packed_before = block_excl_scan<THREADS>((my_eq << 16) | my_gt, s_scan, &packed_total);
    const int gt_before = packed_before & 0xffff, eq_before = packed_before >> 16;
    const int need_eq = k - (packed_total & 0xffff);  // the ties taken, lowest blocks first
    int gt_seen = 0, eq_seen = 0;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int blk = KPT * tid + i;
      if (blk < n) {
        const bool gt = key[i] > T, eq = key[i] == T;
        const int eq_rank = eq_before + eq_seen;
        if (gt || (eq && eq_rank < need_eq)) {
          const int at = gt_before + gt_seen + min(eq_rank, need_eq);
          sel[at] = blk;
          out_idx[at] = blk;
        }
        gt_seen += gt;
        eq_seen += eq;
      }
    }
  }
  for (int i = m + tid; i < k; i += THREADS) out_idx[i] = -1;
  __syncthreads();

  // ---- page-16 expansion (pages from shared memory), zero fill bounded by the row width
  for (int i = tid; i < p.tbl_stride; i += THREADS) {
    const int e = i >> 3, j = i & 7;
    int v = 0;
    if (e < m) {
      const int blk = sel[e];
      const int valid = min(kBlock, L - kBlock * blk);
      if (j < (valid + kPage16 - 1) / kPage16) v = 8 * pages[blk] + j;
    }
    out_tbl[i] = v;
  }
  if (tid == 0) {
    // only the block holding the row's last token can be partial, and it is
    // the highest selected block when selected
    p.sparse_len[r] = m > 0 ? kBlock * (m - 1) + min(kBlock, L - kBlock * sel[m - 1]) : 0;
    if (p.attn_counters) p.attn_counters[r] = 0;
  }
  if (p.route) {
    const bool routed = qlen >= kPrefillMinRows;
    if (tid == 0) p.route[r] = routed ? q + 1 : 0;
    if (routed)
      for (int i = tid; i < m; i += THREADS) prefill_append(p, q0, qlen, r, i, sel[i]);
  }
}

// One key per thread, radix select (few long rows): at most 40
// registers, so that a 1024-thread CTA still fits beside an attention CTA
// (launched early by PDL) on one SM.
__global__ void __maxnreg__(40) topk_table_kernel_radix(const TopkLaunch p) {
  topk_table_body<1, 1024, true>(p);
}

// One key per thread, bit search (thousands of rows): it needs 32 registers,
// so two 1024-thread CTAs share an SM (held to 40 it ran one per SM: 166
// against 106 us for 4096 rows).
__global__ void __launch_bounds__(1024) topk_table_kernel(const TopkLaunch p) {
  topk_table_body<1, 1024, false>(p);
}

template <int KPT>
__global__ void __launch_bounds__(256) topk_table_kernel_multi(const TopkLaunch p) {
  topk_table_body<KPT, 256, false>(p);
}

// ------------------------------------------------- one warp per row
//
// Thousands of rows with at most 1024 candidate blocks each (a prefill
// chunk: every new token is a row): a 1024-thread CTA per row spends most of
// its time on CTA-wide barriers and per-row set-up, so here one warp owns a
// row and a CTA of 8 warps shares the batch checks.  Lane l holds the KPL
// consecutive blocks l*KPL .. l*KPL+KPL-1, so lane order is block order; the
// k-th largest key comes from the same bit-by-bit search (one warp
// reduction per bit, no barrier), or, for 8 keys a lane and k <= 32, from k
// rounds of extraction: each lane sorts its keys once (descending), then
// every round takes the warp's largest head (one reduction) and the lowest
// lane holding it drops its head, the k-th value taken being T.  Either way
// one warp scan of the packed (== T, > T) counts places the selection, as
// in the CTA form above.
constexpr int kWarpRows = 8;            // rows (warps) per CTA
constexpr int kWarpTopkMax = 128;       // largest k of the warp form
constexpr int kExtractMaxK = 32;        // largest k found by extraction

// Sorts 8 keys into descending order (Batcher's odd-even merge network,
// 19 compare-exchanges).
__device__ __forceinline__ void sort8_desc(uint32_t (&v)[8]) {
  constexpr int kNet[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6},
                               {5, 7}, {1, 2}, {5, 6}, {0, 4}, {1, 5}, {2, 6}, {3, 7},
                               {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) {
    const uint32_t a = v[kNet[c][0]], b = v[kNet[c][1]];
    v[kNet[c][0]] = max(a, b);
    v[kNet[c][1]] = min(a, b);
  }
}

template <int KPL>
__global__ void __launch_bounds__(kWarpRows * 32) topk_table_kernel_warp(const TopkLaunch p) {
  extern __shared__ int wsm[];
  int* cuq = wsm;                             // [R + 1] cu_seqlens_q
  int* sel_all = wsm + p.batch.num_reqs + 1;  // [kWarpRows][topk] selected blocks
  __shared__ int s_bad;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const msa_batch& b = p.batch;
  const int R = b.num_reqs;
  const int k = p.topk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned full = 0xffffffffu;

  // ---- batch checks shared by the CTA's rows: cu_seqlens_q tiles the rows
  if (tid == 0)
    s_bad = (b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows) ? 0 : MSA_DEV_MALFORMED;
  bool mono = true;
  for (int q = tid; q <= R; q += blockDim.x) {
    const int c = b.cu_seqlens_q[q];
    cuq[q] = c;
    if (q < R) mono &= b.cu_seqlens_q[q + 1] >= c;
  }
  const bool all_mono = __syncthreads_and(mono) != 0;
  if (!all_mono && tid == 0) s_bad = MSA_DEV_MALFORMED;
  __syncthreads();

  const int r = blockIdx.x * kWarpRows + warp;
  if (r >= b.num_rows) return;
  int* sel = sel_all + warp * k;
  uint32_t bad = (uint32_t)s_bad;
  int q = -1, q0 = 0, qlen = 0, ctx = 0, nbq = 0;
  if (!bad) {
    // the row's request: the last q with cu_q[q] <= r (cu_q sorted, r < cu_q[R])
    int lo = 0, hi = R;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cuq[mid] <= r) lo = mid; else hi = mid;
    }
    q = lo;
    bad = request_lengths(b, q, &q0, &qlen, &ctx, &nbq);
  }
  if (!bad) {
    int page_bad = 0;
    for (int blk = lane; blk < nbq; blk += 32) {
      const int page = b.block_table[(long long)q * b.bt_stride + blk];
      page_bad |= (page < 0 || page >= b.num_pages);
    }
    if (__any_sync(full, page_bad)) bad = MSA_DEV_BAD_PAGE;
  }
  // everything above reads only the batch geometry; the scores come from the
  // previous kernel on the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int32_t* out_idx = p.topk_idx + (long long)r * k;
  int32_t* out_tbl = p.tbl + (long long)r * p.tbl_stride;
  if (bad) {
    const bool report = (q >= 0) ? (r == q0) : (r == 0);
    if (lane == 0 && report) atomicOr(p.status, bad);
    for (int i = lane; i < k; i += 32) out_idx[i] = -1;
    for (int i = lane; i < p.tbl_stride; i += 32) out_tbl[i] = 0;
    if (lane == 0) {
      p.sparse_len[r] = 0;
      if (p.attn_counters) p.attn_counters[r] = 0;
      if (p.route) p.route[r] = 0;  // an empty row, left to the decode attention
    }
    return;
  }
  const int L = ctx + (r - q0) + 1;  // visible tokens
  const int n = (L + kBlock - 1) / kBlock;
  const float* srow = p.scores + (long long)r * p.score_stride;
  const int m = min(k, n);
  if (n <= k) {  // every candidate is selected
    for (int i = lane; i < n; i += 32) {
      sel[i] = i;
      out_idx[i] = i;
    }
  } else {
    uint32_t key[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int blk = KPL * lane + i;
      key[i] = blk < n ? score_key(srow[blk]) : 0u;  // 0 ranks below every candidate
    }
    // ---- the k-th largest key T
    uint32_t T = 0;
    if (KPL == 8 && k <= kExtractMaxK) {
      // k rounds of extraction: each lane's keys sorted, the largest head
      // taken per round (ties: any holder; only the value matters)
      uint32_t h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = key[i % KPL];
      sort8_desc(h);
#pragma unroll 1
      for (int t = 0; t < k; ++t) {
        T = __reduce_max_sync(full, h[0]);
        if (T == 0u) break;  // every key left is 0: so is the k-th
        const unsigned holders = __ballot_sync(full, h[0] == T);
        if (lane == __ffs(holders) - 1) {
#pragma unroll
          for (int i = 0; i < 7; ++i) h[i] = h[i + 1];
          h[7] = 0u;
        }
      }
    } else {
      // bit by bit from the top: T takes a bit whenever at least k keys are
      // >= the candidate
#pragma unroll 1
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = T | (1u << bit);
        int c = 0;
#pragma unroll
        for (int i = 0; i < KPL; ++i) c += key[i] >= cand;
        if (__reduce_add_sync(full, c) >= k) T = cand;
      }
    }
    // ---- keys > T, then the lowest-indexed keys == T until k are taken
    int my_gt = 0, my_eq = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const bool live = KPL * lane + i < n;
      my_gt += live && key[i] > T;
      my_eq += live && key[i] == T;
    }
    const int packed = (my_eq << 16) | my_gt;
    int incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(full, incl, o);
      if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(full, incl, 31);
    const int before = incl - packed;
    const int gt_before = before & 0xffff, eq_before = before >> 16;
    const int need_eq = k - (total & 0xffff);
    int gt_seen = 0, eq_seen = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int blk = KPL * lane + i;
      if (blk < n) {
        const bool gt = key[i] > T, eq = key[i] == T;
        const int eq_rank = eq_before + eq_seen;
        if (gt || (eq && eq_rank < need_eq)) {
          const int at = gt_before + gt_seen + min(eq_rank, need_eq);
          sel[at] = blk;
          out_idx[at] = blk;
        }
        gt_seen += gt;
        eq_seen += eq;
      }
    }
  }
  for (int i = m + lane; i < k; i += 32) out_idx[i] = -1;
  __syncwarp();

  // ---- page-16 expansion, zero fill bounded by the row width
  const int32_t* bt_row = b.block_table + (long long)q * b.bt_stride;
  for (int i = lane; i < p.tbl_stride; i += 32) {
    const int e = i >> 3, j = i & 7;
    int v = 0;
    if (e < m) {
      const int blk = sel[e];
      const int valid = min(kBlock, L - kBlock * blk);
      if (j < (valid + kPage16 - 1) / kPage16) v = 8 * __ldg(bt_row + blk) + j;
    }
    out_tbl[i] = v;
  }
  if (lane == 0) {
    // only the block holding the row's last token can be partial, and it is
    // the highest selected block when selected
    p.sparse_len[r] = m > 0 ? kBlock * (m - 1) + min(kBlock, L - kBlock * sel[m - 1]) : 0;
    if (p.attn_counters) p.attn_counters[r] = 0;
  }
  if (p.route) {
    const bool routed = qlen >= kPrefillMinRows;
    if (lane == 0) p.route[r] = routed ? q + 1 : 0;
    if (routed)
      for (int i = lane; i < m; i += 32) prefill_append(p, q0, qlen, r, i, sel[i]);
  }
}

template <int KPL>
cudaError_t launch_warp(const TopkLaunch& p, cudaStream_t stream, bool programmatic) {
  auto kern = topk_table_kernel_warp<KPL>;
  const size_t smem = (size_t)(p.batch.num_reqs + 1 + kWarpRows * p.topk) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.batch.num_rows + kWarpRows - 1) / kWarpRows);
  cfg.blockDim = dim3(kWarpRows * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int KPT, int THREADS, bool RADIX = false>
cudaError_t launch_kpt(const TopkLaunch& p, cudaStream_t stream, bool programmatic) {
  void (*kern)(const TopkLaunch);
  if constexpr (KPT == 1 && RADIX)
    kern = topk_table_kernel_radix;
  else if constexpr (KPT == 1)
    kern = topk_table_kernel;
  else
    kern = topk_table_kernel_multi<KPT>;
  const size_t smem = (size_t)(p.topk + p.batch.bt_stride) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch.num_rows);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_topk_table(const TopkLaunch& p, cudaStream_t stream, bool programmatic) {
  if (p.batch.num_rows == 0) return cudaSuccess;
  // a row has at most bt_stride candidate blocks
  if (p.batch.num_rows >= MSA_TOPK_WARP_MIN_ROWS && p.topk <= kWarpTopkMax &&
      p.batch.bt_stride <= 1024) {
    if (p.batch.bt_stride <= 256) return launch_warp<8>(p, stream, programmatic);
    if (p.batch.bt_stride <= 512) return launch_warp<16>(p, stream, programmatic);
    return launch_warp<32>(p, stream, programmatic);
  }
  if (p.batch.bt_stride <= 1024) {
    if (p.batch.num_rows <= MSA_TOPK_RADIX_MAX_ROWS && p.batch.bt_stride > 512)
      return launch_kpt<1, 1024, true>(p, stream, programmatic);
    return launch_kpt<1, 1024, false>(p, stream, programmatic);
  }
  if (p.batch.bt_stride <= 256 * 16) return launch_kpt<16, 256>(p, stream, programmatic);
  return launch_kpt<64, 256>(p, stream, programmatic);
}

}  // namespace msa
