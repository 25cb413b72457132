// index_score.cu -- step 1: block scores of the index query against the paged
// index-K cache.
//
// Definition ("Optimise MiniMax-M3 decode index and top-k on gfx950", vLLM PR
// 54682, "Implementation breakdown" item 1 and "Key files"): each cached
// 128-token block of a request gets, for every query row of that request, the
// maximum over the block's visible tokens (t <= the row's position) and over
// index heads of the dot product idx_q[row] . idx_k[t].
//
// GB300 design.  The index-K scan is the dominant byte stream of the decode
// path and is HBM-bound (~1 FMA per 2 bytes for one row), so the kernel is a
// persistent, bandwidth-first streamer:
//   * work = the flattened list of (request, block) items over all requests;
//     each CTA takes an equal contiguous slice (balanced by actual block
//     count, the lesson of the PR 54682 balanced scorer; consecutive items
//     share block-table lines, so the producer's lookups stay cache hits);
//   * two producer threads (one per producer warp, alternate items) issue
//     one async copy per 128-token index-K page (16 or 32 KB, contiguous in
//     the page-128 layout), plus one for the query rows that see it, into a
//     ring of shared-memory stages guarded by mbarriers;
//   * each consumer warp owns one stage and scores the whole page
//     (warp-per-block): every lane holds 4*Hi token sub-rows, walks their
//     16-byte chunks in a lane-rotated order (bank-conflict free), and keeps
//     fp32 dot products for up to 4 query rows of the request at once, so a
//     staged page is shared by all rows of the request;
//   * a warp max-reduce produces the block score; integer-valued inputs give
//     exact fp32 scores.
#include <cfloat>

#include <string.h>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kRowGroup = 4;
// bf16 keys: requests of at least this many rows (max_q_len hint) -> MMA scorer
constexpr int kMmaMinRows = 2;

// Scoring kinds: bf16 keys on CUDA-core FMAs, OCP e4m3 keys on warp MMA
// (fp16 operands), and bf16 keys on warp MMA with two consumer warps per
// stage, each scoring half of a page's token tiles (one warp took ~4.9 K
// cycles for a 32 KiB page, about as long as the page's copy, and a stage
// is held for both, so halving the scoring lets the 6-page ring turn over
// faster).
enum { kFmaBf16 = 0, kMmaFp8 = 2, kMmaBf16Pair = 3 };

// producer warps of the score kernel (each issues every kProducers-th item)
#ifndef MSA_SCORE_PRODUCERS
#define MSA_SCORE_PRODUCERS 2
#endif
#ifndef MSA_SCORE_PRODUCERS_FP8
#define MSA_SCORE_PRODUCERS_FP8 2
#endif

// Shared-memory budget of the stage ring: 200 KB leaves room for the
// request prefix of the largest batches; e4m3 pages (~18.5 KB a stage) take
// a second build of the kernel with a 222 KB ring (12 stages instead of 10)
// whenever the batch's prefix still fits beside it: the ring is what hides
// the copy latency (a stage is held for a page's load plus its scoring).
constexpr int kStageBudget = 204800;
constexpr int kStageBudgetWide = 227328;
constexpr size_t kMaxDynSmem = 232448;  // the opt-in limit per CTA (227 KB)

template <int DI, int HI, int KIND, int BUDGET = kStageBudget>
struct ScoreCfg {
  static constexpr int kProducers = KIND == kMmaFp8 ? MSA_SCORE_PRODUCERS_FP8 : MSA_SCORE_PRODUCERS;
  static constexpr int kElem = KIND == kMmaFp8 ? 1 : 2;
  static constexpr int kPageBytes = kBlock * HI * DI * kElem;
  // query rows scored per pass: 4 for bf16 keys (FMA or MMA: the stage's
  // query copy stays small, so the ring keeps 6 stages), 8 / HI for e4m3
  // keys (the MMA's 8 columns)
  static constexpr int kRows = KIND == kMmaFp8 ? 8 / HI : kRowGroup;
  static constexpr int kQBytes = kRows * HI * DI * 2;  // query rows staged with a page
  static constexpr int kScaleBytes = KIND == kMmaFp8 ? kBlock * HI * 4 : 0;  // per-token scales
  // stages within the budget (the rest holds barriers and the request
  // prefix): 6 for 32 KB pages, 10-12 for 16 KB ones
  static constexpr int kStageBytes = kPageBytes + kQBytes + kScaleBytes;
  static constexpr int kStages =
      (BUDGET / kStageBytes < 12 ? BUDGET / kStageBytes : 12) / kProducers * kProducers;
  // consumer warps per stage: one (for the FMA scorer a pair of warps per
  // page measured slower: more instructions without more bytes in flight),
  // two for kMmaBf16Pair
  static constexpr int kCps = KIND == kMmaBf16Pair ? 2 : 1;
  static constexpr int kThreads = 32 * (kProducers + kStages * kCps);
  static_assert(kStages % kProducers == 0, "every stage needs a single producer");
};

// Pages for the MMA scorer with 128 dims and one head arrive by tensor
// copies with the 128-byte swizzle: e4m3 keys as one box of 128 rows x 128 B,
// bf16 keys as two (dims 0-63, then 64-127, 16 KB apart), so that the
// scorer's reads of rows a page row apart fall in distinct banks
#ifndef MSA_SCORE_FP8_SWIZZLE
#define MSA_SCORE_FP8_SWIZZLE 1
#endif
template <int DI, int HI, int KIND>
constexpr bool kSwizzledPages = MSA_SCORE_FP8_SWIZZLE && KIND != kFmaBf16 && DI == 128 && HI == 1;

struct StageInfo {  // written by the producer before it arms the stage
  int req, blk, valid, q0, qlen, ctx, jstart, pad;
};

// The two consumer warps of one stage (named barrier 1 + stage, 64 threads):
// AND of a predicate over both, and a plain rendezvous.
__device__ __forceinline__ bool pair_and(bool v, int id) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, 64, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

template <int DI, int HI, int KIND, int BUDGET = kStageBudget>
struct ScoreSmem {
  using C = ScoreCfg<DI, HI, KIND, BUDGET>;
  static constexpr size_t kPages = 0;
  static constexpr size_t kQ = kPages + (size_t)C::kStages * C::kPageBytes;
  static constexpr size_t kScale = kQ + (size_t)C::kStages * C::kQBytes;
  static constexpr size_t kBars = kScale + (size_t)C::kStages * C::kScaleBytes;
  static constexpr size_t kInfo = kBars + 2 * C::kStages * sizeof(uint64_t);
  static constexpr size_t kMisc = kInfo + C::kStages * sizeof(StageInfo);
  // two consumers per stage: the second one's row maxima, by row-group parity
  static constexpr size_t kRed = kMisc + 64;
  static constexpr size_t kPrefix =
      kRed + (C::kCps == 2 ? (size_t)C::kStages * 2 * kRowGroup * sizeof(float) : 0);
  static size_t bytes(int num_reqs) { return kPrefix + (size_t)(num_reqs + 1) * sizeof(int); }
};

// Scores of one staged page for NR (<= kRowGroup) query rows held in q_s.
// Returns, in lane 0..NR-1 order via out[], the per-row block maxima.
template <int DI, int HI, int NR>
__device__ __forceinline__ void score_page(const uint8_t* page, const uint8_t* q_s, int lane,
                                           int blk, const int (&pos)[kRowGroup],
                                           float (&out)[kRowGroup]) {
  constexpr int kSubPerLane = kBlock * HI / 32;  // token sub-rows of a lane
  constexpr int kChunks = DI / 8;                 // 16-byte chunks per bf16 sub-row
  constexpr int kSubRowBytes = DI * 2;
  float acc[kSubPerLane][NR];
#pragma unroll
  for (int j = 0; j < kSubPerLane; ++j)
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[j][r] = 0.f;
  const int head = lane % HI;  // sub-row lane+32j holds index head (lane % HI)
#pragma unroll 2
  for (int i = 0; i < kChunks; ++i) {
    const int c = (i + lane) & (kChunks - 1);
    float qf[NR][8];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const uint4 w = lds128(q_s + ((r * HI + head) * DI + c * 8) * 2);
      qf[r][0] = bf16lo(w.x);
      qf[r][1] = bf16hi(w.x);
      qf[r][2] = bf16lo(w.y);
      qf[r][3] = bf16hi(w.y);
      qf[r][4] = bf16lo(w.z);
      qf[r][5] = bf16hi(w.z);
      qf[r][6] = bf16lo(w.w);
      qf[r][7] = bf16hi(w.w);
    }
#pragma unroll
    for (int j = 0; j < kSubPerLane; ++j) {
      const int sr = lane + 32 * j;
      const uint4 w = lds128(page + sr * kSubRowBytes + c * 16);
      const float k0 = bf16lo(w.x), k1 = bf16hi(w.x), k2 = bf16lo(w.y), k3 = bf16hi(w.y);
      const float k4 = bf16lo(w.z), k5 = bf16hi(w.z), k6 = bf16lo(w.w), k7 = bf16hi(w.w);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float a = acc[j][r];
        a = fmaf(qf[r][0], k0, a);
        a = fmaf(qf[r][1], k1, a);
        a = fmaf(qf[r][2], k2, a);
        a = fmaf(qf[r][3], k3, a);
        a = fmaf(qf[r][4], k4, a);
        a = fmaf(qf[r][5], k5, a);
        a = fmaf(qf[r][6], k6, a);
        a = fmaf(qf[r][7], k7, a);
        acc[j][r] = a;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kSubPerLane; ++j) {
      const int token = (lane + 32 * j) / HI;
      if (blk * kBlock + token <= pos[r]) m = fmaxf(m, acc[j][r]);  // NaN never wins
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    out[r] = m;
  }
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p))
               : "memory");
  return v;
}

// Scores of one staged page on warp MMA: S^T = K Q^T with m16n8k16 tiles of
// 16 (token, head) sub-rows x 8 columns (query row, index head) x 16 dims,
// fp32 accumulation; e4m3 keys enter as their exact fp16 images and the
// queries as fp16, bf16 keys and queries as they are.  Lane (g, c) holds, for
// k-step kk, the dims c*DI/4 + 4kk + {0..3} of its rows (the same k-slot
// permutation on both operands), so each sub-row span is a contiguous read.
// Then, per column, the masked maximum over the block's tokens of
// scale_t * S (a column only sees sub-rows of its own head).  Returns in
// best[0..8/HI) the block score of each query row (all lanes).
template <int DI, int HI, bool F8, bool SWZ>
__device__ __forceinline__ void score_page_mma(const uint8_t* page, const float* tscale,
                                               const uint8_t* q_s, int nr, int lane, int blk,
                                               const int (&pos)[8], float (&best)[8],
                                               int mt0, int mt1) {
  constexpr int kK = DI / 16;                 // k-steps
  constexpr int kD4 = DI / 4;                 // dims of a lane per sub-row
  constexpr int kElem = F8 ? 1 : 2;
  constexpr int kRowB = DI * kElem;           // bytes per sub-row
  constexpr int kSpanW = kD4 * kElem / 4;     // 32-bit words of a lane's span
  constexpr int kSpanC = kSpanW / 4;          // 16-byte chunks of a lane's span
  const int g = lane >> 2, c = lane & 3;
  // B: column g = (query row g / HI, index head g % HI)
  uint32_t bq[kK][2];
  {
    const int r = g / HI, h = g % HI;
    const uint8_t* qrow = q_s + ((r * HI + h) * DI + c * kD4) * 2;
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      uint2 w = make_uint2(0u, 0u);
      if (r < nr) w = lds64(qrow + 8 * kk);
      if constexpr (F8) {
        bq[kk][0] = pack_f16x2(bf16lo(w.x), bf16hi(w.x));
        bq[kk][1] = pack_f16x2(bf16lo(w.y), bf16hi(w.y));
      } else {
        bq[kk][0] = w.x;
        bq[kk][1] = w.y;
      }
    }
  }
  // the lane's two columns: their query row, head and last visible token
  int lim[2], hcol[2];
  bool live[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int col = 2 * c + k, r = col / HI;
    int pr = pos[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (i == r) pr = pos[i];
    live[k] = r < nr;
    lim[k] = pr - blk * kBlock;  // tokens t <= lim are visible
    hcol[k] = col % HI;
  }
  // every sub-row of the block visible to both columns: no per-token mask
  const bool whole = (!live[0] || lim[0] >= kBlock - 1) && (!live[1] || lim[1] >= kBlock - 1);
  float m[2] = {-INFINITY, -INFINITY};
#pragma unroll 2
  for (int mt = mt0; mt < mt1; ++mt) {
    // spans of sub-rows 16mt + g and 16mt + g + 8.  Unswizzled, lanes of one
    // column group read the same bytes of rows a page row apart (bank
    // conflicts; rotating the read order per lane would need run-time
    // register indexing, which measured far more costly); swizzled pages
    // place those bytes in distinct banks.
    uint32_t w[2][kSpanW];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint8_t* row = page + (16 * mt + g + 8 * half) * kRowB;
#pragma unroll
      for (int i = 0; i < kSpanC; ++i) {
        // swizzled pages: 16-byte chunk j of sub-row t sits in box j / 8
        // (128 rows x 128 B each) at chunk (j % 8) ^ (t % 8) (t % 8 == g here)
        const int chunk = c * kSpanC + i;
        const uint4 v =
            SWZ ? lds128(page + (chunk >> 3) * (kBlock * 128) + (16 * mt + g + 8 * half) * 128 +
                         16 * ((chunk & 7) ^ g))
                : lds128(row + 16 * chunk);
        w[half][4 * i] = v.x;
        w[half][4 * i + 1] = v.y;
        w[half][4 * i + 2] = v.z;
        w[half][4 * i + 3] = v.w;
      }
    }
    // two accumulators (even / odd k-steps) halve the dependent MMA chain
    float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      uint32_t a[4];
      if constexpr (F8) {
        a[0] = e4m3x2_to_f16x2((uint16_t)(w[0][kk] & 0xffffu));
        a[1] = e4m3x2_to_f16x2((uint16_t)(w[1][kk] & 0xffffu));
        a[2] = e4m3x2_to_f16x2((uint16_t)(w[0][kk] >> 16));
        a[3] = e4m3x2_to_f16x2((uint16_t)(w[1][kk] >> 16));
      } else {
        a[0] = w[0][2 * kk];
        a[1] = w[1][2 * kk];
        a[2] = w[0][2 * kk + 1];
        a[3] = w[1][2 * kk + 1];
      }
      mma16816<F8>((kk & 1) ? d2 : d, a, bq[kk][0], bq[kk][1]);
    }
    float sc[2] = {1.f, 1.f};
    if (tscale) {
      sc[0] = tscale[16 * mt + g];
      sc[1] = tscale[16 * mt + g + 8];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int sr = 16 * mt + g + 8 * (e >> 1);  // sub-row = token * HI + head
      const int k = e & 1;
      const float v = (d[e] + d2[e]) * sc[e >> 1];
      const bool ok = whole ? (HI == 1 || (sr % HI) == hcol[k]) && live[k]
                            : live[k] && (sr % HI) == hcol[k] && sr / HI <= lim[k];
      if (ok) m[k] = fmaxf(m[k], v);  // NaN never wins
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) m[k] = fmaxf(m[k], __shfl_xor_sync(0xffffffffu, m[k], o));
  // lane c now holds columns 2c, 2c+1; gather the rows
#pragma unroll
  for (int r = 0; r < 8 / HI; ++r) {
    if constexpr (HI == 1) {
      const float a0 = __shfl_sync(0xffffffffu, m[0], r >> 1);
      const float a1 = __shfl_sync(0xffffffffu, m[1], r >> 1);
      best[r] = (r & 1) ? a1 : a0;
    } else {
      best[r] = fmaxf(__shfl_sync(0xffffffffu, m[0], r), __shfl_sync(0xffffffffu, m[1], r));
    }
  }
}

template <int DI, int HI, int KIND, int BUDGET>
__global__ void __launch_bounds__(ScoreCfg<DI, HI, KIND, BUDGET>::kThreads, 1)
    index_score_kernel(const ScoreLaunch p, const __grid_constant__ CUtensorMap kmap) {
  using C = ScoreCfg<DI, HI, KIND, BUDGET>;
  using S = ScoreSmem<DI, HI, KIND, BUDGET>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
  uint64_t* empty = full + C::kStages;
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + S::kInfo);
  int* misc = reinterpret_cast<int*>(smem + S::kMisc);
  int* prefix = reinterpret_cast<int*>(smem + S::kPrefix);

  const msa_batch& b = p.batch;
  const int R = b.num_reqs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the next kernel on the stream may start its prologue now; it waits on the
  // device for this grid's scores before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- setup: per-request block counts, batch checks, prefix sums
  if (tid == 0) {
    misc[0] = 0;  // per-request status bits seen by this CTA
    // rows must be tiled by cu_seqlens_q, else no row maps to a request
    misc[1] = !(b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows);
  }
  if (tid < C::kStages) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], C::kCps);
  }
  fence_barrier_init();
  __syncthreads();
  for (int q = tid; q < R; q += blockDim.x) {
    int q0, ql, ctx, nb;
    const uint32_t bad = request_lengths(b, q, &q0, &ql, &ctx, &nb);
    if (ql < 0) misc[1] = 1;
    if (bad) {
      atomicOr(reinterpret_cast<unsigned*>(&misc[0]), bad);
      nb = 0;
    }
    if (ql <= 0) nb = 0;  // no query row needs these blocks
    if (p.tc_min_rows > 0 && ql >= p.tc_min_rows) nb = 0;  // scored on the tensor cores
    prefix[q + 1] = nb;
  }
  __syncthreads();
  if (misc[1]) {  // the batch cannot be mapped: score nothing
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.status, MSA_DEV_MALFORMED);
    return;
  }
  if (warp == 0) {  // inclusive scan of block counts -> prefix[0..R]
    int carry = 0;
    if (lane == 0) prefix[0] = 0;
    for (int base = 0; base < R; base += 32) {
      const int q = base + lane;
      int v = q < R ? prefix[q + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (q < R) prefix[q + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0 && misc[0]) atomicOr(p.status, (unsigned)misc[0]);

  const long long total = prefix[R];
  const int i0 = (int)(total * blockIdx.x / gridDim.x);
  const int i1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const int n_items = i1 - i0;

  if (warp < C::kProducers) {
    // ---- producer warps: warp pw issues the items j = pw (mod kProducers),
    // so every stage has one producer (kStages is a multiple of kProducers).
    // An item lookup (request by binary search over the prefix, its row
    // range, and the page id from the block table) costs a global-memory
    // round trip; a warp's share of the first ring is looked up by one lane
    // each in parallel, then its elected lane keeps one lookup in flight
    // ahead of the copy it is about to issue.  One producer paces the e4m3
    // stream: its per-item lookup and three copy issues take longer than the
    // consumers need for a 16 KB page.
    // consecutive items mostly share a request: its row range and context
    // are kept from the previous lookup of this lane
    int c_req = -1, c_q0 = 0, c_qlen = 0, c_ctx = 0;
    auto lookup = [&](int j, StageInfo* si, int* page) {
      const int it = i0 + j;
      int lo;
      if (c_req >= 0 && prefix[c_req] <= it && it < prefix[c_req + 1]) {
        lo = c_req;
      } else {
        lo = 0;
        int hi = R;  // largest q with prefix[q] <= it
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (prefix[mid] <= it) lo = mid; else hi = mid;
        }
        c_req = lo;
        c_q0 = b.cu_seqlens_q[lo];
        c_qlen = b.cu_seqlens_q[lo + 1] - c_q0;
        c_ctx = b.context_lens[lo];
      }
      si->req = lo;
      si->blk = it - prefix[lo];
      si->q0 = c_q0;
      si->qlen = c_qlen;
      si->ctx = c_ctx;
      si->jstart = max(0, si->blk * kBlock - si->ctx);  // first row that sees the block
      si->pad = 0;
      *page = b.block_table[(long long)lo * b.bt_stride + si->blk];
      si->valid = *page >= 0 && *page < b.num_pages;
    };
    // One stage = the index-K page plus the query rows of the first row
    // group that sees it (up to 4 rows, contiguous), so that consumers need
    // no global load in the common (decode) case.
    auto issue = [&](int j, const StageInfo& si, int page) {  // elected lane only
      const int s = j % C::kStages;
      info[s] = si;
      if (si.valid) {
        const uint32_t qb = (uint32_t)min(C::kRows, si.qlen - si.jstart) * HI * DI * 2;
        const uint32_t sb = (KIND == kMmaFp8 && p.idx_scale) ? (uint32_t)C::kScaleBytes : 0u;
        mbar_arrive_expect_tx(&full[s], C::kPageBytes + qb + sb);
        if (sb)
          bulk_g2s(smem + S::kScale + (size_t)s * C::kScaleBytes,
                   p.idx_scale + (long long)page * kBlock * HI, sb, &full[s]);
        bulk_g2s(smem + S::kQ + (size_t)s * C::kQBytes,
                 p.idx_q + (long long)(si.q0 + si.jstart) * HI * DI, qb, &full[s]);
        if constexpr (kSwizzledPages<DI, HI, KIND>) {  // 128 x 128 B boxes, 128-byte swizzle
#pragma unroll
          for (int h = 0; h < C::kPageBytes / (kBlock * 128); ++h)
            tma_load_2d(smem + S::kPages + (size_t)s * C::kPageBytes + h * (kBlock * 128), &kmap,
                        64 * h, page * kBlock, &full[s]);
        } else
          bulk_g2s(smem + S::kPages + (size_t)s * C::kPageBytes,
                   p.idx_k + (long long)page * C::kPageBytes, C::kPageBytes, &full[s]);
      } else {
        atomicOr(p.status, MSA_DEV_BAD_PAGE);
        mbar_arrive(&full[s]);
      }
    };
    const int pw = warp;
    constexpr int kProducers = C::kProducers;
    const int n_mine = n_items > pw ? (n_items - pw + kProducers - 1) / kProducers : 0;
    const int first = min(C::kStages / kProducers, n_mine);  // this warp's share of the empty ring
    StageInfo mine{0, 0, 0, 0, 0, 0, 0, 0};
    int my_page = -1;
    if (lane < first) lookup(pw + kProducers * lane, &mine, &my_page);
    for (int t = 0; t < first; ++t) {  // the ring starts empty: no waits
      StageInfo si;
      si.req = __shfl_sync(0xffffffffu, mine.req, t);
      si.blk = __shfl_sync(0xffffffffu, mine.blk, t);
      si.valid = __shfl_sync(0xffffffffu, mine.valid, t);
      si.q0 = __shfl_sync(0xffffffffu, mine.q0, t);
      si.qlen = __shfl_sync(0xffffffffu, mine.qlen, t);
      si.ctx = __shfl_sync(0xffffffffu, mine.ctx, t);
      si.jstart = __shfl_sync(0xffffffffu, mine.jstart, t);
      si.pad = 0;
      const int pg = __shfl_sync(0xffffffffu, my_page, t);
      if (lane == 0) issue(pw + kProducers * t, si, pg);
    }
    if (lane == 0 && first < n_mine) {
      StageInfo next;
      int next_page;
      lookup(pw + kProducers * first, &next, &next_page);
      for (int t = first; t < n_mine; ++t) {
        const int j = pw + kProducers * t;
        const StageInfo cur = next;
        const int cur_page = next_page;
        if (t + 1 < n_mine) lookup(j + kProducers, &next, &next_page);  // in flight during the wait
        const int s = j % C::kStages, use = j / C::kStages;
        if (!mbar_wait(&empty[s], (use - 1) & 1)) {
          atomicOr(p.status, MSA_DEV_TIMEOUT);
          break;
        }
        issue(j, cur, cur_page);
      }
    }
    return;
  }

  // ---- consumers: warps kProducers + kCps s .. + kCps - 1 own stage s; with
  // two, warp `part` scores m-tiles [part, part + 1) * kMt / 2 of each page
  // and the pair joins its row maxima through shared memory.  The pair
  // decides together whether to go on (a timed-out wait ends both), so
  // neither is left at their barrier.
  constexpr int kCps = C::kCps;
  constexpr int kMt = kBlock * HI / 16;  // m-tiles of a page
  const int st = (warp - C::kProducers) / kCps, part = (warp - C::kProducers) % kCps;
  const int bar_id = 1 + st;
  const int mt0 = part * (kMt / kCps), mt1 = mt0 + kMt / kCps;
  const uint8_t* page = smem + S::kPages + (size_t)st * C::kPageBytes;
  uint8_t* q_s = smem + S::kQ + (size_t)st * C::kQBytes;
  float* red = reinterpret_cast<float*>(smem + S::kRed) + st * 2 * kRowGroup;
  for (int j = st, use = 0; j < n_items; j += C::kStages, ++use) {
    // warp-uniform: the page is scored with warp shuffles
    bool ok = __all_sync(0xffffffffu, mbar_wait(&full[st], use & 1));
    if constexpr (kCps == 2) ok = pair_and(ok, bar_id);
    if (!ok) {
      if (lane == 0) atomicOr(p.status, MSA_DEV_TIMEOUT);
      break;
    }
    const StageInfo si = info[st];
    const int q0 = si.q0, qlen = si.qlen, ctx = si.ctx;
    bool wrote_q = false;
    // rows j >= jstart (ctx + j >= 128*blk) can see this block
    for (int g0 = si.jstart, grp = 0; g0 < qlen; g0 += C::kRows, ++grp) {
      const int nr = min(C::kRows, qlen - g0);
      int pos[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) pos[r] = ctx + g0 + min(r, nr - 1);
      float best[8];
      if (si.valid) {
        if (g0 != si.jstart) {  // later row groups (requests with > 4 rows): from global
          if constexpr (kCps == 2) pair_sync(bar_id);  // both have read the previous rows
          if (part == 0) {
            __syncwarp();
            const int chunks = nr * HI * DI / 8;
            const uint4* src = reinterpret_cast<const uint4*>(
                p.idx_q + (long long)(q0 + g0) * HI * DI);
            for (int c = lane; c < chunks; c += 32)
              *reinterpret_cast<uint4*>(q_s + c * 16) = src[c];
            __syncwarp();
            wrote_q = true;
          }
          if constexpr (kCps == 2) pair_sync(bar_id);  // the rows are there for both
        }
        if constexpr (KIND == kFmaBf16) {
          int pos4[kRowGroup];
          float best4[kRowGroup];
#pragma unroll
          for (int r = 0; r < kRowGroup; ++r) pos4[r] = pos[r];
          if (nr == 1)
            score_page<DI, HI, 1>(page, q_s, lane, si.blk, pos4, best4);
          else if (nr == 2)
            score_page<DI, HI, 2>(page, q_s, lane, si.blk, pos4, best4);
          else
            score_page<DI, HI, 4>(page, q_s, lane, si.blk, pos4, best4);  // rows >= nr unused
#pragma unroll
          for (int r = 0; r < kRowGroup; ++r) best[r] = best4[r];
        } else {
          const float* tscale = (KIND == kMmaFp8 && p.idx_scale)
              ? reinterpret_cast<const float*>(smem + S::kScale + (size_t)st * C::kScaleBytes)
              : nullptr;
          score_page_mma<DI, HI, KIND == kMmaFp8, kSwizzledPages<DI, HI, KIND>>(
              page, tscale, q_s, nr, lane, si.blk, pos, best, mt0, mt1);
        }
      } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) best[r] = -INFINITY;
      }
      if constexpr (kCps == 2) {
        // the second warp's maxima to the first (slots by row-group parity:
        // the first has read group g's before either passes group g + 1's
        // rendezvous)
        float* slot = red + (grp & 1) * kRowGroup;
        if (part == 1 && lane == 0) {
#pragma unroll
          for (int r = 0; r < kRowGroup; ++r) slot[r] = best[r];
        }
        pair_sync(bar_id);
        if (part == 0) {
#pragma unroll
          for (int r = 0; r < kRowGroup; ++r) best[r] = fmaxf(best[r], slot[r]);  // NaN never wins
        }
      }
      if (part == 0) {
#pragma unroll
        for (int r = 0; r < C::kRows; ++r)
          if (lane == r && r < nr)
            p.scores[(long long)(q0 + g0 + r) * p.score_stride + si.blk] = best[r];
      }
    }
    // the next bulk copy into q_s must follow this warp's own writes to it
    if (wrote_q) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

template <int DI, int HI, int KIND, int BUDGET = kStageBudget>
cudaError_t launch_cfg(const ScoreLaunch& p, cudaStream_t stream) {
  using C = ScoreCfg<DI, HI, KIND, BUDGET>;
  const size_t smem = ScoreSmem<DI, HI, KIND, BUDGET>::bytes(p.batch.num_reqs);
  auto kern = index_score_kernel<DI, HI, KIND, BUDGET>;
  CUtensorMap kmap;
  memset(&kmap, 0, sizeof(kmap));
  if constexpr (kSwizzledPages<DI, HI, KIND>) {
    // the pool as [P * 128 rows][DI keys]; boxes of 128 B x 128 rows;
    // row coordinates must fit an int
    const long long rows = (long long)p.batch.num_pages * kBlock;
    const bool ok = KIND == kMmaFp8
        ? encode_map_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.idx_k, DI, rows, DI, DI, kBlock)
        : encode_map_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.idx_k, DI, rows, DI * 2, 64,
                        kBlock);
    if (rows > 0x7fffffffll || !ok) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<device_sm_count(), C::kThreads, smem, stream>>>(p, kmap);
  return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_kind(const ScoreLaunch& p, cudaStream_t stream) {
  if constexpr (KIND == kMmaFp8) {  // the wider ring when the prefix fits beside it
    const int R = p.batch.num_reqs;
    if (p.index_heads == 1 && p.index_dim == 128 &&
        ScoreSmem<128, 1, KIND, kStageBudgetWide>::bytes(R) <= kMaxDynSmem)
      return launch_cfg<128, 1, KIND, kStageBudgetWide>(p, stream);
    if (p.index_heads == 2 && p.index_dim == 64 &&
        ScoreSmem<64, 2, KIND, kStageBudgetWide>::bytes(R) <= kMaxDynSmem)
      return launch_cfg<64, 2, KIND, kStageBudgetWide>(p, stream);
  }
  if (p.index_heads == 1 && p.index_dim == 128) return launch_cfg<128, 1, KIND>(p, stream);
  if (p.index_heads == 1 && p.index_dim == 64) return launch_cfg<64, 1, KIND>(p, stream);
  if (p.index_heads == 2 && p.index_dim == 64) return launch_cfg<64, 2, KIND>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_index_score(const ScoreLaunch& p, cudaStream_t stream) {
  if (p.idx_fp8) return launch_kind<kMmaFp8>(p, stream);
  // bf16 keys: one query row per request streams at the copy rate on FMAs;
  // several rows (speculative decode) multiply the FMA work per byte, and
  // the warp MMA scorer takes them
  if (MSA_SCORE_BF16_KIND == 1 || p.batch.max_q_len >= kMmaMinRows)
    return launch_kind<kMmaBf16Pair>(p, stream);
  return launch_kind<kFmaBf16>(p, stream);
}

}  // namespace msa
