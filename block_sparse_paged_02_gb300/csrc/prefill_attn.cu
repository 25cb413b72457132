// prefill_attn.cu -- step 4 for the rows of prefill requests (a chunk of new
// tokens, every token a query row with its own causal top-k), block-major on
// the 5th-generation tensor cores.
//
// Definitions as in sparse_attn.cu: "Add ROCm AITER sparse paged attention
// for MiniMax-M3" (vLLM PR 47287), "Implementation breakdown" items 2-3 (a
// separate prefill attention path over the same page-16 sparse selection,
// k_scale / v_scale) and "Attention sinks for ROCm AITER sparse MLA" (vLLM PR
// 54404), "Features and motivation" / "Key source snippets" (sinks in the
// denominator, natural-log LSE, empty rows without NaN).
//
// Why block-major.  Each row of a prefill request picks its own k blocks;
// with independent index queries two rows share few of them (8 consecutive
// rows of the 2 x 2048-token chunk select ~102 distinct blocks out of 128
// picks), so a tile of rows against the union of their blocks would waste
// most of its MMA work, while a row-at-a-time kernel re-reads every block
// from L2 once per row and stalls on shared-memory operand reads.  Turned
// around, every block of a request is picked by ~k * q_len / nb rows (~130
// here).  So the top-k kernel appends each (row, slot) to its block's list;
// this file then
//   plan:      one CTA compacts the non-empty (request, block) lists into
//              items of 8-row chunks with prefixes of their chunks and of
//              their estimated costs;
//   attention: a persistent CTA per SM takes the chunks of an equal share
//              of the estimated cost; per
//              item it loads the block's K and V once (two 32 KB tensor
//              copies, 128-byte swizzle), per chunk it gathers the 8 rows'
//              queries (16 head slots each: M = 128) and computes
//                S = Q K^T     tcgen05.mma M128 N128 K128, fp32 in TMEM
//                P = exp2(S' - max)  per TMEM lane (= row, head), written
//                              back into TMEM as bf16 over S
//                O = P V       tcgen05.mma with A = P from TMEM, B = V
//                              (MN-major), fp32 in TMEM
//              and stores the chunk's per-(row, slot) partial: the sum of
//              p v (bf16) and the max and sum of p;
//   merge:     per row, the k partials are combined through their LSEs,
//              the sink joins the denominator, O and the natural-log LSE
//              are written.
// CTA roles in the attention kernel: warp 0 issues the tensor copies (its
// lanes and warp 15's gather the chunks' query rows), warp 1 allocates TMEM
// and one of its threads issues the S MMAs, one thread of warp 14 the P V
// MMAs, warps 2-5 and 6-9 are two softmax groups that take alternate
// chunks, warps 10-13 store every chunk's O.  TMEM (512 columns): three
// S / P buffers (chunk j in buffer j % 3, P over S) and one O, so S of
// chunk j + 3 waits only for P V of chunk j while two later chunks are in
// their softmax.  Every wait is bounded; on expiry the kernel records
// MSA_DEV_TIMEOUT, stops and still frees its TMEM.
#include <string.h>

#include "tcgen05.cuh"

namespace msa {
namespace {

constexpr int kChunkRows = 8;  // query rows per chunk (x 16 head slots = the MMA's M = 128)
constexpr int kHeadSlots = 16;
// warps: copies, S issue, two softmax groups of four, four O-epilogue
// warps, P V issue, query gathers
constexpr int kPaThreads = 512;
constexpr int kPvWarp = 14;
// A chunk's query rows are gathered by two warps, rows 0-3 by warp 0 and
// rows 4-7 by warp 15: each tensor copy costs its warp ~100 cycles to issue,
// and sixteen per chunk from one warp bounded the kernel.
constexpr int kGatherWarp2 = 15;
constexpr int kGatherRowsA = 4;
constexpr int kQStages = 3;
constexpr int kKvStages = 2;
constexpr int kHalf = 128 * 128;     // 128 rows x 128 B: one swizzle-atom column of a tile
constexpr int kTile = 2 * kHalf;     // a 128 x 128 bf16 tile
constexpr int kSmK = 0;
constexpr int kSmV = kSmK + kKvStages * kTile;
constexpr int kSmQ = kSmV + kKvStages * kTile;
constexpr int kSmBars = kSmQ + kQStages * kTile;
// kv_full[2] kv_empty[2] q_full[3] q_empty[3] s_full[3] sp_free[3] p_full[3] o_full o_empty
// kv_fill
constexpr int kSpBufs = 3;  // S / P buffers in TMEM
constexpr int kNumBars = 2 * kKvStages + 2 * kQStages + 3 * kSpBufs + 2 + 1;
constexpr int kSmMisc = kSmBars + kNumBars * 8;
constexpr int kPaSmem = kSmMisc + 64 + 1024;  // + slack for the 1024-byte alignment
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmS = 0;    // S / P [3]: 128 fp32 columns each (P: bf16 pairs in the first 64)
constexpr uint32_t kTmO = 384;  // O: 128 fp32 columns
constexpr uint32_t kIdescS = tc::idesc_bf16(128, 128, 0);
constexpr uint32_t kIdescO = tc::idesc_bf16(128, 128, 1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kPlanThreads = 1024;
// Estimated cost of the attention's work, to split it evenly across CTAs:
// per item its K / V load, per chunk its products and softmax, more for a
// block that holds some row's own position (the masked softmax).  Items of
// such blocks have few rows each, so a range of them loads many blocks: an
// equal split by chunks left the CTAs that got them ~20 % behind.
constexpr int kCostItem = 4;
constexpr int kCostChunk = 4;
constexpr int kCostDiagChunk = 6;
constexpr int kMergeThreads = 128;

// ------------------------------------------------------------------ plan

// Exclusive scan over the CTA; *total gets the sum.  scratch: 33 ints.
__device__ __forceinline__ int cta_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int t = lane < nw ? scratch[lane] : 0;
    int y = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += n;
    }
    if (lane < nw) scratch[lane] = y - t;
    if (lane == 31) scratch[32] = y;
  }
  __syncthreads();
  const int before = scratch[warp];
  *total = scratch[32];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PrefillLaunch p) {
  __shared__ int scratch[33];
  __shared__ int s_ok;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const msa_batch& b = p.batch;
  const int R = b.num_reqs, tid = threadIdx.x;
  const long long bt = b.bt_stride;

  // ---- routed requests (geometry only): q_len >= kPrefillMinRows and sane
  if (tid == 0) s_ok = b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows;
  bool mono = true;
  for (int q = tid; q < R; q += kPlanThreads) mono &= b.cu_seqlens_q[q + 1] >= b.cu_seqlens_q[q];
  if (!__syncthreads_and(mono)) s_ok = 0;
  __syncthreads();
  const bool ok = s_ok != 0;
  int n_req = 0, n_cand = 0;
  for (int base = 0; ok && base < R; base += kPlanThreads) {
    const int q = base + tid;
    int nb = 0, q0 = 0, ql = 0, ctx = 0;
    const bool routed_q =
        q < R && request_lengths(b, q, &q0, &ql, &ctx, &nb) == 0 && ql >= kPrefillMinRows;
    if (!routed_q) nb = 0;
    const int routed = nb > 0;
    int t_req, t_cand;
    const int at = n_req + cta_excl_scan(routed, scratch, &t_req);
    const int cand = n_cand + cta_excl_scan(nb, scratch, &t_cand);
    if (routed && at < p.max_routed_reqs) {
      p.plan_req_q[at] = q;
      p.plan_req_item[at] = cand;  // first candidate (request, block) of q
    }
    n_req += t_req;
    n_cand += t_cand;
  }
  if (n_req > p.max_routed_reqs || n_cand > p.max_items) {  // cannot happen by construction
    n_req = 0;
    n_cand = 0;
  }
  __syncthreads();  // the request list is visible to the whole CTA

  // wait for the top-k kernel's lists
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- candidates (request, block) -> non-empty items with a chunk prefix
  int n_items = 0, n_chunks = 0, n_cost = 0;
  for (int base = 0; base < n_cand; base += kPlanThreads) {
    const int c = base + tid;
    int q = 0, blk = 0, cnt = 0;
    long long cidx = 0;
    if (c < n_cand) {
      int lo = 0, hi = n_req;  // last routed request with first candidate <= c
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.plan_req_item[mid] <= c) lo = mid; else hi = mid;
      }
      q = p.plan_req_q[lo];
      blk = c - p.plan_req_item[lo];
      cidx = (long long)b.cu_seqlens_q[q] * bt / kPrefillMinRows + blk;
      // a list never holds more entries than the request has rows
      cnt = min(p.pf_counts[cidx], b.cu_seqlens_q[q + 1] - b.cu_seqlens_q[q]);
    }
    const int live = cnt > 0;
    const int chunks = (cnt + kChunkRows - 1) / kChunkRows;
    // a block reaching past the request's first row position is diagonal
    const bool diag = live && (long long)kBlock * blk + kBlock - 1 >= b.context_lens[q];
    const int cost = live ? kCostItem + chunks * (diag ? kCostDiagChunk : kCostChunk) : 0;
    int t_items, t_chunks, t_cost;
    const int at = n_items + cta_excl_scan(live, scratch, &t_items);
    const int first = n_chunks + cta_excl_scan(chunks, scratch, &t_chunks);
    const int first_cost = n_cost + cta_excl_scan(cost, scratch, &t_cost);
    if (live) {
      const int q0 = b.cu_seqlens_q[q], ql = b.cu_seqlens_q[q + 1] - q0;
      const int ctx = b.context_lens[q];
      p.item_rec[at] = make_int4((int)((long long)q0 * bt + (long long)blk * ql), cnt, ctx - q0, blk);
      p.item_kv[at] = make_int2(b.block_table[(long long)q * bt + blk],
                                min(kBlock, ctx + ql - kBlock * blk));
      p.item_chunk[at] = first;
      p.item_cost[at] = first_cost;
    }
    n_items += t_items;
    n_chunks += t_chunks;
    n_cost += t_cost;
  }
  if (tid == 0) {
    p.plan_hdr[0] = n_items;
    p.plan_hdr[1] = n_chunks;
    p.plan_hdr[2] = n_cost;
    p.item_chunk[n_items] = n_chunks;
    p.item_cost[n_items] = n_cost;
  }
}

// --------------------------------------------------------------- attention

// Walks the chunks of the plan in order: item `it`, chunk `ci` of it, with
// the item's record (list base, rows, position of row 0, block).
struct Cursor {
  int it, ci, n_items;
  int4 rec;

  __device__ __forceinline__ void seek(const PrefillLaunch& p, int chunk) {
    int lo = 0, hi = n_items;  // last item whose first chunk <= chunk (items are non-empty)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.item_chunk[mid] <= chunk) lo = mid; else hi = mid;
    }
    it = lo;
    rec = p.item_rec[it];
    ci = chunk - p.item_chunk[it];
  }
  __device__ __forceinline__ void next(const PrefillLaunch& p) {
    if (kChunkRows * (++ci) < rec.y) return;
    ci = 0;
    if (++it < n_items) rec = p.item_rec[it];
  }
  __device__ __forceinline__ int rows() const { return min(kChunkRows, rec.y - kChunkRows * ci); }
  __device__ __forceinline__ long long list_base() const { return (long long)rec.x + kChunkRows * ci; }
  __device__ __forceinline__ int blk() const { return rec.w; }
};

// p = 2^x of two logits at once on the multi-function unit: x rounded to
// f16 (x <= 0; the rounding moves p by at most ~2^-11 relative per unit of
// |x|, so a term's absolute error stays below 2e-4 of the row's largest),
// 2^x in f16, widened back for the sum and the bf16 pack
__device__ __forceinline__ void ex2_pair_f16(float x0, float x1, float& p0, float& p1) {
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(x1), "f"(x0));
  asm("ex2.approx.f16x2 %0, %0;" : "+r"(h));
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(p0), "=f"(p1)
      : "r"(h));
}

// max of three (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// all lanes wait; the result is the same on every lane
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
}

// ---- the softmax of one TMEM lane (128 logits from column sa), warp-collective

// 32 fp32 O columns of a lane as bf16, to dims chunks 0..3 of dst (chunk
// stride: the 16 heads)
__device__ __forceinline__ void store_o32(uint4* dst, const uint32_t (&r)[32]) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
    dst[kHeadSlots * x] =
        make_uint4(pack_bf16x2(__uint_as_float(r[8 * x]), __uint_as_float(r[8 * x + 1])),
                   pack_bf16x2(__uint_as_float(r[8 * x + 2]), __uint_as_float(r[8 * x + 3])),
                   pack_bf16x2(__uint_as_float(r[8 * x + 4]), __uint_as_float(r[8 * x + 5])),
                   pack_bf16x2(__uint_as_float(r[8 * x + 6]), __uint_as_float(r[8 * x + 7])));
}

// 32 fp32 columns as 16 bf16 pairs
__device__ __forceinline__ void pack32(const uint32_t (&r)[32], uint32_t* pk) {
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
}

// 16 packed pairs (32 O columns of a lane) to dims chunks 0..3 of dst
__device__ __forceinline__ void store_pk16(uint4* dst, const uint32_t* pk) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
    dst[kHeadSlots * x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
}

// The softmax of one TMEM lane: 128 logits from column sa, warp-collective.
// A block that holds some row's own position counts only its first `valid`
// tokens (MASKED); the masked code performs exactly the same arithmetic
// with the masked tokens' terms replaced by -inf / 0, so a row's result never
// depends on which path its warp took.

// running max over 32 raw scores (negated when NEG)
template <bool NEG, bool MASKED>
__device__ __forceinline__ float max32(const uint32_t (&r)[32], float acc, int base, int valid) {
  float g8[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) g8[x] = acc;
#pragma unroll
  for (int t = 0; t < 32; t += 2) {
    float v0 = NEG ? -__uint_as_float(r[t]) : __uint_as_float(r[t]);
    float v1 = NEG ? -__uint_as_float(r[t + 1]) : __uint_as_float(r[t + 1]);
    if (MASKED && base + t >= valid) v0 = -INFINITY;
    if (MASKED && base + t + 1 >= valid) v1 = -INFINITY;
    g8[(t >> 1) & 7] = fmax3(g8[(t >> 1) & 7], v0, v1);
  }
  return fmaxf(fmax3(g8[0], g8[1], g8[2]), fmax3(g8[3], g8[4], fmax3(g8[5], g8[6], g8[7])));
}

// max over the 128 raw scores (of their negations when NEG), loads in flight
template <bool NEG, bool MASKED>
__device__ __forceinline__ float row_max(uint32_t sa, int valid) {
  uint32_t ra[32], rb[32];
  float g = -INFINITY;
  tc::tmem_ld32_issue(sa, ra);
#pragma unroll 1
  for (int c = 0; c < 4; c += 2) {
    tc::tmem_wait_ld(ra);
    tc::tmem_ld32_issue(sa + 32 * (c + 1), rb);
    g = max32<NEG, MASKED>(ra, g, 32 * c, valid);
    tc::tmem_wait_ld(rb);
    if (c + 2 < 4) tc::tmem_ld32_issue(sa + 32 * (c + 2), ra);
    g = max32<NEG, MASKED>(rb, g, 32 * c + 32, valid);
  }
  return g;
}

// p = 2^(s * scale2 - m) of 32 columns, two at a time in f16 on the
// multi-function unit, packed as bf16 pairs into w; returns their sum
template <bool MASKED>
__device__ __forceinline__ float exp32(const uint32_t (&r)[32], float scale2, float m,
                                       uint32_t (&w)[16], int base, int valid) {
  float l8[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) l8[x] = 0.f;
#pragma unroll
  for (int t = 0; t < 32; t += 2) {
    float p0, p1;
    ex2_pair_f16(fmaf(__uint_as_float(r[t]), scale2, -m), fmaf(__uint_as_float(r[t + 1]), scale2, -m),
                 p0, p1);
    if (MASKED) {
      p0 = base + t < valid ? p0 : 0.f;
      p1 = base + t + 1 < valid ? p1 : 0.f;
    }
    l8[t & 7] += p0;
    l8[(t + 1) & 7] += p1;
    w[t >> 1] = pack_bf16x2(p0, p1);
  }
  return ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
}

// P of the 128 columns as bf16 pairs at pa (the 32 logits of load c give
// columns 16c .. 16c + 15; with pa = sa, P lands on columns already read),
// loads in flight; returns the sum of p
template <bool MASKED>
__device__ __forceinline__ float row_exp(uint32_t sa, uint32_t pa, float scale2, float m,
                                         int valid) {
  uint32_t ra[32], rb[32], w[16];
  float l = 0.f;
  tc::tmem_ld32_issue(sa, ra);
#pragma unroll 1
  for (int c = 0; c < 4; c += 2) {
    tc::tmem_wait_ld(ra);
    tc::tmem_ld32_issue(sa + 32 * (c + 1), rb);
    l += exp32<MASKED>(ra, scale2, m, w, 32 * c, valid);
    tc::tmem_st16(pa + 16 * c, w);
    tc::tmem_wait_ld(rb);
    if (c + 2 < 4) tc::tmem_ld32_issue(sa + 32 * (c + 2), ra);
    l += exp32<MASKED>(rb, scale2, m, w, 32 * c + 32, valid);
    tc::tmem_st16(pa + 16 * (c + 1), w);
  }
  return l;
}

// max of s * scale2 over one lane's logits = |scale2| * max(sign(scale2) * s)
template <bool MASKED>
__device__ __forceinline__ float row_max_scaled(uint32_t sa, float scale2, int valid) {
  return scale2 >= 0.f ? row_max<false, MASKED>(sa, valid) * scale2
                       : row_max<true, MASKED>(sa, valid) * -scale2;
}

// (16 warps: four share a sub-partition's 16K registers, so at most 128
// registers a thread; one CTA per SM by its shared memory)
template <bool SCALAR>
__global__ void __maxnreg__(128)
    prefill_attn_kernel(const PrefillLaunch p, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmBars);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = kv_full + kKvStages;
  uint64_t* q_full = kv_empty + kKvStages;
  uint64_t* q_empty = q_full + kQStages;
  uint64_t* s_full = q_empty + kQStages;   // [kSpBufs]
  uint64_t* sp_free = s_full + kSpBufs;    // [kSpBufs]
  uint64_t* p_full = sp_free + kSpBufs;    // [kSpBufs]
  uint64_t* o_full = p_full + kSpBufs;
  uint64_t* o_empty = o_full + 1;
  uint64_t* kv_fill = o_empty + 1;
  int* misc = reinterpret_cast<int*>(smem + kSmMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 4);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq = p.num_heads;

  if (tid == 0) {
    misc[1] = 0;  // timeout seen
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&q_full[s], 2);  // the two gathering warps
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < kSpBufs; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&sp_free[s], 1);
      mbar_init(&p_full[s], 4);  // the four warps of the chunk's softmax group
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, 4);  // the four O-epilogue warps
    mbar_init(kv_fill, 1);
    fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the plan (and the top-k lists)

  const int n_items = p.plan_hdr[0];
  // this CTA's chunks [c0, c1): an equal share of the estimated cost.  The
  // boundary at cost x is the number of chunks that start below x (chunk 0
  // of an item starts with the item's K / V load, chunk i > 0 at kCostItem +
  // i chunk costs into the item); the item holding x is found by all threads
  // at once.
  {
    const long long cost = p.plan_hdr[2];
    const long long x0 = cost * blockIdx.x / gridDim.x, x1 = cost * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0) {
      misc[8] = 0;
      misc[9] = p.plan_hdr[1];
    }
    __syncthreads();
    for (int it = tid; it < n_items; it += kPaThreads) {
      const int s0 = p.item_cost[it], s1 = p.item_cost[it + 1];
      const int f0 = p.item_chunk[it], n = p.item_chunk[it + 1] - f0;
      const int cw = (s1 - s0 - kCostItem) / max(n, 1);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const long long x = k ? x1 : x0;
        if (s0 < x && x <= s1) {
          const long long v = x - s0 - kCostItem;
          misc[8 + k] = f0 + (v <= 0 ? 1 : 1 + min(n - 1, (int)((v + cw - 1) / cw) - 1));
        }
      }
    }
    __syncthreads();
  }
  const int c0 = misc[8], c1 = misc[9];
  const int nj = c1 - c0;

  if (nj > 0) {
    if (warp == 0) {
      // ---------------- copies: K / V once per item, the chunk's query rows
      Cursor cur;
      cur.n_items = n_items;
      cur.seek(p, c0);
      int e_cur = lane < cur.rows() ? p.pf_lists[cur.list_base() + lane] : 0;
      int kv_seq = 0, fills = 0;
      for (int j = 0; j < nj; ++j) {
        Cursor nxt = cur;
        int e_nxt = 0;
        if (j + 1 < nj) {  // the next chunk's list entries, in flight during this one
          nxt.next(p);
          e_nxt = lane < nxt.rows() ? p.pf_lists[nxt.list_base() + lane] : 0;
        }
        if (j == 0 || cur.ci == 0) {
          const int kvs = kv_seq & 1;
          if (kv_seq >= 2 && !warp_wait(&kv_empty[kvs], ((kv_seq >> 1) - 1) & 1)) {
            misc[1] = 1;
            break;
          }
          const int2 kv = p.item_kv[cur.it];
          const int page = kv.x, ntok = kv.y;
          // a partial last block: the tokens past the request's end are not
          // data (never written); they are zeroed before P V reads them
          uint64_t* land = ntok < kBlock ? kv_fill : &kv_full[kvs];
          if (lane == 0) {
            mbar_arrive_expect_tx(land, 2 * kTile);
            uint8_t* kd = smem + kSmK + kvs * kTile;
            uint8_t* vd = smem + kSmV + kvs * kTile;
            for (int h = 0; h < 2; ++h) {
              tma_load_2d(kd + h * kHalf, &kmap, 64 * h, page * kBlock, land);
              tma_load_2d(vd + h * kHalf, &vmap, 64 * h, page * kBlock, land);
            }
          }
          if (ntok < kBlock) {
            if (!warp_wait(kv_fill, fills & 1)) {
              misc[1] = 1;
              break;
            }
            ++fills;
            uint4* vd = reinterpret_cast<uint4*>(smem + kSmV + kvs * kTile);
            // rows ntok..127 of both halves (each row 128 B; the swizzle
            // only permutes 16-byte chunks inside a row)
            for (int i = ntok * 8 + lane; i < kBlock * 8; i += 32) {
              vd[i] = make_uint4(0u, 0u, 0u, 0u);
              vd[kHalf / 16 + i] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // generic writes before the MMA's async reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&kv_full[kvs]);
          }
          ++kv_seq;
        }
        const int qs = j % kQStages;
        if (j >= kQStages && !warp_wait(&q_empty[qs], ((j / kQStages) - 1) & 1)) {
          misc[1] = 1;
          break;
        }
        const int n = cur.rows();
        const int na = min(n, kGatherRowsA);  // this warp's rows 0 .. na - 1
        if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], (uint32_t)(na * hq * 256));
        __syncwarp();
        if (lane < na) {
          // (an entry outside the batch, impossible from the top-k kernel,
          // reads row 0 and is never written back)
          const int er = e_cur >> 8;
          const int r = er < p.batch.num_rows ? er : 0;
          uint8_t* qd = smem + kSmQ + qs * kTile + lane * (kHeadSlots * 128);
          tma_load_2d(qd, &qmap, 0, r * hq, &q_full[qs]);
          tma_load_2d(qd + kHalf, &qmap, 64, r * hq, &q_full[qs]);
        }
        cur = nxt;
        e_cur = e_nxt;
      }
    } else if (warp == kGatherWarp2) {
      // ---------------- query rows kGatherRowsA .. 7 of every chunk
      Cursor cur;
      cur.n_items = n_items;
      cur.seek(p, c0);
      const int slot = kGatherRowsA + lane;
      int e_cur = slot < cur.rows() ? p.pf_lists[cur.list_base() + slot] : 0;
      for (int j = 0; j < nj; ++j) {
        Cursor nxt = cur;
        int e_nxt = 0;
        if (j + 1 < nj) {
          nxt.next(p);
          e_nxt = slot < nxt.rows() ? p.pf_lists[nxt.list_base() + slot] : 0;
        }
        const int qs = j % kQStages;
        if (j >= kQStages && !warp_wait(&q_empty[qs], ((j / kQStages) - 1) & 1)) {
          misc[1] = 1;
          break;
        }
        const int nb = max(cur.rows() - kGatherRowsA, 0);
        if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], (uint32_t)(nb * hq * 256));
        __syncwarp();
        if (lane < nb) {
          const int er = e_cur >> 8;
          const int r = er < p.batch.num_rows ? er : 0;
          uint8_t* qd = smem + kSmQ + qs * kTile + slot * (kHeadSlots * 128);
          tma_load_2d(qd, &qmap, 0, r * hq, &q_full[qs]);
          tma_load_2d(qd + kHalf, &qmap, 64, r * hq, &q_full[qs]);
        }
        cur = nxt;
        e_cur = e_nxt;
      }
    } else if (warp == 1) {
      // ---------------- S = Q K^T issue (one thread).  S / P of chunk j live
      // in TMEM columns 128 (j % 3); S(j) may overwrite its buffer once P V
      // of chunk j - 3 has completed (sp_free).  (One thread issuing both
      // products was the kernel's bound: ~100 cycles per MMA instruction.)
      if (lane == 0) {
        Cursor cur;
        cur.n_items = n_items;
        cur.seek(p, c0);
        int kv_seq = 0, cur_kvs = 0;
        bool ok = true;
        for (int j = 0; j < nj; ++j) {
          const int buf = j % kSpBufs, qs = j % kQStages;
          if (j == 0 || cur.ci == 0) {
            cur_kvs = kv_seq & 1;
            ok = mbar_wait(&kv_full[cur_kvs], (kv_seq >> 1) & 1);
            ++kv_seq;
          }
          ok = ok && mbar_wait(&q_full[qs], (j / kQStages) & 1);
          ok = ok && (j < kSpBufs || mbar_wait(&sp_free[buf], ((j / kSpBufs) - 1) & 1));
          if (!ok) break;
          tc::fence_after();
          const uint64_t qd = tc::desc_kmajor_sw128(smem_u32(smem + kSmQ + qs * kTile));
          const uint64_t kd = tc::desc_kmajor_sw128(smem_u32(smem + kSmK + cur_kvs * kTile));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            tc::mma_ss(tmem + kTmS + buf * 128, tc::desc_advance(qd, off),
                       tc::desc_advance(kd, off), kIdescS, kk > 0 ? 1u : 0u);
          }
          tc::commit(&q_empty[qs]);
          tc::commit(&s_full[buf]);
          cur.next(p);
        }
        if (!ok) misc[1] = 1;
      }
    } else if (warp == kPvWarp) {
      // ---------------- O = P V issue (one thread): P of chunk i from TMEM
      // columns 128 (i % 3), O into kTmO once the epilogue has read O of
      // chunk i - 1 (o_empty); the S / P buffer is released to the S issuer
      // (sp_free) and O handed to the epilogue (o_full) by commits.
      // After the last chunk of an item its K / V stage is released (its
      // scores were read before that chunk's P was written).
      if (lane == 0) {
        Cursor cur;
        cur.n_items = n_items;
        cur.seek(p, c0);
        int kv_seq = 0, cur_kvs = 0;
        bool ok = true;
        for (int i = 0; i < nj; ++i) {
          const int pb = i % kSpBufs;
          if (i == 0 || cur.ci == 0) {
            cur_kvs = kv_seq & 1;
            ok = mbar_wait(&kv_full[cur_kvs], (kv_seq >> 1) & 1);
            ++kv_seq;
          }
          ok = ok && mbar_wait(&p_full[pb], (i / kSpBufs) & 1) &&
               (i < 1 || mbar_wait(o_empty, (i - 1) & 1));
          if (!ok) break;
          tc::fence_after();
          const uint64_t vd = tc::desc_mnmajor_sw128(smem_u32(smem + kSmV + cur_kvs * kTile), kHalf);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_ts(tmem + kTmO, tmem + kTmS + pb * 128 + kk * 8,
                       tc::desc_advance(vd, kk * 2048), kIdescO, kk > 0 ? 1u : 0u);
          tc::commit(&sp_free[pb]);
          tc::commit(o_full);
          const int before = cur.it;
          cur.next(p);
          if (i == nj - 1 || cur.it != before) tc::commit(&kv_empty[cur_kvs]);
        }
        if (!ok) misc[1] = 1;
      }
    } else if (warp >= 2 && warp < 10) {
      // ---------------- softmax, chunks j = grp, grp + 2, ...
      // Thread = TMEM lane = (row slot, head) of the chunk; 128 logits each.
      // The max and the sum run on 8 independent accumulators (the warp has
      // little else to overlap with); rows whose block is entirely visible
      // skip the per-token mask.  The group stores the chunk's (max, sum)
      // and goes on; its O is drained by the epilogue warps.
      const int grp = (warp - 2) >> 2, quarter = warp & 3;
      const int m = quarter * 32 + lane, slot = m >> 4, head = m & 15;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      float scale2 = p.softmax_scale * kLog2e;
      if constexpr (SCALAR) scale2 *= __ldg(p.k_scale);
      Cursor cur;
      cur.n_items = n_items;
      cur.seek(p, c0);
      if (grp == 1 && nj > 1) cur.next(p);
      int e = (slot < cur.rows()) ? p.pf_lists[cur.list_base() + slot] : 0;
      for (int j = grp; j < nj; j += 2) {
        const int buf = j % kSpBufs;
        const int r = e >> 8, si = e & 255;
        const bool live = slot < cur.rows() && head < hq && r < p.batch.num_rows && si < p.topk;
        const int pos = r + cur.rec.z;
        const int valid = live ? max(1, min(kBlock, pos + 1 - kBlock * cur.blk())) : 0;
        const bool whole = __all_sync(0xffffffffu, valid == kBlock || !live);
        // the next chunk of this group: its list entry is in flight meanwhile
        Cursor nx = cur;
        int e_nx = 0;
        if (j + 2 < nj) {
          nx.next(p);
          nx.next(p);
          e_nx = (slot < nx.rows()) ? p.pf_lists[nx.list_base() + slot] : 0;
        }
        if (!warp_wait(&s_full[buf], (j / kSpBufs) & 1)) {
          misc[1] = 1;
          break;
        }
        tc::fence_after();
        const uint32_t sa = tmem + lanes + kTmS + buf * 128;
        // Two passes over the 128 logits, 32 columns per load with the next
        // load in flight: the max, then p = 2^(x - max) written back over S
        // as bf16 and summed.  Whole blocks (every lane of the warp sees all
        // 128 tokens) take the unrolled path; a block holding some row's own
        // position takes a compact masked loop.
        float m = whole ? row_max_scaled<false>(sa, scale2, kBlock)
                        : row_max_scaled<true>(sa, scale2, valid);
        if (!live) m = 0.f;
        const float l = whole ? row_exp<false>(sa, sa, scale2, m, kBlock)
                              : row_exp<true>(sa, sa, scale2, m, valid);
        tc::tmem_wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[buf]);
        if (live) p.part_ml[((long long)r * p.topk + si) * kHeadSlots + head] = make_float2(m, l);
        cur = nx;
        e = e_nx;
      }
    } else if (warp >= 10 && warp < 14) {
      // ---------------- O epilogue, every chunk in order: warp w drains TMEM
      // lanes 32 (w % 4) .. +31 of the chunk's O.  Partial per (row, slot):
      // the unnormalised sum of p v as bf16 in [16 dim chunks][16 heads][8
      // dims], so the 16 head lanes of a slot store 256 contiguous bytes.
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane, slot = m >> 4, head = m & 15;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      Cursor cur;
      cur.n_items = n_items;
      cur.seek(p, c0);
      int e = (slot < cur.rows()) ? p.pf_lists[cur.list_base() + slot] : 0;
      for (int j = 0; j < nj; ++j) {
        const int r = e >> 8, si = e & 255;
        const bool live = slot < cur.rows() && head < hq && r < p.batch.num_rows && si < p.topk;
        Cursor nx = cur;
        int e_nx = 0;
        if (j + 1 < nj) {
          nx.next(p);
          e_nx = (slot < nx.rows()) ? p.pf_lists[nx.list_base() + slot] : 0;
        }
        if (!warp_wait(o_full, j & 1)) {
          misc[1] = 1;
          break;
        }
        tc::fence_after();
        uint4* dst = reinterpret_cast<uint4*>(
                         p.part_o + ((long long)r * p.topk + si) * kHeadSlots * kHeadDim) +
                     head;
        {
          // O leaves tensor memory in two rounds of two loads in flight (the
          // first 64 columns packed to bf16 meanwhile), and the buffer is
          // released before any store: P V of the next chunk waits on it
          const uint32_t oa = tmem + lanes + kTmO;
          uint32_t ra[32], rb[32], pk[32];
          tc::tmem_ld32_issue(oa, ra);
          tc::tmem_ld32_issue(oa + 32, rb);
          tc::tmem_wait_ld(ra);
          tc::tmem_wait_ld(rb);
          pack32(ra, pk);
          pack32(rb, pk + 16);
          tc::tmem_ld32_issue(oa + 64, ra);
          tc::tmem_ld32_issue(oa + 96, rb);
          tc::tmem_wait_ld(ra);
          tc::tmem_wait_ld(rb);
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty);
          if (live) {
            store_pk16(dst, pk);
            store_pk16(dst + kHeadSlots * 4, pk + 16);
            store_o32(dst + kHeadSlots * 4 * 2, ra);
            store_o32(dst + kHeadSlots * 4 * 3, rb);
          }
        }
        cur = nx;
        e = e_nx;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (misc[1] && tid == 0) atomicOr(p.status, MSA_DEV_TIMEOUT);
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ merge

// One CTA per row: thread t owns head t % 16 and the 8-dim chunks t / 16
// and t / 16 + 8, so that a warp reads 512 contiguous bytes of a partial
// ([16 dim chunks][16 heads][8 dims]) per load.  Rows not routed to the
// prefill path leave at once, or, when no decode attention runs, are
// written as empty rows.
template <bool SCALAR>
__global__ void __launch_bounds__(kMergeThreads) prefill_merge_kernel(const PrefillLaunch p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x, tid = threadIdx.x;
  const int head = tid & 15, ca = tid >> 4;  // chunks ca and ca + 8
  float sink2 = -INFINITY, vs = 1.f;
  if (p.sinks && head < p.num_heads) sink2 = __ldg(p.sinks + head) * kLog2e;
  if constexpr (SCALAR) vs = __ldg(p.v_scale);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a row left to the decode attention; with none launched (every request
  // known to be a prefill request) such a row is poisoned: written here as
  // an empty row (O = 0, LSE = sink or -inf)
  const bool routed = p.route[r] != 0;
  if (!routed && !p.finish_unrouted) return;
  // the row's selections (ascending blocks, then -1; topk <= kMergeThreads):
  // one partial per selected block
  const bool has = routed && tid < p.topk && p.topk_idx[(long long)r * p.topk + tid] >= 0;
  const int nsel = __syncthreads_count(has);
  if (head >= p.num_heads) return;
  const long long pbase = (long long)r * p.topk;
  // one pass over the partials, four at a time with all their loads in
  // flight together; the running max moves once per group of four
  float M = sink2;
  float L = p.sinks ? 1.f : 0.f;  // the sink's term, relative to M
  float acc[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) acc[x] = 0.f;
  for (int i0 = 0; i0 < nsel; i0 += 4) {
    float2 ml[4];
    uint4 va[4], vb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ml[u] = make_float2(-INFINITY, 0.f);
      va[u] = vb[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i0 + u < nsel) {
        const long long slot = pbase + i0 + u;
        ml[u] = p.part_ml[slot * kHeadSlots + head];
        const uint4* src = reinterpret_cast<const uint4*>(p.part_o + slot * kHeadSlots * kHeadDim) +
                           ca * kHeadSlots + head;
        va[u] = src[0];
        vb[u] = src[8 * kHeadSlots];
      }
    }
    float mb = M;
#pragma unroll
    for (int u = 0; u < 4; ++u) mb = fmaxf(mb, ml[u].x);
    if (mb > M) {  // rescale what was gathered so far to the new max
      const float f = M == -INFINITY ? 0.f : exp2f(M - mb);
      L *= f;
#pragma unroll
      for (int x = 0; x < 16; ++x) acc[x] *= f;
      M = mb;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (ml[u].x == -INFINITY) continue;  // (a missing or empty partial adds nothing)
      const float w = exp2f(ml[u].x - M);
      L += w * ml[u].y;
      const uint32_t uu[8] = {va[u].x, va[u].y, va[u].z, va[u].w, vb[u].x, vb[u].y, vb[u].z, vb[u].w};
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        acc[2 * x] += w * bf16lo(uu[x]);
        acc[2 * x + 1] += w * bf16hi(uu[x]);
      }
    }
  }
  const float inv = L > 0.f ? vs / L : 0.f;
  uint32_t packed[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) packed[x] = pack_bf16x2(acc[2 * x] * inv, acc[2 * x + 1] * inv);
  uint4* o = reinterpret_cast<uint4*>(p.out + ((long long)r * p.num_heads + head) * kHeadDim);
  o[ca] = make_uint4(packed[0], packed[1], packed[2], packed[3]);      // dims 8 ca ..
  o[ca + 8] = make_uint4(packed[4], packed[5], packed[6], packed[7]);  // dims 64 + 8 ca ..
  if (ca == 0)
    p.lse[(long long)r * p.num_heads + head] =
        (M == -INFINITY || L <= 0.f) ? -INFINITY : (M + log2f(L)) * kLn2;
}

cudaError_t launch_pdl(const void* kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

template <bool SCALAR>
cudaError_t launch_all(const PrefillLaunch& p, cudaStream_t stream) {
  CUtensorMap qmap, kmap, vmap;
  memset(&qmap, 0, sizeof(qmap));
  if (!encode_map_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, kHeadDim,
                     (long long)p.batch.num_rows * p.num_heads, kHeadDim * 2, 64, p.num_heads) ||
      !encode_map_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, kHeadDim,
                     (long long)p.batch.num_pages * kBlock, kHeadDim * 2, 64, kBlock) ||
      !encode_map_2d(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, kHeadDim,
                     (long long)p.batch.num_pages * kBlock, kHeadDim * 2, 64, kBlock))
    return cudaErrorInvalidValue;
  PrefillLaunch pp = p;
  void* plan_args[] = {&pp};
  cudaError_t e = launch_pdl(reinterpret_cast<const void*>(prefill_plan_kernel), dim3(1),
                             dim3(kPlanThreads), 0, stream, plan_args);
  if (e != cudaSuccess) return e;
  auto attn = prefill_attn_kernel<SCALAR>;
  e = cudaFuncSetAttribute(attn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPaSmem);
  if (e != cudaSuccess) return e;
  void* attn_args[] = {&pp, &qmap, &kmap, &vmap};
  e = launch_pdl(reinterpret_cast<const void*>(attn), dim3(device_sm_count()), dim3(kPaThreads),
                 kPaSmem, stream, attn_args);
  if (e != cudaSuccess) return e;
  // the merge as a plain launch: programmatic, its 4096 CTAs waiting on the
  // attention measured 14 us slower per chunked-prefill step
  void* merge_args[] = {&pp};
  return cudaLaunchKernel(reinterpret_cast<const void*>(prefill_merge_kernel<SCALAR>),
                          dim3(p.batch.num_rows), dim3(kMergeThreads), merge_args, 0, stream);
}

}  // namespace

bool prefill_attn_available() { return tensor_maps_available(); }

cudaError_t launch_prefill_attn(const PrefillLaunch& p, cudaStream_t stream) {
  if (p.batch.num_rows == 0 || p.batch.num_reqs == 0) return cudaSuccess;
  if (p.k_scale) return launch_all<true>(p, stream);
  return launch_all<false>(p, stream);
}

}  // namespace msa
