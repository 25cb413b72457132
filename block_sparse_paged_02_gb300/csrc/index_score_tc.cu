// index_score_tc.cu -- step 1 for requests with many query rows (chunked
// prefill): the block score as the row-wise masked max of a dense
// contraction, on the 5th-generation tensor cores.
//
// Definition as in index_score.cu ("Optimise MiniMax-M3 decode index and
// top-k on gfx950", vLLM PR 54682, "Implementation breakdown" item 1): for
// each query row and 128-token block, the max over the block's visible
// tokens of idx_q[row] . idx_k[token].
//
// When a request brings >= kTcMinRows query rows, 128 rows x 128 tokens x Di
// is a real dense tile: D = Q_tile . K_block^T runs as tcgen05.mma
// (kind::f16, bf16 in, fp32 accumulate in TMEM), and the epilogue reduces
// each TMEM lane (= query row) to its causal-masked max.  Integer-valued
// index vectors keep every partial sum an exact fp32 integer, so the scores
// equal the CUDA-core kernel's and the oracle's bit for bit.
//
// CTA roles (persistent grid, one CTA per SM, work = the flat list of
// (request, 128-row tile, block) items split evenly across CTAs):
//   warp 0  TMA producer: the K block of each item, 128-byte-swizzled
//           tiles via cp.async.bulk.tensor into a 4-stage ring with
//           mbarrier completion;
//   warps 10-13 load each row tile's 128 index queries into TMEM (two
//           buffers): the A operand, reused by every block of the tile,
//           so the MMAs read only the K tile from shared memory (with both
//           operands there, M128 N128 MMAs plus the tile copies saturate
//           the shared-memory port);
//   warp 1  allocates 512 TMEM columns (two 128-column accumulators, two
//           query tiles); one thread of warp 1 and one of warp 14 issue the
//           MMAs of alternate items and commit (one issuing thread left the
//           tensor pipe idle while it waited and did its per-item
//           bookkeeping);
//   warps 2-9 epilogue: every item by all eight, the two warps of a TMEM
//           lane quarter taking 64 columns each (tcgen05.ld, masked max),
//           one of them storing the 32 rows' scores; each releases the
//           accumulator once it holds its columns in registers.
// Every wait is bounded; on expiry the kernel records MSA_DEV_TIMEOUT, stops
// issuing work and still frees its TMEM.
#include "tcgen05.cuh"

namespace msa {
namespace {

constexpr int kTcStages = 4;
// threads issuing the MMAs: with two, items alternate between them, so one
// issues while the other waits and does its per-item bookkeeping
#ifndef MSA_TC_ISSUERS
#define MSA_TC_ISSUERS 2
#endif
constexpr int kIssuers = MSA_TC_ISSUERS;
static_assert(kIssuers == 1 || kIssuers == 2, "one or two MMA issuers");
// warps: copies, MMA, 2 x 4 epilogue, 4 query loaders, the second MMA issuer
constexpr int kTcThreads = 32 * (13 + kIssuers);
constexpr int kIssuerWarp2 = 14;
constexpr int kTileRows = 128;
// epilogue: every item drained by all eight warps, two per TMEM lane quarter
// taking 64 columns each (1), or by one group of four on alternate items (0)
#ifndef MSA_TC_EPI_SPLIT
#define MSA_TC_EPI_SPLIT 1
#endif
constexpr bool kEpiSplit = MSA_TC_EPI_SPLIT != 0;
// 128-column fp32 accumulators in TMEM: with two issuers each owns one
// (three shared ones, safe with the in-order epilogue, measured slower)
constexpr int kAccBufs = kIssuers == 2 ? 2 : 3;
constexpr uint32_t kTmemA = 128 * kAccBufs;  // then two query tiles (A operands), 64 columns each
static_assert(kTcStages % kIssuers == 0 && kAccBufs % kIssuers == 0,
              "each ring stage and accumulator belongs to one issuer");
constexpr uint32_t kTmemCols = 512;

template <int DI>
struct TcCfg {
  static constexpr int kHalves = DI / 64;          // 128-byte swizzle atoms along K
  static constexpr int kTileBytes = kTileRows * DI * 2;
  static constexpr int kHalfBytes = kTileRows * 128;
  static constexpr int kKSteps = DI / 16;
  static constexpr int kACols = DI / 2;            // a query row in TMEM: bf16 pairs
  // smem: B ring, then barriers / bookkeeping, then request prefix
  static constexpr int kB = 0;
  static constexpr int kBars = kB + kTcStages * kTileBytes;
  // b_full / b_empty [kTcStages], a_full / a_empty [2], acc_full / acc_empty [kAccBufs]
  static constexpr int kNumBars = 2 * kTcStages + 4 + 2 * kAccBufs;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kRed = kMisc + 64;  // [2][128] floats: the split epilogue's hand-off
  static constexpr int kPrefix = kRed + 2 * kTileRows * 4;
  static_assert(8 + kTcStages <= 16, "misc area holds 16 ints");
  static size_t bytes(int num_reqs) { return 1024 + kPrefix + (size_t)(num_reqs + 1) * 4; }
};

// Max over 64 accumulator columns loaded into ra (0..31) and rb (32..63),
// columns c <= last only when MASKED.
template <bool MASKED>
__device__ __forceinline__ float row_max64(const uint32_t (&ra)[32], const uint32_t (&rb)[32],
                                           int last) {
  float g8[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) g8[x] = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (!MASKED || i <= last) g8[i & 7] = fmaxf(g8[i & 7], __uint_as_float(ra[i]));
    if (!MASKED || 32 + i <= last) g8[i & 7] = fmaxf(g8[i & 7], __uint_as_float(rb[i]));
  }
  return fmaxf(fmaxf(fmaxf(g8[0], g8[1]), fmaxf(g8[2], g8[3])),
               fmaxf(fmaxf(g8[4], g8[5]), fmaxf(g8[6], g8[7])));
}

// The two epilogue warps of one TMEM lane quarter (named barrier 1 + quarter,
// 64 threads): AND of a predicate over both, and a plain rendezvous.
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

using tc::commit;
using tc::fence_after;
using tc::fence_before;
using tc::tmem_ld32;

// Instruction descriptor of the score tile: M = 128 rows, N = 128 tokens.
constexpr uint32_t kIdesc = tc::idesc_bf16(128, 128, 0);

// Max over the 128 accumulator columns of this thread's lane at ta, columns
// c <= last only when MASKED (a block holding some row's own position);
// 32 columns per load with the next load in flight (warp-collective).
template <bool MASKED>
__device__ __forceinline__ float row_max128(uint32_t ta, int last) {
  uint32_t ra[32], rb[32];
  float g8[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) g8[x] = -INFINITY;
  tc::tmem_ld32_issue(ta, ra);
#pragma unroll 1
  for (int c = 0; c < 4; c += 2) {
    tc::tmem_wait_ld(ra);
    tc::tmem_ld32_issue(ta + 32 * (c + 1), rb);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (!MASKED || 32 * c + i <= last) g8[i & 7] = fmaxf(g8[i & 7], __uint_as_float(ra[i]));
    tc::tmem_wait_ld(rb);
    if (c + 2 < 4) tc::tmem_ld32_issue(ta + 32 * (c + 2), ra);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (!MASKED || 32 * c + 32 + i <= last) g8[i & 7] = fmaxf(g8[i & 7], __uint_as_float(rb[i]));
  }
  return fmaxf(fmaxf(fmaxf(g8[0], g8[1]), fmaxf(g8[2], g8[3])),
               fmaxf(fmaxf(g8[4], g8[5]), fmaxf(g8[6], g8[7])));
}

// ------------------------------------------------------------ work cursor

// Walks the (request, row tile, block) items of the tensor-core requests in
// order.  prefix[q] = items before request q (smem).
struct Cursor {
  int q, tile, blk, nb, ntiles, q0, qlen, ctx;

  __device__ void load_request(const msa_batch& b) {
    q0 = b.cu_seqlens_q[q];
    qlen = b.cu_seqlens_q[q + 1] - q0;
    ctx = b.context_lens[q];
    ntiles = (qlen + kTileRows - 1) / kTileRows;
  }
  __device__ int tile_blocks(int t) const {
    const int last_row = min(t * kTileRows + kTileRows - 1, qlen - 1);
    return (ctx + last_row) / kBlock + 1;
  }
  __device__ void seek(const msa_batch& b, const int* prefix, int R, int item) {
    int lo = 0, hi = R;  // largest q with prefix[q] <= item
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= item) lo = mid; else hi = mid;
    }
    while (lo < R - 1 && prefix[lo + 1] <= item) ++lo;
    q = lo;
    load_request(b);
    int rem = item - prefix[q];
    tile = 0;
    nb = tile_blocks(0);
    while (rem >= nb) {
      rem -= nb;
      ++tile;
      nb = tile_blocks(tile);
    }
    blk = rem;
  }
  __device__ void next(const msa_batch& b, const int* prefix, int R) {
    if (++blk < nb) return;
    blk = 0;
    if (++tile < ntiles) {
      nb = tile_blocks(tile);
      return;
    }
    do { ++q; } while (q < R - 1 && prefix[q + 1] == prefix[q]);  // skip item-less requests
    if (q >= R) return;
    load_request(b);
    tile = 0;
    nb = tile_blocks(0);
  }
};

// (15 warps: at most four share a sub-partition's 16K registers, so at most 128
// registers a thread; one CTA per SM)
template <int DI>
__global__ void __maxnreg__(128)
    index_score_tc_kernel(const ScoreLaunch p, const __grid_constant__ CUtensorMap kmap) {
  using C = TcCfg<DI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint64_t* b_full = bars;                   // [kTcStages]
  uint64_t* b_empty = bars + kTcStages;      // [kTcStages]
  uint64_t* a_full = bars + 2 * kTcStages;   // [2]
  uint64_t* a_empty = a_full + 2;            // [2]
  uint64_t* acc_full = a_empty + 2;          // [kAccBufs]
  uint64_t* acc_empty = acc_full + kAccBufs; // [kAccBufs]
  int* misc = reinterpret_cast<int*>(smem + C::kMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 4);
  int* stage_valid = misc + 8;  // [kTcStages], written by the producer before arming
  int* prefix = reinterpret_cast<int*>(smem + C::kPrefix);

  const msa_batch& b = p.batch;
  const int R = b.num_reqs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- setup (same request checks as the CUDA-core kernel)
  if (tid == 0) {
    misc[0] = !(b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows);
    misc[1] = 0;  // timeout seen
    misc[2] = 0;  // per-request status bits
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 4);  // the four query-loader warps
      mbar_init(&a_empty[i], kIssuers);  // each issuer commits once per row tile
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiSplit ? 8 : 4);  // the epilogue warps draining it
    }
    fence_barrier_init();
  }
  __syncthreads();
  for (int q = tid; q < R; q += blockDim.x) {
    int q0, ql, ctx, nb;
    const uint32_t bad = request_lengths(b, q, &q0, &ql, &ctx, &nb);
    if (ql < 0) misc[0] = 1;
    if (bad) atomicOr(reinterpret_cast<unsigned*>(&misc[2]), bad);
    int items = 0;
    if (!bad && ql >= kTcMinRows) {
      for (int t = 0; t * kTileRows < ql; ++t) {
        const int last_row = min(t * kTileRows + kTileRows - 1, ql - 1);
        items += (ctx + last_row) / kBlock + 1;
      }
    }
    prefix[q + 1] = items;
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  __syncthreads();
  const bool batch_ok = misc[0] == 0;
  // the same status bits as the CUDA-core kernel (which msa_decode does not
  // launch when every request has tensor-core rows)
  if (blockIdx.x == 0 && tid == 0 && p.report_status)
    atomicOr(p.status, batch_ok ? (unsigned)misc[2] : MSA_DEV_MALFORMED);
  if (batch_ok && warp == 0) {
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
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long total = batch_ok ? prefix[R] : 0;
  const int i0 = (int)(total * blockIdx.x / gridDim.x);
  const int i1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const int n_items = i1 - i0;

  if (n_items > 0) {
    if (warp == 0) {
      // ---------------- TMA producer warp: lanes look up 32 items at a time
      // (request, tile, block, page id); one elected lane then arms the
      // stages and issues the tile copies in order
      bool stop = false;
      for (int j0 = 0; j0 < n_items && !stop; j0 += 32) {
        int mpage = -1;
        if (j0 + lane < n_items) {
          Cursor cur;
          cur.seek(b, prefix, R, i0 + j0 + lane);
          mpage = b.block_table[(long long)cur.q * b.bt_stride + cur.blk];
        }
        const int cnt = min(32, n_items - j0);
        for (int jj = 0; jj < cnt; ++jj) {
          const int j = j0 + jj;
          const int page = __shfl_sync(0xffffffffu, mpage, jj);
          int ok = 1;
          if (lane == 0) {
            const int s = j % kTcStages;
            if (ok && j >= kTcStages && !mbar_wait(&b_empty[s], ((j / kTcStages) - 1) & 1))
              ok = 0;
            if (ok) {
              const bool valid = page >= 0 && page < b.num_pages;
              stage_valid[s] = valid;
              if (valid) {
                mbar_arrive_expect_tx(&b_full[s], C::kTileBytes);
                for (int h = 0; h < C::kHalves; ++h)
                  tma_load_2d(smem + C::kB + s * C::kTileBytes + h * C::kHalfBytes, &kmap, 64 * h,
                              page * kBlock, &b_full[s]);
              } else {
                mbar_arrive(&b_full[s]);  // nothing to load; the epilogue writes -inf
              }
            } else {
              misc[1] = 1;
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            stop = true;
            break;
          }
        }
      }
    } else if ((warp == 1 || (kIssuers == 2 && warp == kIssuerWarp2)) && lane == 0) {
      // ---------------- MMA issuer(s): D = Q_tile (TMEM) x K_block^T (shared).
      // Issuer ii takes items j = ii mod kIssuers: ring stages and
      // accumulators are then each used by one issuer, in order.  Both walk
      // every row tile: each waits for its queries and commits once to its
      // release (after its own MMAs of the tile, if any).
      const int ii = warp == 1 ? 0 : 1;
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      int a_key_q = -1, a_key_t = -1, a_seq = 0, abuf = 0;
      for (int j = 0; j < n_items; ++j) {
        if (cur.q != a_key_q || cur.tile != a_key_t) {  // the next row tile's queries
          abuf = a_seq & 1;
          if (!mbar_wait(&a_full[abuf], (a_seq >> 1) & 1)) {
            misc[1] = 1;
            break;
          }
          a_key_q = cur.q;
          a_key_t = cur.tile;
          ++a_seq;
        }
        if (j % kIssuers == ii) {
          const int s = j % kTcStages, buf = j % kAccBufs;
          if (j >= kAccBufs && !mbar_wait(&acc_empty[buf], ((j / kAccBufs) - 1) & 1)) {
            misc[1] = 1;
            break;
          }
          if (!mbar_wait(&b_full[s], (j / kTcStages) & 1)) {
            misc[1] = 1;
            break;
          }
          fence_after();
          if (stage_valid[s]) {
            const uint64_t bd = tc::desc_kmajor_sw128(smem_u32(smem + C::kB + s * C::kTileBytes));
            const uint32_t a_tm = tmem + kTmemA + abuf * 64u;
#pragma unroll
            for (int kk = 0; kk < C::kKSteps; ++kk) {
              const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
              tc::mma_ts(tmem + buf * 128u, a_tm + kk * 8, tc::desc_advance(bd, off), kIdesc,
                         kk > 0 ? 1u : 0u);
            }
          }
          commit(&b_empty[s]);
          commit(&acc_full[buf]);
        }
        Cursor nx = cur;
        nx.next(b, prefix, R);
        if (j == n_items - 1 || nx.q != cur.q || nx.tile != cur.tile) commit(&a_empty[abuf]);
        cur = nx;
      }
    } else if (warp >= 10 && warp < 14) {
      // ---------------- query loaders: each row tile of the CTA's items into
      // TMEM (lane = query row, column c = dims 2c, 2c+1), double-buffered;
      // rows past the request's end are zero
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      int a_seq = 0;
      for (int j = 0; j < n_items; ++j) {
        const bool new_tile = j == 0 || cur.blk == 0;  // a tile's items start at block 0
        if (new_tile) {
          const int ab = a_seq & 1;
          if (a_seq >= 2 && !__all_sync(0xffffffffu, mbar_wait(&a_empty[ab], ((a_seq >> 1) - 1) & 1))) {
            misc[1] = 1;
            break;
          }
          const int row = cur.tile * kTileRows + m;
          const uint4* src = reinterpret_cast<const uint4*>(p.idx_q + (long long)(cur.q0 + row) * DI);
          const bool have = row < cur.qlen;
#pragma unroll
          for (int c = 0; c < C::kACols / 16; ++c) {
            uint32_t w[16];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const uint4 v = have ? __ldg(src + 4 * c + x) : make_uint4(0u, 0u, 0u, 0u);
              w[4 * x] = v.x;
              w[4 * x + 1] = v.y;
              w[4 * x + 2] = v.z;
              w[4 * x + 3] = v.w;
            }
            tc::tmem_st16(tmem + lanes + kTmemA + ab * 64u + 16 * c, w);
          }
          tc::tmem_wait_st();
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[ab]);
          ++a_seq;
        }
        cur.next(b, prefix, R);
      }
    } else if (kEpiSplit && warp >= 2 && warp < 10) {
      // ---------------- epilogue: every item by all eight warps.  The two
      // warps of lane quarter w % 4 (= 32 query rows) take columns 0..63 and
      // 64..127 of the accumulator; the second hands its 32 maxima to the
      // first through shared memory, which stores the scores.  Both decide
      // together whether to go on (a timed-out wait ends both), so neither
      // is left at their barrier.
      const int half = (warp - 2) >> 2, quarter = warp & 3, bar_id = 1 + quarter;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      float* red = reinterpret_cast<float*>(smem + C::kRed);  // maxima of the second half
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      int page = b.block_table[(long long)cur.q * b.bt_stride + cur.blk];
      for (int j = 0; j < n_items; ++j) {
        const int buf = j % kAccBufs;
        Cursor nx = cur;
        int page_nx = 0;
        if (j + 1 < n_items) {
          nx.next(b, prefix, R);
          page_nx = b.block_table[(long long)nx.q * b.bt_stride + nx.blk];
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j / kAccBufs) & 1));
        if (!pair_and(ok, bar_id)) {
          misc[1] = 1;
          break;
        }
        fence_after();
        const int m = quarter * 32 + lane;
        const int row_in_req = cur.tile * kTileRows + m;
        const int pos = cur.ctx + row_in_req;
        const bool page_ok = page >= 0 && page < b.num_pages;
        const int last = pos - cur.blk * kBlock - 64 * half;  // visible columns of this half
        const uint32_t ta = tmem + lanes + buf * 128u + 64u * half;
        uint32_t ra[32], rb[32];
        tc::tmem_ld32_issue(ta, ra);
        tc::tmem_ld32_issue(ta + 32, rb);
        tc::tmem_wait_ld(ra);
        tc::tmem_wait_ld(rb);
        // the columns are in registers: the accumulator is free again
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        float best = __all_sync(0xffffffffu, last >= 63) ? row_max64<false>(ra, rb, last)
                                                         : row_max64<true>(ra, rb, last);
        if (half == 1) red[(j & 1) * kTileRows + m] = best;
        pair_sync(bar_id);
        if (half == 0) {
          best = fmaxf(best, red[(j & 1) * kTileRows + m]);
          if (row_in_req < cur.qlen && last >= 0)
            p.scores[(long long)(cur.q0 + row_in_req) * p.score_stride + cur.blk] =
                page_ok ? best : -INFINITY;
        }
        cur = nx;
        page = page_nx;
      }
    } else if (!kEpiSplit && warp >= 2 && warp < 10) {
      // ---------------- epilogue: two groups of four warps take alternate
      // items (accumulator j % 4); warp w reads TMEM lanes 32 (w % 4) .. +31
      // = 32 query rows, each reduced to its causal-masked max over the 128
      // token columns.  Blocks every row of the warp sees in full skip the
      // mask; the next item's page id is loaded while this one is reduced.
      const int grp = (warp - 2) >> 2, quarter = warp & 3;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      if (grp == 1 && n_items > 1) cur.next(b, prefix, R);
      int page = grp < n_items ? b.block_table[(long long)cur.q * b.bt_stride + cur.blk] : 0;
      for (int j = grp; j < n_items; j += 2) {
        const int buf = j % kAccBufs;
        Cursor nx = cur;
        int page_nx = 0;
        if (j + 2 < n_items) {
          nx.next(b, prefix, R);
          nx.next(b, prefix, R);
          page_nx = b.block_table[(long long)nx.q * b.bt_stride + nx.blk];
        }
        // warp-uniform decision: tcgen05.ld below needs the whole warp
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j / kAccBufs) & 1))) {
          misc[1] = 1;
          break;
        }
        fence_after();
        const int m = quarter * 32 + lane;
        const int row_in_req = cur.tile * kTileRows + m;
        const int pos = cur.ctx + row_in_req;
        const bool page_ok = page >= 0 && page < b.num_pages;
        const int last = pos - cur.blk * kBlock;  // visible columns: c <= last
        const uint32_t ta = tmem + lanes + buf * 128u;
        const float best = __all_sync(0xffffffffu, last >= kBlock - 1)
                               ? row_max128<false>(ta, last)
                               : row_max128<true>(ta, last);
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        if (row_in_req < cur.qlen && last >= 0)
          p.scores[(long long)(cur.q0 + row_in_req) * p.score_stride + cur.blk] =
              page_ok ? best : -INFINITY;
        cur = nx;
        page = page_nx;
      }
    }
  }
  fence_before();
  __syncthreads();
  if (misc[1] && tid == 0) atomicOr(p.status, MSA_DEV_TIMEOUT);
  if (warp == 1) {
    fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// 2-D bf16 tensor [rows, di] (row stride di*2 bytes), 64 x 128 boxes, 128-B swizzle
bool make_map(CUtensorMap* map, const void* base, long long rows, int di) {
  return encode_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, di, rows, (long long)di * 2, 64,
                       kTileRows);
}

template <int DI>
cudaError_t launch_tc(const ScoreLaunch& p, cudaStream_t stream) {
  CUtensorMap kmap;
  if (!make_map(&kmap, p.idx_k, (long long)p.batch.num_pages * kBlock, DI))
    return cudaErrorInvalidValue;
  const size_t smem = TcCfg<DI>::bytes(p.batch.num_reqs);
  auto kern = index_score_tc_kernel<DI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<device_sm_count(), kTcThreads, smem, stream>>>(p, kmap);
  return cudaGetLastError();
}

}  // namespace

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}
}  // namespace

bool tensor_maps_available() { return encode_fn() != nullptr; }

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, long long inner,
                   long long rows, long long row_stride_bytes, int box_inner, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_score_supported(int index_heads, int index_dim) {
  return index_heads == 1 && (index_dim == 64 || index_dim == 128) && tensor_maps_available();
}

cudaError_t launch_index_score_tc(const ScoreLaunch& p, cudaStream_t stream) {
  if (p.batch.num_rows == 0 || p.batch.num_reqs == 0) return cudaSuccess;
  if (p.index_dim == 128) return launch_tc<128>(p, stream);
  return launch_tc<64>(p, stream);
}

}  // namespace msa
