// index_score_tc.cu -- step 1 for requests with many query rows (chunked
// prefill): the block score as the row-wise masked max of a dense
// contraction, on the 5th-generation tensor cores.
//
// Definition as in index_score.cu ("Optimise MiniMax-M3 decode index and
// top-k on gfx950", vLLM PR 54682, "Implementation breakdown" item 1): for
// each query row and 128-token block, the max over the block's visible
// tokens of idx_q[row] . idx_k[token].
//
// When a request brings >= kTcMinRows query rows, 128 rows x 256 tokens x Di
// is a real dense tile: D = Q_tile . [K_block0; K_block1]^T runs as
// tcgen05.mma (kind::f16, M128 N256, bf16 in, fp32 accumulate in TMEM), and
// the epilogue reduces each TMEM lane (= query row) to its causal-masked
// max per block.  Integer-valued index vectors keep every partial sum an
// exact fp32 integer, so the scores equal the CUDA-core kernel's and the
// oracle's bit for bit.
//
// Work = the flat list of (request, 128-row tile, pair of consecutive
// blocks) items, split evenly across a persistent grid of one CTA per SM.
// Two blocks per MMA: with one block per MMA the issuing thread spent ~100
// cycles on each M128 N128 K16 tcgen05.mma, a step that keeps the tensor
// pipe busy for only 64, so the pipe waited on the issue; an M128 N256 step
// carries 128 cycles of work per instruction.
// CTA roles:
//   warp 0  TMA producer: the two K blocks of each item, 128-byte-swizzled
//           tiles via cp.async.bulk.tensor into a 4-slot ring, mbarrier
//           completion; a slot holds one 64-dim swizzle atom of a pair
//           (block 0's 128 rows, then block 1's: one 256-row operand), so
//           a Di = 128 item takes two slots, and the first is refilled as
//           soon as the MMAs of its 64 dims are done;
//   warps 10-13 store each row tile's 128 index queries into shared memory
//           in the same swizzled layout (two buffers): the A operand, reused
//           by every pair of the tile;
//   warp 1  allocates the 512 TMEM columns (two 256-column accumulators);
//           one thread of warp 1 and one of warp 14 issue the MMAs of
//           alternate items and commit, each owning one ring stage in two
//           and one accumulator;
//   warps 2-9 epilogue: warps 2-5 reduce block 0 of every item, warps 6-9
//           block 1, each warp the 32 query rows of its TMEM lane quarter
//           (tcgen05.ld, masked max) and storing their scores.
// Every wait is bounded; on expiry the kernel records MSA_DEV_TIMEOUT, stops
// issuing work and still frees its TMEM.
#include "tcgen05.cuh"

namespace msa {
namespace {

// two threads issue the MMAs: items alternate between them, so one issues
// while the other waits and does its per-item bookkeeping
constexpr int kIssuers = 2;
// warps: copies, MMA, 2 x 4 epilogue, 4 query loaders, the second MMA issuer
constexpr int kTcThreads = 32 * 15;
constexpr int kIssuerWarp2 = 14;
constexpr int kTileRows = 128;
constexpr int kPairCols = 2 * kBlock;  // accumulator columns of one item
constexpr int kAccBufs = 2;            // one per issuer
constexpr uint32_t kTmemCols = kAccBufs * kPairCols;

template <int DI>
struct TcCfg {
  static constexpr int kHalves = DI / 64;          // 128-byte swizzle atoms along K
  static constexpr int kTileBytes = kTileRows * DI * 2;  // one block (or the query tile)
  static constexpr int kHalfBytes = kTileRows * 128;     // one atom column of 128 rows
  static constexpr int kStageBytes = 2 * kHalfBytes;     // a ring slot: one atom column of the pair's 256 rows
  static constexpr int kStages = 4;
  static constexpr int kAtomSteps = 4;                   // K16 steps per atom column
  // smem: B ring, A (query) buffers, then barriers / bookkeeping, then request prefix
  static constexpr int kB = 0;
  static constexpr int kA = kB + kStages * kStageBytes;
  static constexpr int kBars = kA + 2 * kTileBytes;
  // b_full / b_empty [kStages], a_full / a_empty [2], acc_full / acc_empty [kAccBufs]
  static constexpr int kNumBars = 2 * kStages + 4 + 2 * kAccBufs;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kPrefix = kMisc + 64;
  static_assert(8 + kStages <= 16, "misc area holds 16 ints");
  // slot u = item * kHalves + h: with items alternating between the
  // issuers, each slot is used by one issuer, in order
  static_assert(kStages % (kIssuers * kHalves) == 0, "each ring slot belongs to one issuer");
  static size_t bytes(int num_reqs) { return 1024 + kPrefix + (size_t)(num_reqs + 1) * 4; }
};

using tc::commit;
using tc::fence_after;
using tc::fence_before;

// Instruction descriptors of the score tile: M = 128 rows, N = 256 tokens
// (a pair), or 128 when the tile's last item holds a single block.
constexpr uint32_t kIdescPair = tc::idesc_bf16(128, kPairCols, 0);
constexpr uint32_t kIdescOne = tc::idesc_bf16(128, kBlock, 0);

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

// Walks the (request, row tile, block pair) items of the tensor-core
// requests in order.  prefix[q] = items before request q (smem).
struct Cursor {
  int q, tile, pr, np, nbk, ntiles, q0, qlen, ctx;

  __device__ void load_request(const msa_batch& b) {
    q0 = b.cu_seqlens_q[q];
    qlen = b.cu_seqlens_q[q + 1] - q0;
    ctx = b.context_lens[q];
    ntiles = (qlen + kTileRows - 1) / kTileRows;
  }
  __device__ void set_tile(int t) {
    tile = t;
    const int last_row = min(t * kTileRows + kTileRows - 1, qlen - 1);
    nbk = (ctx + last_row) / kBlock + 1;  // blocks the tile's last row sees
    np = (nbk + 1) >> 1;
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
    set_tile(0);
    while (rem >= np) {
      rem -= np;
      set_tile(tile + 1);
    }
    pr = rem;
  }
  __device__ void next(const msa_batch& b, const int* prefix, int R) {
    if (++pr < np) return;
    pr = 0;
    if (tile + 1 < ntiles) {
      set_tile(tile + 1);
      return;
    }
    do { ++q; } while (q < R - 1 && prefix[q + 1] == prefix[q]);  // skip item-less requests
    if (q >= R) return;
    load_request(b);
    set_tile(0);
  }
  // page of block e (0 or 1) of the current pair; -2 when the pair has no such block
  __device__ int page(const msa_batch& b, int e) const {
    const int blk = 2 * pr + e;
    return blk < nbk ? b.block_table[(long long)q * b.bt_stride + blk] : -2;
  }
};

// (15 warps: at most four share a sub-partition's 16K registers, so at most 128
// registers a thread; one CTA per SM)
template <int DI>
__global__ void __maxnreg__(128)
    index_score_tc_kernel(const ScoreLaunch p, const __grid_constant__ CUtensorMap kmap) {
  using C = TcCfg<DI>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint64_t* b_full = bars;                   // [S]
  uint64_t* b_empty = bars + S;              // [S]
  uint64_t* a_full = bars + 2 * S;           // [2]
  uint64_t* a_empty = a_full + 2;            // [2]
  uint64_t* acc_full = a_empty + 2;          // [kAccBufs]
  uint64_t* acc_empty = acc_full + kAccBufs; // [kAccBufs]
  int* misc = reinterpret_cast<int*>(smem + C::kMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 4);
  // [S] bit e = block e loaded, bit 2 = the pair has a block 1; written by
  // the producer before arming the slot
  int* stage_valid = misc + 8;
  int* prefix = reinterpret_cast<int*>(smem + C::kPrefix);

  const msa_batch& b = p.batch;
  const int R = b.num_reqs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- setup (same request checks as the CUDA-core kernel)
  if (tid == 0) {
    misc[0] = !(b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows);
    misc[1] = 0;  // timeout seen
    misc[2] = 0;  // per-request status bits
    for (int s = 0; s < S; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 4);          // the four query-loader warps
      mbar_init(&a_empty[i], kIssuers);  // each issuer commits once per row tile
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 8);  // the eight epilogue warps
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
        items += ((ctx + last_row) / kBlock + 2) >> 1;
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
      // (request, tile, pair, two page ids); one elected lane then arms the
      // stages and issues the tile copies in order
      bool stop = false;
      for (int j0 = 0; j0 < n_items && !stop; j0 += 32) {
        int mpage0 = -1, mpage1 = -2;
        if (j0 + lane < n_items) {
          Cursor cur;
          cur.seek(b, prefix, R, i0 + j0 + lane);
          mpage0 = cur.page(b, 0);
          mpage1 = cur.page(b, 1);
        }
        const int cnt = min(32, n_items - j0);
        for (int jj = 0; jj < cnt; ++jj) {
          const int j = j0 + jj;
          const int page0 = __shfl_sync(0xffffffffu, mpage0, jj);
          const int page1 = __shfl_sync(0xffffffffu, mpage1, jj);
          int ok = 1;
          if (lane == 0) {
            const bool v0 = page0 >= 0 && page0 < b.num_pages;
            const bool v1 = page1 >= 0 && page1 < b.num_pages;
            for (int h = 0; h < C::kHalves && ok; ++h) {
              const int u = j * C::kHalves + h, s = u % S;
              if (u >= S && !mbar_wait(&b_empty[s], ((u / S) - 1) & 1)) {
                ok = 0;
                misc[1] = 1;
                break;
              }
              stage_valid[s] = (v0 ? 1 : 0) | (v1 ? 2 : 0) | (page1 != -2 ? 4 : 0);
              if (v0 || v1) {
                uint8_t* st = smem + C::kB + s * C::kStageBytes;
                mbar_arrive_expect_tx(&b_full[s], (v0 + v1) * C::kHalfBytes);
                if (v0) tma_load_2d(st, &kmap, 64 * h, page0 * kBlock, &b_full[s]);
                if (v1) tma_load_2d(st + C::kHalfBytes, &kmap, 64 * h, page1 * kBlock, &b_full[s]);
              } else {
                mbar_arrive(&b_full[s]);  // nothing to load; the epilogue writes -inf
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            stop = true;
            break;
          }
        }
      }
    } else if ((warp == 1 || warp == kIssuerWarp2) && lane == 0) {
      // ---------------- MMA issuers: D = Q_tile x [K_block0; K_block1]^T, both
      // operands in shared memory.  Issuer ii takes items j = ii mod 2: ring
      // stages and accumulators are then each used by one issuer, in order.
      // Both walk every row tile: each waits for its queries and commits
      // once to their release (after its own MMAs of the tile, if any).
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
          const int buf = j % kAccBufs;
          if (j >= kAccBufs && !mbar_wait(&acc_empty[buf], ((j / kAccBufs) - 1) & 1)) {
            misc[1] = 1;
            break;
          }
          const uint64_t ad = tc::desc_kmajor_sw128(smem_u32(smem + C::kA + abuf * C::kTileBytes));
          bool stop = false;
          for (int h = 0; h < C::kHalves; ++h) {
            const int u = j * C::kHalves + h, s = u % S;
            if (!mbar_wait(&b_full[s], (u / S) & 1)) {
              stop = true;
              break;
            }
            fence_after();
            const int sv = stage_valid[s];
            if (sv & 3) {
              const uint64_t bd = tc::desc_kmajor_sw128(smem_u32(smem + C::kB + s * C::kStageBytes));
              const uint32_t idesc = (sv & 4) ? kIdescPair : kIdescOne;
#pragma unroll
              for (int kk = 0; kk < C::kAtomSteps; ++kk)
                tc::mma_ss(tmem + buf * kPairCols,
                           tc::desc_advance(ad, h * C::kHalfBytes + kk * 32),
                           tc::desc_advance(bd, kk * 32), idesc, (h | kk) ? 1u : 0u);
            }
            commit(&b_empty[s]);
          }
          if (stop) {
            misc[1] = 1;
            break;
          }
          commit(&acc_full[buf]);
        }
        Cursor nx = cur;
        nx.next(b, prefix, R);
        if (j == n_items - 1 || nx.q != cur.q || nx.tile != cur.tile) commit(&a_empty[abuf]);
        cur = nx;
      }
    } else if (warp >= 10 && warp < 14) {
      // ---------------- query loaders: each row tile of the CTA's items into
      // shared memory, double-buffered, in the 128-byte-swizzled K-major
      // layout the MMA reads (row m's 16-byte chunk c of atom column h at
      // h * 16 KB + m * 128 + 16 * (c ^ (m & 7))); rows past the request's
      // end are zero
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      int a_seq = 0;
      for (int j = 0; j < n_items; ++j) {
        const bool new_tile = j == 0 || cur.pr == 0;  // a tile's items start at pair 0
        if (new_tile) {
          const int ab = a_seq & 1;
          if (a_seq >= 2 && !__all_sync(0xffffffffu, mbar_wait(&a_empty[ab], ((a_seq >> 1) - 1) & 1))) {
            misc[1] = 1;
            break;
          }
          const int row = cur.tile * kTileRows + m;
          const uint4* src = reinterpret_cast<const uint4*>(p.idx_q + (long long)(cur.q0 + row) * DI);
          const bool have = row < cur.qlen;
          uint8_t* dst = smem + C::kA + ab * C::kTileBytes + m * 128;
#pragma unroll
          for (int c = 0; c < DI / 8; ++c) {
            const uint4 v = have ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(dst + (c >> 3) * C::kHalfBytes + 16 * ((c & 7) ^ (m & 7))) = v;
          }
          fence_proxy_async_smem();  // generic stores before the MMA's async reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[ab]);
          ++a_seq;
        }
        cur.next(b, prefix, R);
      }
    } else if (warp >= 2 && warp < 10) {
      // ---------------- epilogue: warps 2-5 reduce block 0 of every item
      // (accumulator columns 0..127), warps 6-9 block 1 (128..255); warp w
      // reads TMEM lanes 32 (w % 4) .. +31 = 32 query rows, each reduced to
      // its causal-masked max.  Blocks every row of the warp sees in full
      // skip the mask; the next item's page id is loaded while this one is
      // reduced.
      const int e = (warp - 2) >> 2, quarter = warp & 3;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      int page = cur.page(b, e);
      for (int j = 0; j < n_items; ++j) {
        const int buf = j % kAccBufs;
        Cursor nx = cur;
        int page_nx = 0;
        if (j + 1 < n_items) {
          nx.next(b, prefix, R);
          page_nx = nx.page(b, e);
        }
        // warp-uniform decision: tcgen05.ld below needs the whole warp
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j / kAccBufs) & 1))) {
          misc[1] = 1;
          break;
        }
        fence_after();
        const int blk = 2 * cur.pr + e;
        const int m = quarter * 32 + lane;
        const int row_in_req = cur.tile * kTileRows + m;
        const int last = cur.ctx + row_in_req - blk * kBlock;  // visible columns: c <= last
        float best = -INFINITY;
        if (page != -2) {  // the pair has this block
          const uint32_t ta = tmem + lanes + buf * kPairCols + e * kBlock;
          best = __all_sync(0xffffffffu, last >= kBlock - 1) ? row_max128<false>(ta, last)
                                                             : row_max128<true>(ta, last);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        if (page != -2 && row_in_req < cur.qlen && last >= 0)
          p.scores[(long long)(cur.q0 + row_in_req) * p.score_stride + blk] =
              (page >= 0 && page < b.num_pages) ? best : -INFINITY;
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
