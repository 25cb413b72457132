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
//   warp 0  TMA producer: Q tile (once per row tile) and K block per item,
//           128-byte-swizzled tiles via cp.async.bulk.tensor into a 4-stage
//           ring with mbarrier completion;
//   warp 1  allocates 256 TMEM columns (two 128-column accumulators);
//           one thread issues the MMAs and tcgen05.commit;
//   warps 2-5 epilogue: tcgen05.ld of 32 rows x 128 columns each, masked
//           max, score store; releases the accumulator.
// Every wait is bounded; on expiry the kernel records MSA_DEV_TIMEOUT, stops
// issuing work and still frees its TMEM.
#include "tcgen05.cuh"

namespace msa {
namespace {

constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr int kTileRows = 128;
constexpr uint32_t kTmemCols = 256;

template <int DI>
struct TcCfg {
  static constexpr int kHalves = DI / 64;          // 128-byte swizzle atoms along K
  static constexpr int kTileBytes = kTileRows * DI * 2;
  static constexpr int kHalfBytes = kTileRows * 128;
  static constexpr int kKSteps = DI / 16;
  // smem: A tile, B ring, then barriers / bookkeeping, then request prefix
  static constexpr int kA = 0;
  static constexpr int kB = kTileBytes;
  static constexpr int kBars = kB + kTcStages * kTileBytes;
  static constexpr int kMisc = kBars + 16 * 8;
  static constexpr int kPrefix = kMisc + 64;
  static_assert(8 + kTcStages <= 16, "misc area holds 16 ints");
  static size_t bytes(int num_reqs) { return 1024 + kPrefix + (size_t)(num_reqs + 1) * 4; }
};

using tc::commit;
using tc::fence_after;
using tc::fence_before;
using tc::tmem_ld32;

// Instruction descriptor of the score tile: M = 128 rows, N = 128 tokens.
constexpr uint32_t kIdesc = tc::idesc_bf16(128, 128, 0);

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

template <int DI>
__global__ void __launch_bounds__(kTcThreads, 1)
    index_score_tc_kernel(const ScoreLaunch p, const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap) {
  using C = TcCfg<DI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint64_t* b_full = bars;                   // [kTcStages]
  uint64_t* b_empty = bars + kTcStages;      // [kTcStages]
  uint64_t* a_full = bars + 2 * kTcStages;
  uint64_t* a_empty = a_full + 1;
  uint64_t* acc_full = a_full + 2;           // [2]
  uint64_t* acc_empty = a_full + 4;          // [2]
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
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    fence_barrier_init();
  }
  __syncthreads();
  for (int q = tid; q < R; q += blockDim.x) {
    int q0, ql, ctx, nb;
    const uint32_t bad = request_lengths(b, q, &q0, &ql, &ctx, &nb);
    if (ql < 0) misc[0] = 1;
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
  const bool batch_ok = misc[0] == 0;  // the CUDA-core kernel reports the status bits
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
      int a_key_q = -1, a_key_t = -1, a_loads = 0;
      bool stop = false;
      for (int j0 = 0; j0 < n_items && !stop; j0 += 32) {
        int mq = 0, mt = 0, mq0 = 0, mpage = -1;
        if (j0 + lane < n_items) {
          Cursor cur;
          cur.seek(b, prefix, R, i0 + j0 + lane);
          mq = cur.q;
          mt = cur.tile;
          mq0 = cur.q0;
          mpage = b.block_table[(long long)cur.q * b.bt_stride + cur.blk];
        }
        const int cnt = min(32, n_items - j0);
        for (int jj = 0; jj < cnt; ++jj) {
          const int j = j0 + jj;
          const int q = __shfl_sync(0xffffffffu, mq, jj);
          const int t = __shfl_sync(0xffffffffu, mt, jj);
          const int q0 = __shfl_sync(0xffffffffu, mq0, jj);
          const int page = __shfl_sync(0xffffffffu, mpage, jj);
          int ok = 1;
          if (lane == 0) {
            if (q != a_key_q || t != a_key_t) {
              if (a_loads > 0 && !mbar_wait(a_empty, (a_loads - 1) & 1)) {
                ok = 0;
              } else {
                mbar_arrive_expect_tx(a_full, C::kTileBytes);
                for (int h = 0; h < C::kHalves; ++h)
                  tma_load_2d(smem + C::kA + h * C::kHalfBytes, &qmap, 64 * h, q0 + t * kTileRows,
                              a_full);
                a_key_q = q;
                a_key_t = t;
                ++a_loads;
              }
            }
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
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      int a_key_q = -1, a_key_t = -1, a_loads = 0;
      for (int j = 0; j < n_items; ++j) {
        if (cur.q != a_key_q || cur.tile != a_key_t) {
          if (!mbar_wait(a_full, a_loads & 1)) {
            misc[1] = 1;
            break;
          }
          a_key_q = cur.q;
          a_key_t = cur.tile;
          ++a_loads;
        }
        const int s = j % kTcStages, buf = j & 1;
        if (j >= 2 && !mbar_wait(&acc_empty[buf], ((j >> 1) - 1) & 1)) {
          misc[1] = 1;
          break;
        }
        if (!mbar_wait(&b_full[s], (j / kTcStages) & 1)) {
          misc[1] = 1;
          break;
        }
        fence_after();
        if (stage_valid[s]) {
          const uint32_t a_base = smem_u32(smem + C::kA);
          const uint32_t b_base = smem_u32(smem + C::kB + s * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < C::kKSteps; ++kk) {
            const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
            tc::mma_ss(tmem + buf * 128, tc::desc_kmajor_sw128(a_base + off),
                       tc::desc_kmajor_sw128(b_base + off), kIdesc, kk > 0 ? 1u : 0u);
          }
        }
        commit(&b_empty[s]);
        commit(&acc_full[buf]);
        Cursor nx = cur;
        nx.next(b, prefix, R);
        if (j == n_items - 1 || nx.q != cur.q || nx.tile != cur.tile) commit(a_empty);
        cur = nx;
      }
    } else if (warp >= 2) {
      // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31
      const int quarter = warp & 3;
      Cursor cur;
      cur.seek(b, prefix, R, i0);
      for (int j = 0; j < n_items; ++j) {
        const int buf = j & 1;
        // warp-uniform decision: tcgen05.ld below needs the whole warp
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j >> 1) & 1))) {
          misc[1] = 1;
          break;
        }
        fence_after();
        const int m = quarter * 32 + lane;
        const int row_in_req = cur.tile * kTileRows + m;
        const int pos = cur.ctx + row_in_req;
        const int page = b.block_table[(long long)cur.q * b.bt_stride + cur.blk];
        const bool page_ok = page >= 0 && page < b.num_pages;
        const int last = pos - cur.blk * kBlock;  // visible columns: c <= last
        float best = -INFINITY;
#pragma unroll
        for (int chunk = 0; chunk < 4; ++chunk) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + buf * 128 + chunk * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (chunk * 32 + i <= last) best = fmaxf(best, v[i]);
        }
        if (row_in_req < cur.qlen && last >= 0)
          p.scores[(long long)(cur.q0 + row_in_req) * p.score_stride + cur.blk] =
              page_ok ? best : -INFINITY;
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        cur.next(b, prefix, R);
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
  CUtensorMap qmap, kmap;
  if (!make_map(&qmap, p.idx_q, (long long)p.batch.num_rows, DI) ||
      !make_map(&kmap, p.idx_k, (long long)p.batch.num_pages * kBlock, DI))
    return cudaErrorInvalidValue;
  const size_t smem = TcCfg<DI>::bytes(p.batch.num_reqs);
  auto kern = index_score_tc_kernel<DI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<device_sm_count(), kTcThreads, smem, stream>>>(p, qmap, kmap);
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
