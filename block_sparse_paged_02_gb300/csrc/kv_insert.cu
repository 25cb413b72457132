// kv_insert.cu -- the step before the path: write the new tokens' K, V and
// index-K into the paged pools.
//
// Definition ("Add ROCm AITER sparse paged attention for MiniMax-M3", vLLM PR
// 47287, "Implementation breakdown" item 1: the fused q/k-norm + RoPE + KV
// insert takes a skip_index flag so that index-reuse layers skip the index
// cache write; item 5: K and V live in separate page pools): every query row
// of a request is a new token at its own absolute position, so its K, V and
// index-K go to page block_table[q, pos/128], slot pos%128.  FP8 caches take
// OCP e4m3 codes: with a scalar scale the value is divided by it; with
// per-token-head scales the scale is max|x|/448 of that token and KV head (1
// for an all-zero vector), written beside the page.  (The norm and RoPE parts
// of the fused op need model weights and are not part of this library.)
//
// One warp per row: lanes own 4 consecutive head dims; the amax is a warp
// max-reduce; division is IEEE fp32 and the codes come from the hardware
// round-to-nearest-even, saturating e4m3 conversion.  An FP8 index cache is
// written the same way per token and index head (the per-token-head rule when
// its scales are kept, scale 1 otherwise).
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kWarpsPerCta = 4;

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// One KV vector of head_dim 128 (4 dims per lane) into the cache slot.
__device__ __forceinline__ void insert_vector(const uint16_t* src, uint8_t* cache, long long dst,
                                              int fp8, int scale_mode, const float* given,
                                              float* scale_out, long long scale_at, int lane) {
  const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
  if (!fp8) {
    *reinterpret_cast<uint2*>(cache + 2 * (dst + 4 * lane)) = raw;
    return;
  }
  const float x0 = bf16lo(raw.x), x1 = bf16hi(raw.x), x2 = bf16lo(raw.y), x3 = bf16hi(raw.y);
  float s = 1.f;
  if (scale_mode == MSA_SCALE_SCALAR) {
    s = __ldg(given);
  } else if (scale_mode == MSA_SCALE_PER_TOKEN_HEAD) {
    float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (lane == 0) scale_out[scale_at] = s;
  }
  const uint32_t codes = pack_e4m3x4(__fdiv_rn(x0, s), __fdiv_rn(x1, s), __fdiv_rn(x2, s),
                                     __fdiv_rn(x3, s));
  *reinterpret_cast<uint32_t*>(cache + dst + 4 * lane) = codes;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32) kv_insert_kernel(const KvInsertLaunch p) {
  const msa_batch& b = p.batch;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * kWarpsPerCta + warp;
  if (r >= b.num_rows) return;
  const int R = b.num_reqs;
  const unsigned full = 0xffffffffu;

  // the row's request and the request's checks (as for top-k)
  bool tiled = true;
  int le = 0;
  for (int base = 0; base < R; base += 32) {
    const int q = base + lane;
    if (q < R) {
      const int c0 = b.cu_seqlens_q[q], c1 = b.cu_seqlens_q[q + 1];
      tiled &= c1 >= c0;
      le += c0 <= r;
    }
  }
  tiled = __all_sync(full, tiled) && b.cu_seqlens_q[0] == 0 && b.cu_seqlens_q[R] == b.num_rows;
  le = __reduce_add_sync(full, le);
  uint32_t bad = tiled ? 0u : MSA_DEV_MALFORMED;
  int q = -1, q0 = 0, qlen = 0, ctx = 0, nbq = 0;
  if (!bad) {
    q = le - 1;
    bad = request_lengths(b, q, &q0, &qlen, &ctx, &nbq);
  }
  if (!bad) {
    bool page_bad = false;
    for (int blk = lane; blk < nbq; blk += 32) {
      const int page = b.block_table[(long long)q * b.bt_stride + blk];
      page_bad |= page < 0 || page >= b.num_pages;
    }
    if (__any_sync(full, page_bad)) bad = MSA_DEV_BAD_PAGE;
  }
  if (bad) {
    if (lane == 0 && ((q >= 0) ? (r == q0) : (r == 0))) atomicOr(p.status, bad);
    return;
  }
  const int pos = ctx + (r - q0);
  const long long page = b.block_table[(long long)q * b.bt_stride + pos / kBlock];
  const long long token = page * kBlock + pos % kBlock;  // flat slot in the [P*128] token space

  for (int h = 0; h < p.num_kv_heads; ++h) {
    const long long src = ((long long)r * p.num_kv_heads + h) * kHeadDim;
    const long long dst = (token * p.num_kv_heads + h) * kHeadDim;
    const long long sat = token * p.num_kv_heads + h;
    insert_vector(p.k_new + src, p.k_cache, dst, p.kv_fp8, p.scale_mode, p.k_scale, p.k_scale,
                  sat, lane);
    insert_vector(p.v_new + src, p.v_cache, dst, p.kv_fp8, p.scale_mode, p.v_scale, p.v_scale,
                  sat, lane);
  }
  if (!p.skip_index && p.idx_fp8) {
    // e4m3 index keys per (token, index head); index_dim 64 or 128, so each
    // lane owns 2 or 4 consecutive dims
    for (int h = 0; h < p.index_heads; ++h) {
      const long long sat = token * p.index_heads + h;
      const uint16_t* src = p.idx_new + ((long long)r * p.index_heads + h) * p.index_dim;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.idx_k_cache) + sat * p.index_dim;
      if (p.index_dim == 128) {
        insert_vector(src, dst, 0, 1, p.idx_scale ? MSA_SCALE_PER_TOKEN_HEAD : MSA_SCALE_NONE,
                      nullptr, p.idx_scale, sat, lane);
      } else {
        const uint32_t raw = *reinterpret_cast<const uint32_t*>(src + 2 * lane);
        const float x0 = bf16lo(raw), x1 = bf16hi(raw);
        float s = 1.f;
        if (p.idx_scale) {
          float amax = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
          if (lane == 0) p.idx_scale[sat] = s;
        }
        uint16_t code;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(code) : "f"(__fdiv_rn(x1, s)), "f"(__fdiv_rn(x0, s)));
        *reinterpret_cast<uint16_t*>(dst + 2 * lane) = code;
      }
    }
  } else if (!p.skip_index) {
    const int n = p.index_heads * p.index_dim;  // bf16 elements, a multiple of 4
    const uint2* src = reinterpret_cast<const uint2*>(p.idx_new + (long long)r * n);
    uint2* dst = reinterpret_cast<uint2*>(p.idx_k_cache + token * n);
    for (int i = lane; i < n / 4; i += 32) dst[i] = src[i];
  }
}

}  // namespace

cudaError_t launch_kv_insert(const KvInsertLaunch& p, cudaStream_t stream) {
  if (p.batch.num_rows == 0) return cudaSuccess;
  const int grid = (p.batch.num_rows + kWarpsPerCta - 1) / kWarpsPerCta;
  kv_insert_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace msa
