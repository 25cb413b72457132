// sparse_mla.cu -- sparse MLA decode with attention sinks and a natural-log
// LSE.
//
// Definition ("Attention sinks for ROCm AITER sparse MLA", vLLM PR 54404,
// "Implementation breakdown" items 1-2 and "Key source snippets"): one
// latent KV head whose cached row per token holds dqk = 576 values (512
// latent + 64 rope); the key is the whole row, the value its first dv = 512
// values.  Query row r attends over the token ids
// kv_indices[kv_indptr[r] .. kv_indptr[r+1]) (the indptr / indices
// convention of the MLA decode op), with the sink in the softmax denominator
// and the natural-log LSE of that denominator; sinks are fp32 [heads].
//
// GB300 design.  16 heads x 16 tokens is a real tensor-core tile: a CTA of 4
// warps owns 16 heads of one row and a contiguous span of its token list.
// Per step of 16 tokens the token rows (1152 B each) are gathered by 16-byte
// asynchronous copies from all threads into a 4-deep shared ring, rows 16 B
// apart more than their size so that ldmatrix reads are conflict-free; warp
// w computes the partial logits over dims [144w, 144w + 144) (mma.sync
// m16n8k16, bf16, fp32 accumulation), the four partials are summed through
// shared memory (one barrier per step, double buffered; the same barrier
// publishes the next step's rows), every warp runs the same online softmax, and warp
// w accumulates O for value dims [128w, 128w + 128) (64 fp32 registers per
// lane).  Up to 8 splits of a (row, head group) form one thread-block
// cluster and merge their (m, l, acc) through distributed shared memory;
// more splits merge through workspace partials, finished by the
// last-arriving CTA (atomic counter; its top bit carries "an id was out of
// range" from any split).
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kMlaDqk = 576, kMlaDv = 512;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStepTok = 16;                       // tokens per step
constexpr int kRowBytes = kMlaDqk * 2;             // 1152 B per cached token
// staged rows are 1168 B apart (16 B more than a row): the 8 rows an
// ldmatrix reads then start 4 banks apart, which makes every read conflict-free
constexpr int kRowPitch = kRowBytes + 16;
constexpr int kStages = 4;
constexpr int kStageBytes = kStepTok * kRowPitch;  // 18.25 KB
constexpr int kKQuarter = kMlaDqk / kWarps;        // 144 dims of the logits per warp
constexpr int kKSteps = kKQuarter / 16;            // 9
constexpr int kVQuarter = kMlaDv / kWarps;         // 128 value dims per warp
constexpr int kXchgFloats = kWarps * 32 * 8;       // one step's partial logits
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.f;  // log2 units
constexpr int kPartHeadFloats = 4 + kMlaDv;        // m, l, 2 pad, acc[512] (16-B aligned)

struct MlaSmem {
  static constexpr int kRing = 0;
  static constexpr int kXchg = kRing + kStages * kStageBytes;
  static constexpr int kIds = kXchg + 2 * kXchgFloats * 4;
  static constexpr int kMaxIds = 2048;  // token ids of one split held in shared memory
  static constexpr int kFlags = kIds + kMaxIds * 4;
  static constexpr int kBytes = kFlags + 64;
};

// FP8 latent cache: e4m3 rows (576 B, 592 B apart) land by 16-byte
// asynchronous copies in a 4-deep ring, the same pipeline as bf16 rows; the
// MMA fragments are read straight from the e4m3 bytes and converted to f16
// (exact) in registers.  Logits: lane (g, c) takes the 4 consecutive dims
// 16kk + 4c .. + 3 of token g as its k-slots (2c, 2c+1, 2c+8, 2c+9) -- one
// 32-bit read; the queries use the same slot order.  Values: lane (g, c)
// reads dims 16g .. 16g + 15 of tokens 2c, 2c+1, 2c+8, 2c+9 (16 bytes each)
// and pairs the tokens' bytes with byte permutes, so n-tile j's column g is
// value dim 16g + j of the warp's 128.  (A converted f16 copy of each step
// in shared memory measured 12.5 us slower on the 64-row workload.)
constexpr int kRowPitch8 = kMlaDqk + 16;            // 592 B: rows 4 banks apart
constexpr int kStageBytes8 = kStepTok * kRowPitch8; // 9.25 KB
struct MlaSmem8 {
  static constexpr int kRing = 0;
  static constexpr int kXchg = kRing + kStages * kStageBytes8;
  static constexpr int kIds = kXchg + 2 * kXchgFloats * 4;
  static constexpr int kFlags = kIds + MlaSmem::kMaxIds * 4;
  static constexpr int kBytes = kFlags + 64;
  static_assert(16 * kPartHeadFloats * 4 <= kXchg, "partials fit before the exchange area");
};

// four 8x8 b16 matrices; lane l gives the row address of matrix l/8, row l%8
// and receives (row g, cols 2c, 2c+1) of each (transposed: (rows 2c, 2c+1, col g))
__device__ __forceinline__ void ldsm_x4(const void* row, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row))
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(const void* row, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row))
               : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool FP8KV>
__global__ void __launch_bounds__(kThreads, 2) sparse_mla_kernel(const MlaLaunch p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem + (FP8KV ? MlaSmem8::kRing : MlaSmem::kRing);
  float* xchg = reinterpret_cast<float*>(smem + (FP8KV ? MlaSmem8::kXchg : MlaSmem::kXchg));
  int* ids = reinterpret_cast<int*>(smem + (FP8KV ? MlaSmem8::kIds : MlaSmem::kIds));
  int* flags = reinterpret_cast<int*>(smem + (FP8KV ? MlaSmem8::kFlags : MlaSmem::kFlags));

  const int split = blockIdx.x, hg = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const unsigned full = 0xffffffffu;

  // ---- this split's span of the row's token list
  const long long b0 = p.indptr[r], b1 = p.indptr[r + 1];
  const long long n_row = b1 - b0;
  const long long lo = (long long)split * p.tokens_per_split;
  const long long hi = (split == p.splits - 1) ? n_row : min(n_row, lo + p.tokens_per_split);
  const int n = n_row < 0 ? 0 : (int)max(0ll, min(hi - lo, (long long)MlaSmem::kMaxIds));
  // rows longer than the caller's bound (which sized the splits) are refused
  bool bad = n_row < 0 || n_row > p.max_tokens || hi - lo > MlaSmem::kMaxIds;
  for (int i = tid; i < n; i += kThreads) {
    const int t = p.indices[b0 + lo + i];
    bad |= t < 0 || (long long)t >= p.num_tokens;
    ids[i] = t;
  }
  const bool cta_bad = __syncthreads_or(bad) != 0;
  const int n_steps = cta_bad ? 0 : (n + kStepTok - 1) / kStepTok;

  // ---- gather: 16-byte asynchronous copies spread over all threads, one
  // commit group per step (empty past the last step).  (One 1152-byte bulk
  // copy per row through the TMA engine measured slower: 67.2 vs 62.9 us.)
  auto gather = [&](int step) {
    if (step < n_steps) {
      const int st = step % kStages;
      const int t0 = step * kStepTok;
      const int cnt = min(kStepTok, n - t0);
      if constexpr (FP8KV) {
        uint8_t* dst = ring + st * kStageBytes8;
        const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
        constexpr int kChunksPerRow = kMlaDqk / 16;  // 36
#pragma unroll
        for (int k = 0; k < (kStepTok * kChunksPerRow + kThreads - 1) / kThreads; ++k) {
          const int q = tid + kThreads * k;
          const int row = q / kChunksPerRow, col = q - row * kChunksPerRow;
          if (row < cnt)
            cp_async16(dst + row * kRowPitch8 + 16 * col,
                       kv8 + (long long)ids[t0 + row] * kMlaDqk + 16 * col);
        }
      } else {
        uint8_t* dst = ring + st * kStageBytes;
        constexpr int kChunksPerRow = kRowBytes / 16;  // 72
#pragma unroll
        for (int k = 0; k < kStepTok * kChunksPerRow / kThreads; ++k) {
          const int q = tid + kThreads * k;
          const int row = q / kChunksPerRow, col = q - row * kChunksPerRow;
          if (row < cnt)
            cp_async16(dst + row * kRowPitch + 16 * col,
                       p.kv + (long long)ids[t0 + row] * kMlaDqk + 8 * col);
        }
      }
    }
    cp_async_commit();
  };
  for (int s = 0; s < kStages; ++s) gather(s);
  cp_async_wait<kStages - 1>();  // step 0 has landed (this thread's part)
  __syncthreads();               // ... everyone's

  // ---- query fragments (A of S = Q K^T): heads 16hg + {g, g+8}, k-step kk
  // of this warp's dims [144 warp, +144): columns 16kk + 2c (+1) and +8
  uint32_t qa[kKSteps][4];
  const bool q_bf16 = !FP8KV;  // (with an e4m3 cache the queries load below)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int h = 16 * hg + g + 8 * half;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        p.q + ((long long)r * p.num_heads + h) * kMlaDqk + kKQuarter * warp + 2 * c);
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      const bool live = q_bf16 && h < p.num_heads;
      qa[kk][half] = live ? __ldg(qrow + 8 * kk) : 0u;          // cols 16kk + 2c, +1
      qa[kk][2 + half] = live ? __ldg(qrow + 8 * kk + 4) : 0u;  // cols 16kk + 8 + 2c, +1
    }
  }
  if constexpr (FP8KV) {
    // f16 operands in the key spans' slot order: k-slots (2c, 2c+1) and
    // (2c+8, 2c+9) of k-step kk are dims 16kk + 4c, +1 and +2, +3 of the
    // warp's 144; bf16 queries convert (|q| < 65504), e4m3 codes exactly
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int h = 16 * hg + g + 8 * half;
      const bool live = h < p.num_heads;
      const long long qoff = ((long long)r * p.num_heads + (live ? h : 0)) * kMlaDqk +
                             kKQuarter * warp + 4 * c;
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        uint32_t lo = 0u, hi = 0u;
        if (p.q_fp8) {
          const uint32_t w = live ? __ldg(reinterpret_cast<const uint32_t*>(
                                          reinterpret_cast<const uint8_t*>(p.q) + qoff + 16 * kk))
                                  : 0u;
          lo = e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
          hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
        } else if (live) {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(p.q + qoff + 16 * kk));
          lo = pack_f16x2(bf16lo(w.x), bf16hi(w.x));
          hi = pack_f16x2(bf16lo(w.y), bf16hi(w.y));
        }
        qa[kk][half] = lo;
        qa[kk][2 + half] = hi;
      }
    }
  }
  // ldmatrix row addresses of this lane: matrix mi = lane / 8, row lane % 8
  const int mi = lane >> 3, mrow = lane & 7;
  // K (B of Q K^T, k = dims, n = tokens): matrices (tokens 0-7 | 8-15) x
  // (dims 16kk + 0-7 | 8-15) give n-tile 0's and 1's two k-halves
  const int k_off = ((mi >> 1) * 8 + mrow) * kRowPitch + (kKQuarter * warp + (mi & 1) * 8) * 2;
  // V (B of P V, k = tokens, n = dims), transposed: matrices (tokens 0-7 |
  // 8-15) x (dims 16jj + 0-7 | 8-15) give n-tiles 2jj and 2jj+1
  const int v_off = ((mi & 1) * 8 + mrow) * kRowPitch + (kVQuarter * warp + (mi >> 1) * 8) * 2;
  float scale2 = p.softmax_scale * kLog2e;  // logits in log2 units
  if constexpr (FP8KV) {
    scale2 *= __ldg(p.kv_scale);
    if (p.q_fp8) scale2 *= __ldg(p.q_scale);
  }

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  for (int step = 0; step < n_steps; ++step) {
    const int st = step % kStages;
    const uint8_t* stage = ring + st * (FP8KV ? kStageBytes8 : kStageBytes);
    const int nvalid = min(kStepTok, n - step * kStepTok);

    // ---- partial logits over this warp's 144 dims: n-tile nt = tokens 8nt + g
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    if constexpr (FP8KV) {
      // token 8nt + g, dims 16kk + 4c .. + 3 of the warp's 144: one word
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint8_t* krow = stage + (8 * nt + g) * kRowPitch8 + kKQuarter * warp + 4 * c;
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(krow + 16 * kk);
          mma16816<true>(s[nt], qa[kk], e4m3x2_to_f16x2((uint16_t)(w & 0xffffu)),
                         e4m3x2_to_f16x2((uint16_t)(w >> 16)));
        }
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        uint32_t kb[4];
        ldsm_x4(stage + k_off + 32 * kk, kb);
        mma16816<false>(s[0], qa[kk], kb[0], kb[1]);
        mma16816<false>(s[1], qa[kk], kb[2], kb[3]);
      }
    }
    float* xw = xchg + (step & 1) * kXchgFloats;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) xw[(warp * 8 + 4 * nt + e) * 32 + lane] = s[nt][e];
    // the next step's rows have landed (this thread's part; steps complete
    // in order), and the one barrier of the step makes them everyone's
    cp_async_wait<kStages - 3>();
    __syncthreads();
    // the same sum, in the same order, in every warp
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += xw[(w * 8 + 4 * nt + e) * 32 + lane];
        const int t = 8 * nt + 2 * c + (e & 1);
        s[nt][e] = t < nvalid ? v * scale2 : -INFINITY;
      }
    // the stage of the previous step is free in every warp now
    if (step >= 1) gather(step - 1 + kStages);

    // ---- online softmax (rows g and g+8), lazy rescaling
    float mx[2];
    mx[0] = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    mx[1] = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    bool move[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(full, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(full, mx[hh], 2));
      move[hh] = mx[hh] > m_run[hh] + kRescaleSlack;
    }
    if (__any_sync(full, move[0] || move[1])) {
      float alpha[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        alpha[hh] = 1.f;
        if (move[hh]) {
          alpha[hh] = m_run[hh] == -INFINITY ? 0.f : exp2f(m_run[hh] - mx[hh]);
          m_run[hh] = mx[hh];
        }
        l_run[hh] *= alpha[hh];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= alpha[0];
        o[j][1] *= alpha[0];
        o[j][2] *= alpha[1];
        o[j][3] *= alpha[1];
      }
    }
    const float base[2] = {m_run[0] == -INFINITY ? 0.f : m_run[0],
                           m_run[1] == -INFINITY ? 0.f : m_run[1]};
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[nt][e] = exp2f(s[nt][e] - base[e >> 1]);
    l_run[0] += pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
    l_run[1] += pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
    uint32_t pa[4];
    if constexpr (FP8KV) {
      pa[0] = pack_f16x2(pr[0][0], pr[0][1]);
      pa[1] = pack_f16x2(pr[0][2], pr[0][3]);
      pa[2] = pack_f16x2(pr[1][0], pr[1][1]);
      pa[3] = pack_f16x2(pr[1][2], pr[1][3]);
    } else {
      pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
      pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
      pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
      pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
    }

    // ---- O += P V over this warp's value dims (n-tile j = dims 8j .. 8j+7);
    // rows past the end of the list hold stale or unwritten data: their
    // value halves are zeroed (their weight is already 0)
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;  // tokens (2c, 2c+1), (2c+8, 2c+9)
    if (nvalid < kStepTok) {
      keep_lo = (2 * c < nvalid ? 0x0000ffffu : 0u) | (2 * c + 1 < nvalid ? 0xffff0000u : 0u);
      keep_hi = (2 * c + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * c + 9 < nvalid ? 0xffff0000u : 0u);
    }
    if constexpr (FP8KV) {
      // tokens 2c, 2c+1, 2c+8, 2c+9: value dims 16g .. 16g + 15 of the
      // warp's 128, 16 bytes each; n-tile j takes byte j of each (column g
      // of n-tile j = value dim 16g + j), the two tokens of a k-slot pair
      // joined by a byte permute
      uint32_t vw[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int t = 2 * c + (a & 1) + 8 * (a >> 1);
        const uint4 v = lds128(stage + t * kRowPitch8 + kVQuarter * warp + 16 * g);
        vw[a][0] = v.x; vw[a][1] = v.y; vw[a][2] = v.z; vw[a][3] = v.w;
      }
#pragma unroll
      for (int j2 = 0; j2 < 8; ++j2) {  // n-tiles 2 j2, 2 j2 + 1
        const int wi = j2 >> 1, by = 2 * (j2 & 1);
        const uint32_t sel = (uint32_t)(by | ((4 + by) << 4) | ((by + 1) << 8) | ((5 + by) << 12));
        const uint32_t lo = prmt(vw[0][wi], vw[1][wi], sel);  // tokens 2c, 2c+1
        const uint32_t hi = prmt(vw[2][wi], vw[3][wi], sel);  // tokens 2c+8, 2c+9
        mma16816<true>(o[2 * j2], pa, e4m3x2_to_f16x2((uint16_t)(lo & 0xffffu)) & keep_lo,
                       e4m3x2_to_f16x2((uint16_t)(hi & 0xffffu)) & keep_hi);
        mma16816<true>(o[2 * j2 + 1], pa, e4m3x2_to_f16x2((uint16_t)(lo >> 16)) & keep_lo,
                       e4m3x2_to_f16x2((uint16_t)(hi >> 16)) & keep_hi);
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t vb[4];
        ldsm_x4_t(stage + v_off + 32 * jj, vb);
        const uint32_t b0[2] = {vb[0] & keep_lo, vb[2] & keep_lo};
        const uint32_t b1[2] = {vb[1] & keep_hi, vb[3] & keep_hi};
        mma16816<false>(o[2 * jj], pa, b0[0], b1[0]);
        mma16816<false>(o[2 * jj + 1], pa, b0[1], b1[1]);
      }
    }
  }

#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(full, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(full, l_run[hh], 2);
  }

  // ---- this split's partial: m, l per head; acc per head and value dim
  float* part = p.partials + (((long long)r * p.head_groups + hg) * p.splits + split) * 16 *
                                 kPartHeadFloats;
  auto put = [&](float* dst, const float (&acc)[16][4], const float (&m)[2], const float (&l)[2]) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float* ph = dst + (g + 8 * half) * kPartHeadFloats;
      if (warp == 0 && c == 0) {
        ph[0] = m[half];
        ph[1] = l[half];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        // c0,c1 (half 0) / c2,c3 (half 1): columns 2c, 2c+1 of n-tile j, i.e.
        // dims 8j + 2c, +1 of this warp's 128 (bf16 cache) or 16 (2c) + j,
        // 16 (2c + 1) + j (e4m3 cache)
        if constexpr (FP8KV) {
          ph[4 + kVQuarter * warp + 32 * c + j] = acc[j][2 * half];
          ph[4 + kVQuarter * warp + 32 * c + 16 + j] = acc[j][2 * half + 1];
        } else {
          ph[4 + kVQuarter * warp + 8 * j + 2 * c] = acc[j][2 * half];
          ph[4 + kVQuarter * warp + 8 * j + 2 * c + 1] = acc[j][2 * half + 1];
        }
      }
    }
  };
  if (p.splits <= kMaxClusterSplits) {
    // ---- the row's splits form one cluster (of 1..8 CTAs): each CTA leaves
    // its (m, l, acc) in its own shared memory, one barrier publishes them,
    // and every CTA merges a share of the 16 x 512 outputs over all partials
    // through distributed shared memory; the second barrier keeps each CTA's
    // memory alive until its readers are done.
    cp_async_wait<0>();
    __syncthreads();  // the ring is free now
    float* mine = reinterpret_cast<float*>(smem);
    put(mine, o, m_run, l_run);
    if (tid == 0) flags[2] = cta_bad ? 1 : 0;
    cluster_sync();
    const uint32_t base = smem_u32(mine);
    int fl = 0;
    if (lane < p.splits) fl = ld_dsmem_s32(mapa_shared(smem_u32(&flags[2]), (uint32_t)lane));
    const bool poisoned = __any_sync(full, fl != 0);
    if (poisoned && split == 0 && tid == 0) atomicOr(p.status, MSA_DEV_BAD_TABLE);
    for (int i4 = split * kThreads + tid; i4 < 16 * kMlaDv / 4; i4 += p.splits * kThreads) {
      const int head = i4 / (kMlaDv / 4), d = 4 * (i4 % (kMlaDv / 4));
      const int h_abs = 16 * hg + head;
      if (h_abs >= p.num_heads) break;
      float M = -INFINITY, Lsum = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
      if (!poisoned) {
        float ms[kMaxClusterSplits], ls[kMaxClusterSplits];
        float4 v[kMaxClusterSplits];
#pragma unroll
        for (int j = 0; j < kMaxClusterSplits; ++j) {
          if (j < p.splits) {
            const uint32_t ph = mapa_shared(base, (uint32_t)j) + 4u * head * kPartHeadFloats;
            ms[j] = ld_dsmem_f32(ph);
            ls[j] = ld_dsmem_f32(ph + 4u);
            v[j] = ld_dsmem_f4(ph + 4u * (4 + d));
          }
        }
#pragma unroll
        for (int j = 0; j < kMaxClusterSplits; ++j) M = j < p.splits ? fmaxf(M, ms[j]) : M;
#pragma unroll
        for (int j = 0; j < kMaxClusterSplits; ++j) {
          if (j < p.splits && ms[j] != -INFINITY) {
            const float f = exp2f(ms[j] - M);
            Lsum += f * ls[j];
            a[0] += f * v[j].x;
            a[1] += f * v[j].y;
            a[2] += f * v[j].z;
            a[3] += f * v[j].w;
          }
        }
      }
      if (p.sinks) {
        const float sink2 = __ldg(p.sinks + h_abs) * kLog2e;
        const float Mn = fmaxf(M, sink2);
        const float f = M == -INFINITY ? 0.f : exp2f(M - Mn);
        Lsum = Lsum * f + exp2f(sink2 - Mn);
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] *= f;
        M = Mn;
      }
      float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
      if constexpr (FP8KV) inv *= __ldg(p.kv_scale);  // values are kv_scale * code
      *reinterpret_cast<uint2*>(p.out + ((long long)r * p.num_heads + h_abs) * kMlaDv + d) =
          make_uint2(pack_bf16x2(a[0] * inv, a[1] * inv), pack_bf16x2(a[2] * inv, a[3] * inv));
      if (d == 0)
        p.lse[(long long)r * p.num_heads + h_abs] =
            (M == -INFINITY || Lsum <= 0.f) ? -INFINITY : (M + log2f(Lsum)) * kLn2;
    }
    cluster_sync();
    return;
  }

  // ---- more than 8 splits: publish this split's partial; the last CTA of
  // the (row, head group) merges all.  A CTA that saw an id outside the
  // pool flags the row in the counter's top bit before counting itself in.
  bool poisoned = cta_bad;
  {
    put(part, o, m_run, l_run);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      unsigned* ctr = p.counters + (long long)r * p.head_groups + hg;
      if (cta_bad) atomicOr(ctr, 0x80000000u);
      const unsigned old = atomicAdd(ctr, 1u);
      flags[0] = (old & 0x7fffffffu) == (unsigned)(p.splits - 1);
      flags[1] = ((old | (cta_bad ? 0x80000000u : 0u)) & 0x80000000u) != 0;
      if (flags[0]) *ctr = 0;  // ready for the next call
    }
    __syncthreads();
    if (!flags[0]) return;
    __threadfence();
    poisoned = flags[1] != 0;
  }

  // ---- final: thread t owns head t/8 (of 16) and value dims 64*(t%8) .. +64
  const int head = tid >> 3, d0 = 64 * (tid & 7);
  const int h_abs = 16 * hg + head;
  float M = -INFINITY, Lsum = 0.f, acc[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) acc[j] = 0.f;
  for (int sp = 0; sp < p.splits; ++sp) {
    const float* ph = p.partials +
        ((((long long)r * p.head_groups + hg) * p.splits + sp) * 16 + head) * kPartHeadFloats;
    const float ms = __ldcg(ph), ls = __ldcg(ph + 1);
    const float mn = fmaxf(M, ms);
    const float fo = M == -INFINITY ? 0.f : exp2f(M - mn);
    const float fs = ms == -INFINITY ? 0.f : exp2f(ms - mn);
    Lsum = Lsum * fo + ls * fs;
    const float4* a4 = reinterpret_cast<const float4*>(ph + 4 + d0);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float4 v = __ldcg(a4 + j);
      acc[4 * j] = acc[4 * j] * fo + v.x * fs;
      acc[4 * j + 1] = acc[4 * j + 1] * fo + v.y * fs;
      acc[4 * j + 2] = acc[4 * j + 2] * fo + v.z * fs;
      acc[4 * j + 3] = acc[4 * j + 3] * fo + v.w * fs;
    }
    M = mn;
  }
  if (tid == 0 && poisoned) atomicOr(p.status, MSA_DEV_BAD_TABLE);
  if (poisoned) {  // a poisoned row is an empty row
    M = -INFINITY;
    Lsum = 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
  }
  if (h_abs < p.num_heads) {
    if (p.sinks) {
      const float sink2 = __ldg(p.sinks + h_abs) * kLog2e;
      const float Mn = fmaxf(M, sink2);
      const float f = M == -INFINITY ? 0.f : exp2f(M - Mn);
      Lsum = Lsum * f + exp2f(sink2 - Mn);
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] *= f;
      M = Mn;
    }
    float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    if constexpr (FP8KV) inv *= __ldg(p.kv_scale);  // values are kv_scale * code
    uint4* dst = reinterpret_cast<uint4*>(p.out + ((long long)r * p.num_heads + h_abs) * kMlaDv + d0);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      dst[j] = make_uint4(pack_bf16x2(acc[8 * j] * inv, acc[8 * j + 1] * inv),
                          pack_bf16x2(acc[8 * j + 2] * inv, acc[8 * j + 3] * inv),
                          pack_bf16x2(acc[8 * j + 4] * inv, acc[8 * j + 5] * inv),
                          pack_bf16x2(acc[8 * j + 6] * inv, acc[8 * j + 7] * inv));
    if ((tid & 7) == 0)
      p.lse[(long long)r * p.num_heads + h_abs] =
          (M == -INFINITY || Lsum <= 0.f) ? -INFINITY : (M + log2f(Lsum)) * kLn2;
  }
}

}  // namespace

int mla_max_tokens_per_split() { return MlaSmem::kMaxIds; }

cudaError_t launch_sparse_mla(const MlaLaunch& p, cudaStream_t stream) {
  if (p.num_rows == 0) return cudaSuccess;
  auto kern = p.kv_fp8 ? sparse_mla_kernel<true> : sparse_mla_kernel<false>;
  const int smem_bytes = p.kv_fp8 ? MlaSmem8::kBytes : MlaSmem::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.head_groups, p.num_rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of a (row, head group)
  attr[0].val.clusterDim.x = (unsigned)p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.splits <= kMaxClusterSplits ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
