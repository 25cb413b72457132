// sparse_attn.cu -- step 4: GQA flash-decode over the tokens a page-16 sparse
// table addresses, with FP8 dequant scales, an optional per-head sink and a
// natural-log LSE.
//
// Definitions: "Add ROCm AITER sparse paged attention for MiniMax-M3" (vLLM PR
// 47287), "Implementation breakdown" items 2-3 (k_scale / v_scale, scalar or
// per_token_head; page-16 view of the page-128 cache); "Attention sinks for
// ROCm AITER sparse MLA" (vLLM PR 54404), "Features and motivation" (learnable
// sinks; empty rows must not produce NaN) and "Key source snippets" (split-KV
// decode returning a natural-log LSE, which every split count must write).
//
// GB300 design.  One KV head serves up to 16 query heads, so a row's heads x
// 8 tokens form a real m16n8k16 tensor-core tile: S = Q K^T and O += P V run
// on warp MMA with fp32 accumulation (the M = heads = 16 tile is below the
// 64/128-row minimum of tcgen05, and the path is HBM-bound).  The row's
// tokens are split across CTAs (grid = splits x rows, sized from the SM
// count); each warp streams its page-16 K and V slabs (2 KB each for FP8,
// contiguous in the pools) into a private shared-memory ring -- FP8 slabs by
// 2-D tensor copies with the 128-byte swizzle, so that the fragment reads of
// every phase hit 32 distinct banks, bf16 slabs by 1-D bulk copies -- and
// converts FP8 to f16 in registers (exact), applies per-token k scales to the
// fp32 logits and folds per-token v scales into P.  The queries sit in
// shared memory in the MMA's k-slot order and are read with ldmatrix.  Warps
// merge in shared memory.  2 to 8 splits of a row form one thread-block
// cluster and merge through distributed shared memory, no global round
// trip: with FP8 slabs each CTA pushes its partials into the owners of the
// output chunks (one cluster barrier), with bf16 slabs each CTA pulls its
// share of the outputs from all partials (two barriers); more splits merge
// through (m, l, acc) partials in the workspace, finished by whichever CTA
// of the row arrives last (atomic counter, reset by that CTA).  No spin-wait
// anywhere.  The sink joins the denominator only in the final merge.
#include <string.h>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.f;  // log2 units: unnormalised weights stay <= 256
constexpr int kAccStride = 132;  // padded head stride of the shared-memory merge area
constexpr int kAccWarpFloats = kMaxHeads * kAccStride;  // 2112
// per-CTA partial for the cluster merge, after the warps' merge area:
// acc [16][128], m [16], l [16], poison flag
constexpr int kCPart = kWarps * (kAccWarpFloats + 2 * kMaxHeads) * 4;
constexpr int kCpM = kMaxHeads * kHeadDim, kCpL = kCpM + kMaxHeads, kCpFlag = kCpL + kMaxHeads;
constexpr int kCPartBytes = (kCpFlag + 4) * 4;
// push merge: the 16 heads' outputs form 4 chunks of 4 heads (128 float4);
// chunk q belongs to CTA q % splits, which receives it from every split:
// [slot = q / splits][source split][128 float4], then (m, l) per head, then
// one poison flag per source.  At most 8 (slot, source) pairs for 1..8 splits.
constexpr int kRecvPairs = 8;
constexpr int kRecvF4Bytes = kRecvPairs * 128 * 16;
constexpr int kRecvMlBytes = kRecvPairs * 8 * 4;
constexpr int kRecvFlagBytes = kMaxClusterSplits * 4;

// PUSH: the push merge (a receive area outside the ring) for bf16 K/V too;
// FP8 always pushes
template <bool FP8, bool PUSH = false>
struct AttnCfg {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kSlab = kPage16 * kHeadDim * kElem;  // one page-16 K (or V) slab
  static constexpr int kStages = FP8 ? MSA_ATTN_STAGES_FP8 : MSA_ATTN_STAGES_BF16;
  // rings of the 4 warps: K slabs, then V slabs (each slab 1024-byte aligned,
  // as the 128-byte swizzle of the FP8 tensor copies needs), then scales
  static constexpr int kSlots = kWarps * kStages;
  static constexpr int kRingK = 0;
  static constexpr int kRingV = kSlots * kSlab;
  static constexpr int kRingS = 2 * kSlots * kSlab;
  static constexpr int kRingBytes = kRingS + kSlots * 128;
  static constexpr int kMergeBytes = kWarps * (kAccWarpFloats + 2 * kMaxHeads) * 4;
  static constexpr int kDataBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
  static constexpr int kQBytes = kMaxHeads * kHeadDim * 2;  // the row's queries, bf16
  static constexpr int kQ = kDataBytes;
  static constexpr int kBarOff = kQ + kQBytes;
  // after the barriers: 2 merge flags, then the sinks (log2 units) and the scalar v scale
  static constexpr int kFlagsOff = kBarOff + (kSlots + 1) * 8;
  static constexpr int kSinkOff = kFlagsOff + 16;
  // FP8 cluster merge: the receive area other CTAs of the row push their
  // partials into, never used by this CTA before the merge (outside the ring)
  static constexpr int kRecvOff = (kSinkOff + (kMaxHeads + 1) * 4 + 15) / 16 * 16;
  static constexpr int kRecvBytes =
      (FP8 || PUSH) ? kRecvF4Bytes + kRecvMlBytes + kRecvFlagBytes : 0;
  static constexpr int kSmemBytes = kRecvOff + kRecvBytes + 64;
  static_assert(kCPart + kCPartBytes <= kDataBytes, "cluster partial must fit the ring");
};

// four 8x8 b16 matrices from a shared-memory address; lane l gives the row
// address of matrix l/8, row l%8 and receives (row g, cols 2c, 2c+1) of each
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ int acc_index(int head, int dim) {
  return head * kAccStride + dim + (dim >> 5);
}

// ---- the row's output: sink in the denominator, 1/L (and the scalar v
// scale), bf16 O for dims d0..d0+N of `head`, natural-log LSE
template <int N, int SCALE>
// (sink_s: the sinks in log2 units, then the scalar v scale, staged in
// shared memory at the kernel's start)
__device__ __forceinline__ void finalize_out(const AttnLaunch& p, const float* sink_s, int r,
                                             int head, int d0, float (&acc)[N], float M,
                                             float Lsum, bool write_lse) {
  if (p.sinks) {
    const float sink2 = sink_s[head];
    const float Mn = fmaxf(M, sink2);
    Lsum = (M == -INFINITY ? 0.f : Lsum * exp2f(M - Mn)) + exp2f(sink2 - Mn);
    const float f = M == -INFINITY ? 0.f : exp2f(M - Mn);
#pragma unroll
    for (int j = 0; j < N; ++j) acc[j] *= f;
    M = Mn;
  }
  float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
  if constexpr (SCALE == MSA_SCALE_SCALAR) inv *= sink_s[kMaxHeads];
  uint32_t packed[N / 2];
#pragma unroll
  for (int j = 0; j < N / 2; ++j) packed[j] = pack_bf16x2(acc[2 * j] * inv, acc[2 * j + 1] * inv);
  uint16_t* o = p.out + ((long long)r * p.num_heads + head) * kHeadDim + d0;
  if constexpr (N == 16) {
    reinterpret_cast<uint4*>(o)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    reinterpret_cast<uint4*>(o)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  } else {
    *reinterpret_cast<uint2*>(o) = make_uint2(packed[0], packed[1]);
  }
  if (write_lse)
    p.lse[(long long)r * p.num_heads + head] =
        (M == -INFINITY || Lsum <= 0.f) ? -INFINITY : (M + log2f(Lsum)) * kLn2;
}

template <bool FP8, int SCALE, bool CL, bool PUSH = false>
__global__ void __launch_bounds__(kThreads, FP8 ? MSA_ATTN_CTAS_FP8 : (PUSH ? 1 : MSA_ATTN_CTAS_BF16))
    sparse_attn_kernel(const AttnLaunch p, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  using C = AttnCfg<FP8, PUSH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* qbar = bars + kWarps * C::kStages;
  int* flags = reinterpret_cast<int*>(smem + C::kFlagsOff);
  float* sink_s = reinterpret_cast<float*>(smem + C::kSinkOff);
  const uint8_t* q_s = smem + C::kQ;

  const int split = blockIdx.x, r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const long long tbl_row = (long long)r * p.tbl_stride;
  const unsigned full = 0xffffffffu;

  // ---- prologue independent of the previous kernel: the row's queries
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t q_bytes = (uint32_t)p.num_heads * kHeadDim * 2;
  if (tid == 0) {
    mbar_init(qbar, 1);
    for (int s = 0; s < kWarps * C::kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    if (!p.route) {  // (with a prefill path the row may not be ours: copy after the wait)
      mbar_arrive_expect_tx(qbar, q_bytes);
      bulk_g2s(smem + C::kQ, p.q + (long long)r * p.num_heads * kHeadDim, q_bytes, qbar);
    }
  }
  // the sinks and the scalar v scale are inputs of the call: read them now,
  // so that no global load sits on the final merge's path
  if (tid < kMaxHeads) sink_s[tid] = (p.sinks && tid < p.num_heads) ? __ldg(p.sinks + tid) * kLog2e : 0.f;
  if (tid == kMaxHeads)
    sink_s[kMaxHeads] = SCALE == MSA_SCALE_SCALAR ? __ldg(p.v_scale) : 1.f;
  // sparse tables and lengths come from the previous kernel on the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (p.route) {
    // a row of a prefill request is written by the block-major prefill
    // attention: leave (uniform over the CTA and over the row's cluster)
    if (p.route[r] != 0) return;
    if (tid == 0) {
      mbar_arrive_expect_tx(qbar, q_bytes);
      bulk_g2s(smem + C::kQ, p.q + (long long)r * p.num_heads * kHeadDim, q_bytes, qbar);
    }
  }

  // this warp's page-16 entries are split*pps + warp + 4*i, one per lane; the
  // table load does not depend on the length, so both are in flight together
  const int e_begin = split * p.pages_per_split;
  const int e_lane = e_begin + warp + kWarps * lane;
  const bool lane_in_split = kWarps * lane + warp < p.pages_per_split && e_lane < p.tbl_stride;
  long long my_e = lane_in_split ? (long long)p.tbl[tbl_row + e_lane] : 0ll;
  int len = p.sparse_len[r];
  const bool len_bad = len < 0 || (long long)len > (long long)kPage16 * p.tbl_stride;
  const int nent = len_bad ? 0 : (len + kPage16 - 1) / kPage16;
  const int n_active = max(1, (nent + p.pages_per_split - 1) / p.pages_per_split);
  const bool active = split < n_active;
  const int e_end = min(nent, e_begin + p.pages_per_split);
  int n_my = active && e_end > e_begin + warp ? (e_end - (e_begin + warp) + kWarps - 1) / kWarps : 0;
  bool entry_bad = false;
  if (lane < n_my) entry_bad = my_e < 0 || my_e >= p.num_pages16;
  __syncthreads();  // barrier inits visible to every warp
  const bool cta_bad = __syncthreads_or(entry_bad) != 0;
  if (!CL && !active) {
    // still drain the query copy this CTA issued before leaving (a CTA of a
    // cluster stays: it takes part in the merge with an empty partial)
    if (tid == 0 && !mbar_wait(qbar, 0)) atomicOr(p.status, MSA_DEV_TIMEOUT);
    return;
  }
  if (cta_bad) n_my = 0;  // never copy from an id outside the pool
  const bool single = n_active == 1;
  if (single && (len_bad || cta_bad) && tid == 0) atomicOr(p.status, MSA_DEV_BAD_TABLE);
  const int slot0 = warp * C::kStages;  // this warp's first ring slot
  uint64_t* wbar = bars + slot0;

  auto issue = [&](int i, long long e) {  // lane 0 only
    const int st = i % C::kStages;
    uint8_t* kd = smem + C::kRingK + (slot0 + st) * C::kSlab;
    uint8_t* vd = smem + C::kRingV + (slot0 + st) * C::kSlab;
    const uint32_t bytes = 2 * C::kSlab + (SCALE == MSA_SCALE_PER_TOKEN_HEAD ? 128 : 0);
    mbar_arrive_expect_tx(&wbar[st], bytes);
    if constexpr (FP8) {
      // 16 rows x 128 B boxes, 128-byte swizzled: the fragment reads below
      // then hit 32 distinct banks per phase
      tma_load_2d(kd, &kmap, 0, (int)(e * kPage16), &wbar[st]);
      tma_load_2d(vd, &vmap, 0, (int)(e * kPage16), &wbar[st]);
    } else {
      bulk_g2s(kd, p.k + e * C::kSlab, C::kSlab, &wbar[st]);
      bulk_g2s(vd, p.v + e * C::kSlab, C::kSlab, &wbar[st]);
    }
    if constexpr (SCALE == MSA_SCALE_PER_TOKEN_HEAD) {
      uint8_t* sd = smem + C::kRingS + (slot0 + st) * 128;
      bulk_g2s(sd, p.k_scale + e * kPage16, 64, &wbar[st]);
      bulk_g2s(sd + 64, p.v_scale + e * kPage16, 64, &wbar[st]);
    }
  };
  for (int i = 0; i < min(n_my, C::kStages); ++i) {
    const long long e = __shfl_sync(full, my_e, i);
    if (lane == 0) issue(i, e);
  }
  const bool q_ok = __syncthreads_and(mbar_wait(qbar, 0)) != 0;  // CTA-uniform decision
  if (!q_ok) {
    if (tid == 0) atomicOr(p.status, MSA_DEV_TIMEOUT);
    n_my = 0;
  }

  // ---- queries into the A-operand order of S = Q K^T, in place: k-step kk,
  // slots (2c, 2c+1) <-> dims 32c+4kk+{0,1} and (2c+8, 2c+9) <-> +{2,3}, so
  // that one 16-byte read per lane covers four k-steps of a key row.  The
  // shared copy is [kk][slot half][head][8 slots] (2-byte elements, f16 for
  // FP8 keys), which makes every ldmatrix phase read 128 contiguous bytes.
  if (q_ok) {
    uint32_t qw[2][4];
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {  // chunks tid and tid + 128: head t/16, dims 8(t%16)..+8
      const int t = tid + kThreads * k2, h = t >> 4;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (h < p.num_heads) v = lds128(q_s + 16 * t);
      qw[k2][0] = v.x; qw[k2][1] = v.y; qw[k2][2] = v.z; qw[k2][3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int t = tid + kThreads * k2, h = t >> 4, q = t & 15;
#pragma unroll
      for (int w = 0; w < 4; ++w) {  // dims 8q+2w, +1: c = q/4, kk = 2(q%4) + w/2, half w%2
        uint32_t x = qw[k2][w];
        if constexpr (FP8) x = pack_f16x2(bf16lo(x), bf16hi(x));  // f16 operands for FP8 keys
        const int kk = 2 * (q & 3) + (w >> 1);
        *reinterpret_cast<uint32_t*>(smem + C::kQ + kk * 512 + (w & 1) * 256 + h * 16 + 4 * (q >> 2)) = x;
      }
    }
  }
  __syncthreads();
  // ldmatrix row address of this lane: matrix lane/8 = (half lane/16, heads 8*((lane/8)&1)..)
  const uint32_t qa_addr = smem_u32(smem + C::kQ) + (lane >> 4) * 256 + (lane & 15) * 16;
  float scale2 = p.softmax_scale * kLog2e;  // logits in log2 units
  if constexpr (SCALE == MSA_SCALE_SCALAR) scale2 *= __ldg(p.k_scale);

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  // 128-byte swizzle of the FP8 slabs: 16-byte chunk j of row t sits at chunk
  // j ^ (t % 8).  K rows of this lane are g (mod 8); V rows are vt[a].
  const int koff0 = 16 * ((2 * c) ^ g), koff1 = 16 * ((2 * c + 1) ^ g);
  const int vt[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
  int voff[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) voff[a] = vt[a] * kHeadDim + 16 * (g ^ (vt[a] & 7));
  bool timed_out = false;
  int issued = min(n_my, C::kStages);  // entries whose copies this warp has issued
  int stopped = n_my;                  // first entry not consumed
  // Two page-16 slabs (A = warp entry i, B = entry i+1) per iteration: four
  // independent S chains, one softmax pass over 32 tokens and 32 P.V MMAs,
  // which doubles the independent work the warp has in flight.  A missing B
  // (odd count) reads A's stage and is masked to zero weight.
  for (int i = 0; i < n_my; i += 2) {
    const bool has_b = i + 1 < n_my;
    const int st_a = i % C::kStages, st_b = has_b ? (i + 1) % C::kStages : st_a;
    // warp-uniform: the MMAs below need the whole warp
    bool ready = mbar_wait(&wbar[st_a], (i / C::kStages) & 1);
    if (has_b) ready = ready && mbar_wait(&wbar[st_b], ((i + 1) / C::kStages) & 1);
    if (!__all_sync(full, ready)) {
      timed_out = true;
      stopped = i;
      break;
    }
    const int sl_a = slot0 + st_a, sl_b = slot0 + st_b;
    const uint8_t* kst[2] = {smem + C::kRingK + sl_a * C::kSlab, smem + C::kRingK + sl_b * C::kSlab};
    const uint8_t* vst[2] = {smem + C::kRingV + sl_a * C::kSlab, smem + C::kRingV + sl_b * C::kSlab};
    const float* sst[2] = {reinterpret_cast<const float*>(smem + C::kRingS + sl_a * 128),
                           reinterpret_cast<const float*>(smem + C::kRingS + sl_b * 128)};
    const int tok_a = (e_begin + warp + kWarps * i) * kPage16;  // row token index of A's slot 0
    const int nvalid[2] = {min(kPage16, len - tok_a),
                           has_b ? min(kPage16, len - tok_a - kWarps * kPage16) : 0};

    // ---- S = Q K^T: n-tile u = 2*slab + half holds tokens 8*half + g of the slab
    float s[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) s[u][0] = s[u][1] = s[u][2] = s[u][3] = 0.f;
    if constexpr (FP8) {
      uint32_t kw[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // row 8(u&1)+g, 16-byte chunks 2c and 2c+1 at their swizzled places
        const uint8_t* krow = kst[u >> 1] + (8 * (u & 1) + g) * kHeadDim;
        const uint4 k0 = lds128(krow + koff0), k1 = lds128(krow + koff1);
        kw[u][0] = k0.x; kw[u][1] = k0.y; kw[u][2] = k0.z; kw[u][3] = k0.w;
        kw[u][4] = k1.x; kw[u][5] = k1.y; kw[u][6] = k1.z; kw[u][7] = k1.w;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t qa[4];
        ldsm_x4(qa_addr + kk * 512u, qa);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mma16816<true>(s[u], qa, e4m3x2_to_f16x2((uint16_t)(kw[u][kk] & 0xffffu)),
                         e4m3x2_to_f16x2((uint16_t)(kw[u][kk] >> 16)));
      }
    } else {
      uint32_t kw[4][16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint8_t* krow = kst[u >> 1] + ((8 * (u & 1) + g) * kHeadDim + 32 * c) * 2;
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4) {
          const uint4 v = lds128(krow + 16 * h4);
          kw[u][4 * h4] = v.x; kw[u][4 * h4 + 1] = v.y; kw[u][4 * h4 + 2] = v.z; kw[u][4 * h4 + 3] = v.w;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t qa[4];
        ldsm_x4(qa_addr + kk * 512u, qa);
#pragma unroll
        for (int u = 0; u < 4; ++u) mma16816<false>(s[u], qa, kw[u][2 * kk], kw[u][2 * kk + 1]);
      }
    }
    // ---- scale, mask, online softmax over the 32 tokens (rows g and g+8)
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 8 * (u & 1) + 2 * c + (e & 1);
        float v = s[u][e] * scale2;
        if constexpr (SCALE == MSA_SCALE_PER_TOKEN_HEAD)
          v *= sst[u >> 1][t];
        s[u][e] = t < nvalid[u >> 1] ? v : -INFINITY;
      }
    float mx[2];
    mx[0] = fmaxf(fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])),
                  fmaxf(fmaxf(s[2][0], s[2][1]), fmaxf(s[3][0], s[3][1])));
    mx[1] = fmaxf(fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3])),
                  fmaxf(fmaxf(s[2][2], s[2][3]), fmaxf(s[3][2], s[3][3])));
    // Lazy rescaling: the reference max m_run only moves when a pair's max
    // exceeds it by more than kRescaleSlack (log2 units), so p <= 2^slack and
    // the accumulators are rescaled only on those (rare) iterations.
    bool move[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
      move[hh] = mx[hh] > m_run[hh] + kRescaleSlack;
    }
    if (__any_sync(0xffffffffu, move[0] || move[1])) {
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
    float pr[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[u][e] = exp2f(s[u][e] - base[e >> 1]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      l_run[0] += pr[u][0] + pr[u][1];
      l_run[1] += pr[u][2] + pr[u][3];
    }
    if constexpr (SCALE == MSA_SCALE_PER_TOKEN_HEAD) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pr[u][e] *= sst[u >> 1][kPage16 + 8 * (u & 1) + 2 * c + (e & 1)];
    }
    // P as the A operand of O += P V, per slab: tokens (2c, 2c+1) from its
    // first n-tile, (2c+8, 2c+9) from its second
    uint32_t pa[2][4];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl) {
      if constexpr (FP8) {
        pa[sl][0] = pack_f16x2(pr[2 * sl][0], pr[2 * sl][1]);
        pa[sl][1] = pack_f16x2(pr[2 * sl][2], pr[2 * sl][3]);
        pa[sl][2] = pack_f16x2(pr[2 * sl + 1][0], pr[2 * sl + 1][1]);
        pa[sl][3] = pack_f16x2(pr[2 * sl + 1][2], pr[2 * sl + 1][3]);
      } else {
        pa[sl][0] = pack_bf16x2(pr[2 * sl][0], pr[2 * sl][1]);
        pa[sl][1] = pack_bf16x2(pr[2 * sl][2], pr[2 * sl][3]);
        pa[sl][2] = pack_bf16x2(pr[2 * sl + 1][0], pr[2 * sl + 1][1]);
        pa[sl][3] = pack_bf16x2(pr[2 * sl + 1][2], pr[2 * sl + 1][3]);
      }
    }
    // ---- V fragments: tokens {2c, 2c+1, 2c+8, 2c+9}, dims 16g + j for n-tile j
    if constexpr (FP8) {
      uint32_t vw[2][4][4];
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const uint4 v = lds128(vst[sl] + voff[a]);
          vw[sl][a][0] = v.x; vw[sl][a][1] = v.y; vw[sl][a][2] = v.z; vw[sl][a][3] = v.w;
        }
        if (nvalid[sl] < kPage16) {  // never let garbage past the end reach P V
#pragma unroll
          for (int a = 0; a < 4; ++a)
            if (vt[a] >= nvalid[sl]) vw[sl][a][0] = vw[sl][a][1] = vw[sl][a][2] = vw[sl][a][3] = 0u;
        }
      }
#pragma unroll
      for (int j2 = 0; j2 < 8; ++j2) {  // n-tiles 2*j2, 2*j2+1
        const int wi = j2 >> 1, by = 2 * (j2 & 1);
        const uint32_t sel = (uint32_t)(by | ((4 + by) << 4) | ((by + 1) << 8) | ((5 + by) << 12));
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
          const uint32_t lo = prmt(vw[sl][0][wi], vw[sl][1][wi], sel);  // tokens 2c, 2c+1
          const uint32_t hi = prmt(vw[sl][2][wi], vw[sl][3][wi], sel);  // tokens 2c+8, 2c+9
          mma16816<true>(o[2 * j2], pa[sl], e4m3x2_to_f16x2((uint16_t)(lo & 0xffffu)),
                         e4m3x2_to_f16x2((uint16_t)(hi & 0xffffu)));
          mma16816<true>(o[2 * j2 + 1], pa[sl], e4m3x2_to_f16x2((uint16_t)(lo >> 16)),
                         e4m3x2_to_f16x2((uint16_t)(hi >> 16)));
        }
      }
    } else {
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        uint32_t vw[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const uint8_t* src = vst[sl] + (vt[a] * kHeadDim + 16 * g) * 2;
          const uint4 v0 = lds128(src), v1 = lds128(src + 16);
          vw[a][0] = v0.x; vw[a][1] = v0.y; vw[a][2] = v0.z; vw[a][3] = v0.w;
          vw[a][4] = v1.x; vw[a][5] = v1.y; vw[a][6] = v1.z; vw[a][7] = v1.w;
        }
        if (nvalid[sl] < kPage16) {  // never let garbage past the end reach P V
#pragma unroll
          for (int a = 0; a < 4; ++a)
            if (vt[a] >= nvalid[sl])
#pragma unroll
              for (int x = 0; x < 8; ++x) vw[a][x] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
          const uint32_t b0 = prmt(vw[0][j >> 1], vw[1][j >> 1], sel);
          const uint32_t b1 = prmt(vw[2][j >> 1], vw[3][j >> 1], sel);
          mma16816<false>(o[j], pa[sl], b0, b1);
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int d = 0; d < 2; ++d) {
      const int nxt = i + d + C::kStages;
      if (nxt < n_my) {
        const long long e = __shfl_sync(full, my_e, nxt);
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(nxt, e);
        }
        issued = nxt + 1;
      }
    }
  }
  if (timed_out && lane == 0) {
    atomicOr(p.status, MSA_DEV_TIMEOUT);
    // let this warp's copies still in flight land (bounded) before the ring
    // is reused for the merge
    for (int j = stopped; j < issued; ++j) mbar_wait(&wbar[j % C::kStages], (j / C::kStages) & 1);
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
  }

  // ---- merge the 4 warps in shared memory (reusing the ring)
  __syncthreads();
  float* acc_s = reinterpret_cast<float*>(smem);
  float* ml_s = acc_s + kWarps * kAccWarpFloats;  // [warp][m 16 | l 16]
  {
    // acc_index(g, 32c + j) = g*132 + 33c + j for j < 32: one base, immediate offsets
    float* aw = acc_s + warp * kAccWarpFloats + acc_index(g, 32 * c);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      aw[j] = o[j][0];
      aw[16 + j] = o[j][1];
      aw[8 * kAccStride + j] = o[j][2];
      aw[8 * kAccStride + 16 + j] = o[j][3];
    }
    if (c == 0) {
      ml_s[warp * 32 + g] = m_run[0];
      ml_s[warp * 32 + g + 8] = m_run[1];
      ml_s[warp * 32 + 16 + g] = l_run[0];
      ml_s[warp * 32 + 16 + g + 8] = l_run[1];
    }
  }
  __syncthreads();
  // thread t: head t/8, dims 16*(t%8) .. +16
  const int head = tid >> 3, d0 = 16 * (tid & 7);
  float mh = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) mh = fmaxf(mh, ml_s[w * 32 + head]);
  float lh = 0.f, acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float mw = ml_s[w * 32 + head];
    const float f = mw == -INFINITY ? 0.f : exp2f(mw - mh);
    lh += f * ml_s[w * 32 + 16 + head];
    const float* ar = acc_s + w * kAccWarpFloats + acc_index(head, d0);  // d0..d0+15: same 32-block
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] += f * ar[j];
  }

  if constexpr (CL && (FP8 || PUSH)) {
    // ---- the row's splits form one cluster.  Each CTA pushes its partial
    // of every 4-head chunk straight into the shared memory of the chunk's
    // owner (asynchronous remote stores), one cluster barrier makes all of
    // them visible, and each owner merges its chunks from its own memory:
    // no remote load on the path and no second barrier.
    const uint32_t recv = smem_u32(smem + C::kRecvOff);
    const uint32_t recv_ml = recv + kRecvF4Bytes, recv_fl = recv_ml + kRecvMlBytes;
    {
      const int q = head >> 2, owner = q % p.splits, slot = q / p.splits;
      const int pair = slot * p.splits + split;
      const uint32_t dst = mapa_shared(recv, (uint32_t)owner) +
                           16u * (pair * 128 + (head & 3) * 32 + (d0 >> 2));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_dsmem_f4(dst + 16u * j, make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
      if ((tid & 7) == 0) {
        const uint32_t ml = mapa_shared(recv_ml, (uint32_t)owner) + 4u * (pair * 8 + (head & 3) * 2);
        st_dsmem_f32(ml, mh);
        st_dsmem_f32(ml + 4u, lh);
      }
      if (tid < p.splits)  // this split's poison flag, to every CTA of the row
        st_dsmem_s32(mapa_shared(recv_fl, (uint32_t)tid) + 4u * split, (len_bad || cta_bad) ? 1 : 0);
    }
    cluster_sync();  // every push of the row has landed
    const int* fl = reinterpret_cast<const int*>(smem + C::kRecvOff + kRecvF4Bytes + kRecvMlBytes);
    const bool poisoned = __any_sync(full, lane < p.splits && fl[lane] != 0);
    if (poisoned && split == 0 && tid == 0) atomicOr(p.status, MSA_DEV_BAD_TABLE);
    const float4* rf4 = reinterpret_cast<const float4*>(smem + C::kRecvOff);
    const float* rml = reinterpret_cast<const float*>(smem + C::kRecvOff + kRecvF4Bytes);
    for (int q = split; q < 4; q += p.splits) {
      const int slot = q / p.splits;
      const int h = 4 * q + (tid >> 5), d = 4 * (tid & 31);
      if (h >= p.num_heads) continue;
      float M = -INFINITY, L = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
      if (!poisoned) {
        for (int j = 0; j < p.splits; ++j) M = fmaxf(M, rml[(slot * p.splits + j) * 8 + (h & 3) * 2]);
        for (int j = 0; j < p.splits; ++j) {
          const int pair = slot * p.splits + j;
          const float ms = rml[pair * 8 + (h & 3) * 2];
          if (ms == -INFINITY) continue;
          const float f = exp2f(ms - M);
          L += f * rml[pair * 8 + (h & 3) * 2 + 1];
          const float4 v = rf4[pair * 128 + tid];
          a[0] += f * v.x;
          a[1] += f * v.y;
          a[2] += f * v.z;
          a[3] += f * v.w;
        }
      }
      finalize_out<4, SCALE>(p, sink_s, r, h, d, a, M, L, (tid & 31) == 0);
    }
    return;
  } else if constexpr (CL) {
    // ---- the row's splits form one cluster: each CTA leaves its partial in
    // its own shared memory, then every CTA merges a share of the (head,
    // 4-dim) outputs over all partials through distributed shared memory.
    float* cp = reinterpret_cast<float*>(smem + kCPart);
    float4* c4 = reinterpret_cast<float4*>(cp + head * kHeadDim + d0);
#pragma unroll
    for (int j = 0; j < 4; ++j) c4[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
    if ((tid & 7) == 0) {
      cp[kCpM + head] = mh;
      cp[kCpL + head] = lh;
    }
    if (tid == 0) reinterpret_cast<int*>(cp)[kCpFlag] = (len_bad || cta_bad) ? 1 : 0;
    cluster_sync();  // every partial of the row is written and visible
    const uint32_t cp_addr = smem_u32(cp);
    int fl = 0;
    if (lane < p.splits) fl = ld_dsmem_s32(mapa_shared(cp_addr + 4u * kCpFlag, (uint32_t)lane));
    const bool poisoned = __any_sync(full, fl != 0);  // an id outside the pool empties the row
    if (poisoned && split == 0 && tid == 0) atomicOr(p.status, MSA_DEV_BAD_TABLE);
    for (int i4 = split * kThreads + tid; i4 < kMaxHeads * kHeadDim / 4; i4 += p.splits * kThreads) {
      const int h = i4 >> 5, d = 4 * (i4 & 31);
      if (h >= p.num_heads) break;
      float M = -INFINITY, L = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
      if (!poisoned) {
        float ms[kMaxClusterSplits], ls[kMaxClusterSplits];
        float4 v[kMaxClusterSplits];
#pragma unroll
        for (int j = 0; j < kMaxClusterSplits; ++j) {
          if (j < p.splits) {
            const uint32_t base = mapa_shared(cp_addr, (uint32_t)j);
            ms[j] = ld_dsmem_f32(base + 4u * (kCpM + h));
            ls[j] = ld_dsmem_f32(base + 4u * (kCpL + h));
            v[j] = ld_dsmem_f4(base + 4u * (h * kHeadDim + d));
          }
        }
#pragma unroll
        for (int j = 0; j < kMaxClusterSplits; ++j) M = j < p.splits ? fmaxf(M, ms[j]) : M;
#pragma unroll
        for (int j = 0; j < kMaxClusterSplits; ++j) {
          if (j < p.splits && ms[j] != -INFINITY) {
            const float f = exp2f(ms[j] - M);
            L += f * ls[j];
            a[0] += f * v[j].x;
            a[1] += f * v[j].y;
            a[2] += f * v[j].z;
            a[3] += f * v[j].w;
          }
        }
      }
      finalize_out<4, SCALE>(p, sink_s, r, h, d, a, M, L, (i4 & 31) == 0);
    }
    cluster_sync();  // no CTA leaves while another may still read its partial
    return;
  }

  bool empty_row = single && (len_bad || cta_bad);
  if (!single) {
    // ---- publish this split's partial; the last CTA of the row merges all.
    // A CTA that saw an id outside the pool flags the row in the counter's
    // top bit before counting itself in.
    float* part = p.partials + ((long long)r * p.splits + split) * kPartFloats;
    if ((tid & 7) == 0) {
      part[head] = mh;
      part[kMaxHeads + head] = lh;
    }
    float4* pa4 = reinterpret_cast<float4*>(part + 2 * kMaxHeads + head * kHeadDim + d0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      pa4[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      if (cta_bad) atomicOr(&p.counters[r], 0x80000000u);
      const unsigned old = atomicAdd(&p.counters[r], 1u);
      flags[0] = ((old & 0x7fffffffu) == (unsigned)(n_active - 1));
      flags[1] = ((old | (cta_bad ? 0x80000000u : 0u)) & 0x80000000u) != 0;
    }
    __syncthreads();
    if (!flags[0]) return;
    __threadfence();
    empty_row = flags[1] != 0;
    mh = -INFINITY;
    lh = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
#pragma unroll 4
    for (int sp = 0; sp < n_active; ++sp) {  // online merge, one pass over the partials
      const float* ps = p.partials + ((long long)r * p.splits + sp) * kPartFloats;
      const float ms = __ldcg(ps + head);
      const float ls = __ldcg(ps + kMaxHeads + head);
      const float4* a4 = reinterpret_cast<const float4*>(ps + 2 * kMaxHeads + head * kHeadDim + d0);
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __ldcg(a4 + j);
      const float mn = fmaxf(mh, ms);
      const float fo = mh == -INFINITY ? 0.f : exp2f(mh - mn);
      const float fs = ms == -INFINITY ? 0.f : exp2f(ms - mn);
      lh = lh * fo + ls * fs;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[4 * j] = acc[4 * j] * fo + v[j].x * fs;
        acc[4 * j + 1] = acc[4 * j + 1] * fo + v[j].y * fs;
        acc[4 * j + 2] = acc[4 * j + 2] * fo + v[j].z * fs;
        acc[4 * j + 3] = acc[4 * j + 3] * fo + v[j].w * fs;
      }
      mh = mn;
    }
    if (tid == 0) {
      p.counters[r] = 0;  // ready for the next call / graph replay
      if (empty_row) atomicOr(p.status, MSA_DEV_BAD_TABLE);
    }
  }
  if (empty_row) {  // a poisoned row is an empty row
    mh = -INFINITY;
    lh = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  }
  if (head < p.num_heads) finalize_out<16, SCALE>(p, sink_s, r, head, d0, acc, mh, lh, (tid & 7) == 0);
}

template <bool FP8, int SCALE>
cudaError_t launch_cfg(const AttnLaunch& p, cudaStream_t stream, bool programmatic) {
  // one split needs no merge at all (the single-split path finalises directly)
  const bool cl = p.splits > 1 && p.splits <= kMaxClusterSplits;
  // bf16 K/V: the push merge's receive area fits only at one CTA per SM,
  // which a grid of no more CTAs than SMs leaves anyway
  const bool push = !FP8 && cl && (long long)p.num_rows * p.splits <= device_sm_count();
  auto kern = push ? sparse_attn_kernel<FP8, SCALE, true, true>
                   : cl ? sparse_attn_kernel<FP8, SCALE, true> : sparse_attn_kernel<FP8, SCALE, false>;
  const int smem_bytes = push ? AttnCfg<FP8, true>::kSmemBytes : AttnCfg<FP8>::kSmemBytes;
  CUtensorMap kmap, vmap;
  memset(&kmap, 0, sizeof(kmap));
  memset(&vmap, 0, sizeof(vmap));
  if constexpr (FP8) {
    // the pools as [8P * 16 rows][128 B]; row coordinates must fit an int
    const long long rows = p.num_pages16 * kPage16;
    if (rows > 0x7fffffffll ||
        !encode_map_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.k, kHeadDim, rows, kHeadDim,
                       kHeadDim, kPage16) ||
        !encode_map_2d(&vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.v, kHeadDim, rows, kHeadDim,
                       kHeadDim, kPage16))
      return cudaErrorInvalidValue;
  }
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.num_rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cl) {  // one cluster per row: its splits
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)p.splits;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (programmatic) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p, kmap, vmap);
}

}  // namespace

cudaError_t launch_sparse_attn(const AttnLaunch& p, cudaStream_t stream, bool programmatic) {
  if (p.num_rows == 0) return cudaSuccess;
  if (p.kv_fp8) {
    if (p.scale_mode == MSA_SCALE_NONE) return launch_cfg<true, MSA_SCALE_NONE>(p, stream, programmatic);
    if (p.scale_mode == MSA_SCALE_SCALAR)
      return launch_cfg<true, MSA_SCALE_SCALAR>(p, stream, programmatic);
    return launch_cfg<true, MSA_SCALE_PER_TOKEN_HEAD>(p, stream, programmatic);
  }
  if (p.scale_mode == MSA_SCALE_NONE) return launch_cfg<false, MSA_SCALE_NONE>(p, stream, programmatic);
  if (p.scale_mode == MSA_SCALE_SCALAR)
    return launch_cfg<false, MSA_SCALE_SCALAR>(p, stream, programmatic);
  return launch_cfg<false, MSA_SCALE_PER_TOKEN_HEAD>(p, stream, programmatic);
}

}  // namespace msa
