// msa_internal.cuh -- shared device helpers and launch interfaces of libmsa.
//
// Blackwell (sm_103a) building blocks written as inline PTX: mbarriers,
// 1-D bulk async copies (the TMA bulk engine), bounded waits, warp MMA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

namespace msa {

constexpr int kBlock = 128;  // tokens per index block == tokens per KV page
constexpr int kPage16 = 16;  // tokens per page of the attention view
constexpr int kHeadDim = 128;
constexpr int kMaxHeads = 16;
constexpr int kMaxReqs = 4096;
constexpr int kMaxBlocksPerRow = 16384;
// requests with at least this many query rows are scored on the tensor cores
constexpr int kTcMinRows = 64;
// ... and, in the fused decode with bf16 KV, attend on the tensor cores too
// (block-major prefill attention); list entries pack a row and a slot < 256
constexpr int kPrefillMinRows = 64;
constexpr int kPrefillMaxTopk = 128;
constexpr int kMaxTopk = 2048;
// at most this many page-16 entries per attention split (<= 32 per warp)
constexpr int kMaxSplitEntries = 128;
// the splits of a row merge inside one thread-block cluster when there are at
// most this many (the portable cluster size); more merge through scratch
// partials finished by the last-arriving CTA
constexpr int kMaxClusterSplits = 8;

// Attention launch shape: stages of each warp's copy ring and the CTAs per SM
// the grid is sized for (compile-time, so that launch-shape sweeps can build
// variants with -D; the defaults are the measured choice).
#ifndef MSA_ATTN_STAGES_FP8
#define MSA_ATTN_STAGES_FP8 4
#endif
#ifndef MSA_ATTN_STAGES_BF16
#define MSA_ATTN_STAGES_BF16 3
#endif
#ifndef MSA_ATTN_CTAS_FP8
#define MSA_ATTN_CTAS_FP8 2
#endif
#ifndef MSA_ATTN_CTAS_BF16
#define MSA_ATTN_CTAS_BF16 2
#endif
// sparse MLA: the grid is sized for this many CTAs per SM (2 resident)
#ifndef MSA_MLA_CTAS
#define MSA_MLA_CTAS 2
#endif
// bf16 index keys: scored on CUDA-core FMAs (0) or on warp MMA (1)
#ifndef MSA_SCORE_BF16_KIND
#define MSA_SCORE_BF16_KIND 0
#endif
// bounded waits: a wait that has not completed after this long gives up
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s

// partial (m, l, acc) record of one attention split: m[16], l[16], acc[16][128]
constexpr int kPartFloats = 2 * kMaxHeads + kMaxHeads * kHeadDim;

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// make mbarrier initialisation visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One test of the phase (the hardware may briefly suspend the thread while
// the phase is incomplete).  A longer suspend-time hint was measured: no gain
// for the streaming kernels and a slower single-thread MMA issuer.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// limit_ns (kWaitNs unless a caller passes a limit) and returns false (the
// caller records MSA_DEV_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (tx bytes).
// src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled tensor copy global -> shared (box of the map at x, y), completion
// on `bar`.  x times the element size is a multiple of 16 bytes; the box
// lies inside the tensor; dst is 1024-byte aligned for 128-byte swizzle.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ---- thread-block clusters: barrier (release / acquire) and distributed
// shared-memory loads
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// the address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_dsmem_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p))
               : "memory");
  return v;
}

// bf16 pair (lo, hi halves of a 32-bit word) -> two fp32 (exact)
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// two OCP e4m3 codes (lo byte -> lo half) -> f16x2 (exact conversion)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t out;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(v));
  return out;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t out;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(out) : "r"(a), "r"(b), "r"(sel));
  return out;
}

// D = A(16x16, row) * B(16x8, col) + D; bf16 or f16 operands, fp32 accumulate
template <bool kF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Orderable unsigned key of an fp32 score: a larger score gives a larger
// key; -0 and +0 share a key; NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;
  const uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// --------------------------------------------------- batch geometry checks

// Request q's lengths.  Returns 0 if usable, else MSA_DEV_BAD_LEN or
// MSA_DEV_MALFORMED; *nb = ceil(seq_len/128) when usable.
__device__ __forceinline__ uint32_t request_lengths(const msa_batch& b, int q, int* q_begin,
                                                    int* q_len, int* ctx, int* nb) {
  const int c0 = b.cu_seqlens_q[q], c1 = b.cu_seqlens_q[q + 1];
  const int slen = b.cu_seqlens_k[q + 1] - b.cu_seqlens_k[q];
  *q_begin = c0;
  *q_len = c1 - c0;
  *ctx = b.context_lens[q];
  *nb = 0;
  if (slen < *q_len || *ctx < 0 || (long long)slen > (long long)kBlock * b.bt_stride ||
      *q_len < b.min_q_len)
    return MSA_DEV_MALFORMED;
  if (*ctx + *q_len != slen) return MSA_DEV_BAD_LEN;
  *nb = (slen + kBlock - 1) / kBlock;
  return 0u;
}

// ------------------------------------------------------- launch interfaces

struct ScoreLaunch {
  msa_batch batch;
  const uint16_t* idx_q;
  const uint8_t* idx_k;
  int index_heads, index_dim;
  float* scores;
  int score_stride;
  uint32_t* status;
  int tc_min_rows;  // > 0: requests with q_len >= this are left to the tensor-core kernel
  int idx_fp8;              // index keys are OCP e4m3 codes
  const float* idx_scale;   // FP8: per-token scales [P, 128, Hi], or null (1)
  int report_status;        // tensor-core kernel: report the batch's status bits (the
                            // CUDA-core kernel, which otherwise does, is not launched)
};

struct TopkLaunch {
  msa_batch batch;
  const float* scores;
  int score_stride;
  int topk;
  int32_t* topk_idx;
  int32_t* tbl;
  int tbl_stride;
  int32_t* sparse_len;
  uint32_t* attn_counters;  // zeroed per row when non-null (fused path)
  uint32_t* status;
  // Prefill routing (fused path only; null pointers when off).  Rows of
  // requests with at least kPrefillMinRows rows get route[r] = q + 1 (others
  // 0), and each selected (row, slot i, block b) is appended as r << 8 | i to
  // the request's list of block b: pf_counts[q0 * bt_stride / 64 + b] counts
  // the entries of pf_lists[q0 * bt_stride + b * q_len ...] (q0 = the
  // request's first row).  The counts start at zero (msa_decode clears them
  // on the stream before the top-k kernel).
  int32_t* route;
  int32_t* pf_counts;
  int32_t* pf_lists;
};

struct AttnLaunch {
  const uint16_t* q;
  int num_rows, num_heads;
  const uint8_t* k;
  const uint8_t* v;
  int kv_fp8;
  long long num_pages16;
  int scale_mode;
  const float* k_scale;
  const float* v_scale;
  const float* sinks;
  float softmax_scale;
  const int32_t* tbl;
  int tbl_stride;
  const int32_t* sparse_len;
  uint16_t* out;
  float* lse;
  float* partials;
  uint32_t* counters;
  int splits;
  int pages_per_split;  // page-16 entries per split
  uint32_t* status;
  const int32_t* route;  // fused path: rows with route[r] != 0 belong to the prefill path
};

cudaError_t launch_index_score(const ScoreLaunch& p, cudaStream_t stream);
// Host: 2-D tensor map [rows][inner] (row pitch row_stride_bytes) with
// box_inner x box_rows boxes and 128-byte swizzle; false if the driver entry
// point is missing or the encoder rejects the shape.
bool tensor_maps_available();
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, long long inner,
                   long long rows, long long row_stride_bytes, int box_inner, int box_rows);
cudaError_t launch_index_score_tc(const ScoreLaunch& p, cudaStream_t stream);
bool tc_score_supported(int index_heads, int index_dim);
struct KvInsertLaunch {
  msa_batch batch;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const uint16_t* idx_new;
  int num_kv_heads, index_heads, index_dim;
  uint8_t* k_cache;
  uint8_t* v_cache;
  uint16_t* idx_k_cache;
  int kv_fp8, scale_mode;
  float* k_scale;
  float* v_scale;
  int skip_index;
  int idx_fp8;        // index cache of e4m3 codes
  float* idx_scale;   // FP8 index: per-token scales written here, or null (scale 1)
  uint32_t* status;
};

cudaError_t launch_kv_insert(const KvInsertLaunch& p, cudaStream_t stream);

struct MlaLaunch {
  const uint16_t* q;        // [num_rows, num_heads, 576] bf16
  const uint16_t* kv;       // [num_tokens, 576] bf16
  long long num_tokens;
  const int32_t* indptr;    // [num_rows + 1]
  const int32_t* indices;
  int num_rows, num_heads, head_groups;  // head_groups = ceil(num_heads / 16)
  int max_tokens;           // bound on a row's count (longer rows are refused)
  int splits, tokens_per_split;
  const float* sinks;
  float softmax_scale;
  uint16_t* out;            // [num_rows, num_heads, 512] bf16
  float* lse;
  float* partials;          // [num_rows, head_groups, splits, 16, 516] fp32
  uint32_t* counters;       // [num_rows, head_groups], zero between calls
  uint32_t* status;
  int kv_fp8, q_fp8;        // e4m3 codes in kv (then q may be e4m3 or bf16)
  const float* q_scale;     // fp32 [1] when q_fp8
  const float* kv_scale;    // fp32 [1] when kv_fp8
};

cudaError_t launch_sparse_mla(const MlaLaunch& p, cudaStream_t stream);

// Block-major attention for the rows of prefill requests (fused decode,
// bf16 KV, no per-token scales): plan -> attention -> merge.  Uses the lists
// the top-k kernel appended (see TopkLaunch) and scratch in the workspace.
struct PrefillLaunch {
  msa_batch batch;
  const uint16_t* q;      // [N, hq, 128] bf16
  int num_heads;
  const uint16_t* k;      // K / V pools [P, 128, 1, 128] bf16
  const uint16_t* v;
  const float* k_scale;   // SCALAR mode: fp32 [1] each, else null
  const float* v_scale;
  const float* sinks;
  float softmax_scale;
  int topk;
  const int32_t* topk_idx;  // [N, topk]
  const int32_t* route;     // [N]
  const int32_t* pf_counts; // list counts (msa_decode clears them before the top-k)
  const int32_t* pf_lists;
  // plan: header [0] = items, [1] = chunks, [2] = estimated cost; routed
  // requests (q, first candidate); items, their first chunks and the
  // exclusive prefix of their costs (entry [items] = the totals)
  int32_t* plan_hdr;
  int32_t* plan_req_q;
  int32_t* plan_req_item;
  int4* item_rec;       // per item: list base, rows, position of row 0 (pos = r + z), block
  int2* item_kv;        // per item: page, tokens of the block that exist
  int32_t* item_chunk;
  int32_t* item_cost;
  int max_routed_reqs;      // capacity of plan_req_*
  int finish_unrouted;      // no decode attention runs: the merge writes unrouted rows
                            // (all poisoned) as empty rows
  int max_items;            // capacity of item_*
  uint16_t* part_o;         // [N, topk, 16 dim chunks, 16 heads, 8 dims] bf16, sum p v
  float2* part_ml;          // [N, topk, 16] (max, sum of p), log2 units
  uint16_t* out;            // [N, hq, 128] bf16
  float* lse;               // [N, hq]
  uint32_t* status;
};

cudaError_t launch_prefill_attn(const PrefillLaunch& p, cudaStream_t stream);
bool prefill_attn_available();
int mla_max_tokens_per_split();

// `programmatic`: the kernel may start while the previous kernel on the
// stream finishes (programmatic dependent launch); it waits for that kernel's
// results on the device before reading them.
cudaError_t launch_topk_table(const TopkLaunch& p, cudaStream_t stream, bool programmatic);
cudaError_t launch_sparse_attn(const AttnLaunch& p, cudaStream_t stream, bool programmatic);

// Step 4 behind its entry points (api.cu).  attn_prepare validates the
// arguments (nothing is launched; *splits = 0 when there are no rows) and
// picks the work split; attn_scratch_need is the scratch that split uses:
// per-row merge counters, plus (m, l, acc) partials when a row has more
// splits than one cluster merges; attn_run launches on that scratch (the
// counters must be zero, and the kernel leaves them zero).
msa_status attn_prepare(const msa_attn_args* attn, const int32_t* sparse_tbl, int tbl_stride,
                        const int32_t* sparse_len, const uint32_t* dev_status, int* pps,
                        int* splits);
size_t attn_scratch_need(int num_rows, int splits);
msa_status attn_run(const msa_attn_args* attn, const int32_t* sparse_tbl, int tbl_stride,
                    const int32_t* sparse_len, void* scratch, int pps, int splits,
                    uint32_t* dev_status, cudaStream_t stream);

int device_sm_count();

}  // namespace msa
