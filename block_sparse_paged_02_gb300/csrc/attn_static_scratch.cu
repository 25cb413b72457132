// attn_static_scratch.cu -- msa_sparse_paged_attn for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// where cudaMalloc is off limits (it synchronises the whole device and so
// stalls a serving loop mid-step), plug-ins whose host framework owns every
// device byte through its own pool and gives extensions no allocator, or
// embedded runtimes that forbid allocation after start-up.  For them this
// entry point runs the same attention kernel with its split-merge scratch
// (per-row counters and (m, l, acc) partials) taken from one file-scope
// device array of fixed size.  Every GPU that loads the library reserves
// that array until the process exits.
//
// The array is shared by every call in the process: the counters are
// cleared on the stream at the start of each call, and two calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on it and give undefined results.
#include <mutex>

#include "msa_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[MSA_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the array on the current device.  The name
// g_attn_scratch is only a host-side stand-in; a kernel must be given the
// address cudaGetSymbolAddress returns.  Looked up once per device, on the
// first call made with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" msa_status msa_sparse_paged_attn_static(const msa_attn_args* attn,
                                                   const int32_t* sparse_tbl, int32_t tbl_stride,
                                                   const int32_t* sparse_len,
                                                   uint32_t* dev_status, cudaStream_t stream) {
  if (!attn) return MSA_ERR_NULL;
  if (attn->num_rows < 0 || tbl_stride < 1) return MSA_ERR_SHAPE;
  const size_t need =
      msa_workspace_size(attn->num_rows, 0, 0, attn->num_heads, attn->head_dim, tbl_stride);
  if (need == 0 || need > (size_t)MSA_STATIC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MSA_ERR_CUDA;
  // the split counters must start at zero; the array keeps the last call's contents
  const size_t counter_bytes = (size_t)(attn->num_rows > 0 ? attn->num_rows : 1) * sizeof(uint32_t);
  if (cudaMemsetAsync(scratch, 0, counter_bytes, stream) != cudaSuccess) return MSA_ERR_CUDA;
  return msa_sparse_paged_attn(attn, sparse_tbl, tbl_stride, sparse_len, scratch,
                               (size_t)MSA_STATIC_SCRATCH_BYTES, dev_status, stream);
}
