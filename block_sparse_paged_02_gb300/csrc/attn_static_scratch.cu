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
// The array is shared by every call in the process.  Rows of 2 to 8 splits
// merge inside their thread-block cluster and rows of one split need no
// merge, so those calls use only the array's first bytes; rows of more
// splits (top-k above 128 blocks) merge through the counters and partials,
// and the counters are cleared on the stream before such a call.  Two calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on the array and give undefined results.
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
  // every argument check first: a refused call touches neither the array nor
  // the stream
  int pps = 0, splits = 0;
  const msa_status st =
      msa::attn_prepare(attn, sparse_tbl, tbl_stride, sparse_len, dev_status, &pps, &splits);
  if (st != MSA_OK || attn->num_rows == 0) return st;
  // only what this launch's split uses: the per-row counters, plus the
  // (m, l, acc) partials when a row has more splits than one cluster merges
  if (msa::attn_scratch_need(attn->num_rows, splits) > (size_t)MSA_STATIC_SCRATCH_BYTES)
    return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MSA_ERR_CUDA;
  if (splits > msa::kMaxClusterSplits) {
    // the last-arriver counters must start at zero; the array keeps whatever
    // the last call (or an interrupted one) left there
    if (cudaMemsetAsync(scratch, 0, (size_t)attn->num_rows * sizeof(uint32_t), stream) !=
        cudaSuccess)
      return MSA_ERR_CUDA;
  }
  return msa::attn_run(attn, sparse_tbl, tbl_stride, sparse_len, scratch, pps, splits,
                       dev_status, stream);
}
