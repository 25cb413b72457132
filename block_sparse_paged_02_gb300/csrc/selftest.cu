// selftest.cu -- a check of the bounded waits every kernel of the library
// relies on to turn a stalled pipeline into a status bit instead of a hang
// ("Attention sinks for ROCm AITER sparse MLA" (vLLM PR 54404), "Key source
// snippets": a missing result must raise, not hang; "Add ROCm AITER sparse
// paged attention for MiniMax-M3" (vLLM PR 47287), "Risks and impact":
// errors are reported, not silent).
//
// One CTA waits, with the library's own mbar_wait and a caller-chosen
// limit, on an mbarrier armed for 1 KiB of transaction bytes that no copy
// ever delivers.  The wait gives up, the kernel records MSA_DEV_TIMEOUT and
// then takes the same exit the streaming kernels take on expiry: with
// MSA_CHECK_WAIT_TMEM it has tensor memory allocated and frees it; with
// MSA_CHECK_WAIT_COPY a real bulk copy is in flight on a second barrier and
// is drained (bounded) before the CTA leaves.  No fault, trap or endless
// loop is involved: the context stays usable.
#include "tcgen05.cuh"

namespace msa {
namespace {

__global__ void __launch_bounds__(128) bounded_wait_kernel(const uint4* src, uint32_t* status,
                                                           unsigned long long limit_ns,
                                                           int flags) {
  __shared__ __align__(16) uint64_t bars[2];
  __shared__ __align__(16) uint4 landing;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool with_tmem = (flags & MSA_CHECK_WAIT_TMEM) != 0;
  const bool with_copy = (flags & MSA_CHECK_WAIT_COPY) != 0;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
    // armed for bytes that never come: this phase cannot complete
    mbar_arrive_expect_tx(&bars[0], 1024);
    if (with_copy) {  // a real copy, completing on the second barrier
      mbar_arrive_expect_tx(&bars[1], 16);
      bulk_g2s(&landing, src, 16, &bars[1]);
    }
  }
  if (with_tmem && warp == 0) tc::tmem_alloc(&tmem_slot, 32);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // the wait every warp of a streaming kernel would take: bounded
  const bool ok = __syncthreads_and(mbar_wait(&bars[0], 0, limit_ns)) != 0;
  if (!ok) {
    if (tid == 0) atomicOr(status, MSA_DEV_TIMEOUT);
    // drain the copy still in flight (bounded too) before shared memory goes
    if (with_copy && tid == 0 && !mbar_wait(&bars[1], 0, limit_ns))
      atomicOr(status, MSA_DEV_TIMEOUT << 1);  // the drain itself gave up
  }
  tc::fence_before();
  __syncthreads();
  if (with_tmem && warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tmem_slot, 32);
  }
}

}  // namespace
}  // namespace msa

extern "C" msa_status msa_check_bounded_wait(uint32_t* dev_status, uint32_t limit_us,
                                             int32_t flags, const void* copy_src,
                                             cudaStream_t stream) {
  if (!dev_status) return MSA_ERR_NULL;
  if (limit_us < 1 || limit_us > 1000000u) return MSA_ERR_SHAPE;
  if (flags & ~(MSA_CHECK_WAIT_TMEM | MSA_CHECK_WAIT_COPY)) return MSA_ERR_UNSUPPORTED;
  if ((flags & MSA_CHECK_WAIT_COPY) &&
      (!copy_src || (reinterpret_cast<uintptr_t>(copy_src) & 15u) != 0))
    return MSA_ERR_NULL;
  msa::bounded_wait_kernel<<<1, 128, 0, stream>>>(static_cast<const uint4*>(copy_src), dev_status,
                                                  1000ull * limit_us, flags);
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
