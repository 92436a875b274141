// Health check of the bounded waits: a barrier that nothing completes must
// make the wait routine give up and report MLA_DEVERR_TIMEOUT, with the
// device left usable. The routine is the one the decode roles call.
#include <cuda_runtime.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

#include "ptx_sm103.cuh"   // the same wait routine (internal linkage per unit)

namespace mla {
namespace {

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);   // one arrival expected; none ever comes
    fence_barrier_init();
  }
  __syncwarp();
  // Phase 0 of a fresh barrier completes only after its arrival, so this
  // wait can end only at the limit.
  const bool done = mbar_wait(smem_addr(&bar), 0);
  if (!done && threadIdx.x == 0) atomicOr(err, MLA_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t* err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace mla
