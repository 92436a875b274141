// Row-list MLA decode for sm_103a: the instances of the decode kernel (bf16
// and FP8 caches) whose producers fetch each tile's rows from a per-request
// list of cache rows with 16-byte cp.async copies spread over six of the
// pair's warps (the sparse decode's second
// step); the kernel itself is in mla_decode_kernel.cuh.
#include "mla_decode_kernel.cuh"

namespace mla {

cudaError_t decode_rows_prepare_device() {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<false, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_decode_kernel<true, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_decode_rows(const DecodeParams& p, int num_clusters, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = dependent_launch(dim3(2 * num_clusters, 1, 1), dim3(kThreads, 1, 1),
                                                  kSmemBytes, stream, attr);
  if (p.kv_fp8) return cudaLaunchKernelEx(&cfg, mla_decode_kernel<true, true>, p);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, true>, p);
}

}  // namespace mla
