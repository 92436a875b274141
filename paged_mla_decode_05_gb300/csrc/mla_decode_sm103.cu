// Paged MLA decode for sm_103a: the paged-mode instances of the decode
// kernel (bf16 and FP8 caches) and the launchers; the kernel itself is in
// mla_decode_kernel.cuh.
#include "mla_decode_kernel.cuh"

namespace mla {

#ifdef MLA_TRACE
extern "C" cudaError_t mla_trace_set_buffer(void* dev_ptr) {
  return cudaMemcpyToSymbol(g_mla_trace, &dev_ptr, sizeof(dev_ptr));
}
#endif

cudaError_t decode_prepare_device() {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_decode_kernel<true, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return decode_rows_prepare_device();
}

cudaError_t decode_max_clusters(int* num_clusters) {
  cudaError_t e = decode_prepare_device();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Both instantiations share the launch shape and shared-memory size.
  return cudaOccupancyMaxActiveClusters(num_clusters, mla_decode_kernel<false, false>, &cfg);
}

cudaError_t launch_decode(const DecodeParams& p, int num_clusters, cudaStream_t stream) {
  if (p.rows) return launch_decode_rows(p, num_clusters, stream);
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = dependent_launch(dim3(2 * num_clusters, 1, 1), dim3(kThreads, 1, 1),
                                                  kSmemBytes, stream, attr);
  if (p.kv_fp8) return cudaLaunchKernelEx(&cfg, mla_decode_kernel<true, false>, p);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, false>, p);
}

}  // namespace mla
