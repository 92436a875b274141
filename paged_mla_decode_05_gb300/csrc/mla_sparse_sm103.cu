// Sparse (top-k) decode, first step, for sm_103a: the row list.
//
// Sparse MLA decode attends each request only to a selected list of its
// tokens (the "FlashInfer sparse MLA" attention backend of "[Kernel][DSV4.1]
// Fuse MXFP8 wo_b GEMM with sequence-parallel reduce-scatter" (vLLM PR
// #57428), serving command; the page names the backend only). The readings:
// topk_indices[b][i] are logical token positions of request b shared by all
// its heads; an entry outside [0, L) is padding; a position listed twice
// counts twice.
//
// This kernel turns each request's list into the cache rows of its valid
// entries (row = block id * block_size + slot), compacted in list order, and
// their count. The decode kernel then runs in row-list mode: its producers
// fetch those rows straight from the paged cache (16-byte cp.async), and
// the count is the request's length, read on the device. Entries whose block
// id lies outside [0, num_blocks) are skipped and raise MLA_DEVERR_BAD_BLOCK.
//
// One CTA of 512 threads per request; each pass takes 2048 entries, four
// consecutive ones per thread, with every list and block-table load of the
// pass issued before any is used, then compacts the valid ones in list order
// with a scan over the threads' counts.
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kRowsThreads = 512;
constexpr int kRowsWarps = kRowsThreads / 32;
constexpr int kRowsPerThread = 4;
constexpr int kRowsChunk = kRowsThreads * kRowsPerThread;

__global__ void __launch_bounds__(kRowsThreads) mla_sparse_rows_kernel(const SparseRowsParams p) {
  __shared__ int warp_n[kRowsWarps];
  // Launched as a dependent: the previous kernel's writes are visible after
  // the wait. It does not release the decode early (the decode then starts
  // at its exit): decode pairs placed while these CTAs still hold SMs ran
  // the top-2048, B=64 step up to 14 % slower.
  grid_dep_wait();
  const int b = blockIdx.x;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int L = max(0, __ldg(&p.seq_lens[b]));
  const int32_t* list = p.topk_indices + static_cast<int64_t>(b) * p.topk;
  const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  int32_t* rows = p.rows + static_cast<int64_t>(b) * p.topk;
  uint32_t err = 0;
  int count = 0;
  for (int c0 = 0; c0 < p.topk; c0 += kRowsChunk) {
    int tok[kRowsPerThread], blk[kRowsPerThread];
    bool valid[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      const int i = c0 + kRowsPerThread * t + k;
      tok[k] = i < p.topk ? __ldg(&list[i]) : -1;
    }
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      valid[k] = tok[k] >= 0 && tok[k] < L && tok[k] / p.block_size < p.max_blocks;
      blk[k] = valid[k] ? __ldg(&table[tok[k] / p.block_size]) : 0;
    }
    int n = 0;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      if (valid[k] && (blk[k] < 0 || static_cast<int64_t>(blk[k]) >= p.num_blocks)) {
        err |= 1u;   // MLA_DEVERR_BAD_BLOCK
        valid[k] = false;
      }
      n += valid[k] ? 1 : 0;
    }
    // Exclusive scan of n over the CTA's threads (thread order = list order).
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_n[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kRowsWarps; ++w) {
      before += w < warp ? warp_n[w] : 0;
      total += warp_n[w];
    }
    int pos = count + before + incl - n;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k)
      if (valid[k])   // num_blocks * block_size < 2^31 (checked by the caller)
        rows[pos++] = blk[k] * p.block_size + tok[k] % p.block_size;
    count += total;
    __syncthreads();   // warp_n[] is rewritten by the next pass
  }
  if (t == 0) p.counts[b] = count;
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0 && err) atomicOr(p.err, err);
}

}  // namespace

cudaError_t launch_sparse_rows(const SparseRowsParams& p, int B, cudaStream_t stream) {
  if (B <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = dependent_launch(dim3(B, 1, 1), dim3(kRowsThreads, 1, 1), 0, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_sparse_rows_kernel, p);
}

}  // namespace mla
