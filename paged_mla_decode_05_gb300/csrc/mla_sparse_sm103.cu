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
// One CTA of 512 threads per request; each pass takes 512 entries and
// compacts the valid ones with a warp ballot and a prefix over the 16 warps.
#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kRowsThreads = 512;
constexpr int kRowsWarps = kRowsThreads / 32;

__global__ void __launch_bounds__(kRowsThreads) mla_sparse_rows_kernel(const SparseRowsParams p) {
  __shared__ int warp_n[kRowsWarps];
  const int b = blockIdx.x;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int L = max(0, __ldg(&p.seq_lens[b]));
  const int32_t* list = p.topk_indices + static_cast<int64_t>(b) * p.topk;
  const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  int32_t* rows = p.rows + static_cast<int64_t>(b) * p.topk;
  uint32_t err = 0;
  int count = 0;
  for (int c0 = 0; c0 < p.topk; c0 += kRowsThreads) {
    const int i = c0 + t;
    const int tok = i < p.topk ? __ldg(&list[i]) : -1;
    bool valid = tok >= 0 && tok < L && tok / p.block_size < p.max_blocks;
    int row = 0;
    if (valid) {
      const int blk = __ldg(&table[tok / p.block_size]);
      if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
        err |= 1u;   // MLA_DEVERR_BAD_BLOCK
        valid = false;
      } else {
        // num_blocks * block_size < 2^31 (checked by the caller)
        row = blk * p.block_size + tok % p.block_size;
      }
    }
    const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) warp_n[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, n = 0;
#pragma unroll
    for (int w = 0; w < kRowsWarps; ++w) {
      before += w < warp ? warp_n[w] : 0;
      n += warp_n[w];
    }
    if (valid) rows[count + before + __popc(ballot & ((1u << lane) - 1u))] = row;
    count += n;
    __syncthreads();   // warp_n[] is rewritten by the next pass
  }
  if (t == 0) p.counts[b] = count;
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0 && err) atomicOr(p.err, err);
}

}  // namespace

cudaError_t launch_sparse_rows(const SparseRowsParams& p, int B, cudaStream_t stream) {
  if (B <= 0) return cudaSuccess;
  mla_sparse_rows_kernel<<<dim3(B, 1, 1), dim3(kRowsThreads, 1, 1), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
