// Sparse (top-k) decode, gather step, for sm_103a.
//
// Sparse MLA decode attends each request only to a selected list of its
// tokens (the "FlashInfer sparse MLA" attention backend of "[Kernel][DSV4.1]
// Fuse MXFP8 wo_b GEMM with sequence-parallel reduce-scatter" (vLLM PR
// #57428), serving command; the page names the backend only). The readings:
// topk_indices[b][i] are logical token positions of request b shared by all
// its heads; an entry outside [0, L) is padding.
//
// This kernel gathers, for each request, the cache rows of its valid entries
// into a compact cache in the caller's workspace: request b's rows occupy
// compact blocks [b * max_blocks_c, (b + 1) * max_blocks_c) in list order,
// its compact length is the number of valid entries, and the rows after it up
// to the next 32-row boundary (the page piece the decode kernel's last TMA box
// of the request covers) are zeroed, so every row the decode reads is finite.
// The decode kernel then runs unchanged over the compact cache, with the plan
// built for lengths that are upper bounds (topk) and the compact lengths read
// on the device. Entries whose block id lies outside [0, num_blocks) are
// skipped and raise MLA_DEVERR_BAD_BLOCK.
//
// One CTA of 256 threads per request: each pass takes 256 entries, compacts
// the valid ones with a warp ballot and a prefix over the 8 warps, then the 8
// warps copy the pass's rows, one row per warp at a time, 16 bytes per lane.
#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherWarps = kGatherThreads / 32;

__global__ void __launch_bounds__(kGatherThreads) mla_sparse_gather_kernel(const SparseGatherParams p) {
  __shared__ int64_t rows[kGatherThreads];   // source row of each compacted entry of the pass
  __shared__ int warp_n[kGatherWarps];
  const int b = blockIdx.x;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int L = max(0, __ldg(&p.seq_lens[b]));
  const int chunks = p.row_bytes / 16;                      // 72 (bf16) or 36 (FP8)
  const uint8_t* src = static_cast<const uint8_t*>(p.kv_cache);
  uint8_t* dst = static_cast<uint8_t*>(p.compact) +
                 static_cast<int64_t>(b) * p.rows_per_request * p.row_bytes;
  uint32_t err = 0;
  int count = 0;
  for (int c0 = 0; c0 < p.topk; c0 += kGatherThreads) {
    const int i = c0 + t;
    const int tok = i < p.topk ? __ldg(&p.topk_indices[static_cast<int64_t>(b) * p.topk + i]) : -1;
    bool valid = tok >= 0 && tok < L && tok / p.block_size < p.max_blocks;
    int64_t row = 0;
    if (valid) {
      const int blk = __ldg(&p.block_table[static_cast<int64_t>(b) * p.max_blocks + tok / p.block_size]);
      if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
        err |= 1u;   // MLA_DEVERR_BAD_BLOCK
        valid = false;
      } else {
        row = static_cast<int64_t>(blk) * p.block_size + tok % p.block_size;
      }
    }
    const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) warp_n[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, n = 0;
#pragma unroll
    for (int w = 0; w < kGatherWarps; ++w) {
      before += w < warp ? warp_n[w] : 0;
      n += warp_n[w];
    }
    if (valid) rows[before + __popc(ballot & ((1u << lane) - 1u))] = row;
    __syncthreads();
    for (int j = warp; j < n; j += kGatherWarps) {
      const uint4* s = reinterpret_cast<const uint4*>(src + rows[j] * p.row_bytes);
      uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(count + j) * p.row_bytes);
      for (int k = lane; k < chunks; k += 32) d[k] = __ldg(s + k);
    }
    count += n;
    __syncthreads();   // rows[] and warp_n[] are rewritten by the next pass
  }
  // Zero the rest of the last 32-row piece of the request.
  const int end = min(p.rows_per_request, (count + 31) & ~31);
  for (int j = count + warp; j < end; j += kGatherWarps) {
    uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(j) * p.row_bytes);
    for (int k = lane; k < chunks; k += 32) d[k] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (t == 0) p.compact_lens[b] = count;
  for (int j = t; j < p.max_blocks_c; j += kGatherThreads)
    p.compact_table[static_cast<int64_t>(b) * p.max_blocks_c + j] = b * p.max_blocks_c + j;
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0 && err) atomicOr(p.err, err);
}

}  // namespace

cudaError_t launch_sparse_gather(const SparseGatherParams& p, int B, cudaStream_t stream) {
  if (B <= 0) return cudaSuccess;
  mla_sparse_gather_kernel<<<dim3(B, 1, 1), dim3(kGatherThreads, 1, 1), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
