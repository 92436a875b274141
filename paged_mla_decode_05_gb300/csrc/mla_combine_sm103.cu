// Split-KV combine kernel for sm_103a.
//
// Merges the split partials of one request, the reduction step of "SM100
// Cutlass MLA decode with unrestricted num_heads (< 128) for DeepSeek TP"
// (vLLM PR #20769), bot summary: each split i of request b carries a
// normalised partial o_i[h, 512] and its log-sum-exp lse_i[h]; the request's
// result is
//     lse = ln sum_i exp(lse_i),   out = sum_i exp(lse_i - lse) * o_i.
// Partials with lse_i = -inf (no tokens) get weight 0.
//
// One CTA of 256 threads (8 warps) per (request, head). The weights
// exp(lse_i - lse) are computed once into shared memory; warp w then sums the
// slots i = w, w + 8, ... with each lane owning 16 of the 512 columns (four
// independent 16-byte loads per slot, two slots per iteration in flight), and
// the eight partial sums are added through shared memory. The partials are
// normally still in L2, written moments earlier by the decode kernel.
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kMaxCombineSlots = 4096;   // the planner's largest forced split count

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(const CombineParams p) {
  extern __shared__ float smem[];                 // [n_slots] weights, then [8][512] sums
  __shared__ float red[kCombineWarps];
  grid_dep_wait();   // the decode kernel's partials are complete and visible
  const CombineItem ci = p.items[blockIdx.x];
  const int h = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int n = ci.n_slots;
  float* wgt = smem;
  float* sums = smem + ((n + 3) & ~3);
  const float* lse_col = p.part_lse + static_cast<int64_t>(ci.first_slot) * p.H + h;

  // Weights: lse = max + ln sum exp(lse_i - max); w_i = exp(lse_i - lse).
  float mx = -INFINITY;
  for (int i = t; i < n; i += kCombineThreads) {
    const float li = __ldg(lse_col + static_cast<int64_t>(i) * p.H);
    wgt[i] = li;
    mx = fmaxf(mx, li);
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, red[w]);
  const int64_t orow = static_cast<int64_t>(ci.b) * p.H + h;
  if (mx == -INFINITY) {   // no tokens in any split
    if (t < kDc / 8) reinterpret_cast<uint4*>(p.out + orow * kDc)[t] = make_uint4(0u, 0u, 0u, 0u);
    if (t == 0) p.lse[orow] = -INFINITY;
    return;
  }
  float z = 0.0f;
  for (int i = t; i < n; i += kCombineThreads) z += __expf(wgt[i] - mx);
  z = warp_sum(z);
  __syncthreads();   // everyone has read red[] and wgt[] as lse values
  if (lane == 0) red[warp] = z;
  __syncthreads();
  z = 0.0f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) z += red[w];
  const float total = mx + __logf(z);
  for (int i = t; i < n; i += kCombineThreads) {
    const float li = wgt[i];
    wgt[i] = li == -INFINITY ? 0.0f : __expf(li - total);
  }
  __syncthreads();

  // Weighted sum: warp w takes slots w, w + 8, ...; lane owns columns
  // 4 * (lane + 32 j), j < 4.
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* base = reinterpret_cast<const float4*>(
      p.part_o + (static_cast<int64_t>(ci.first_slot) * p.H + h) * kDc);
  const int64_t slot_stride = static_cast<int64_t>(p.H) * (kDc / 4);   // in float4
  int i = warp;
  for (; i + kCombineWarps < n; i += 2 * kCombineWarps) {
    const float w0 = wgt[i], w1 = wgt[i + kCombineWarps];
    float4 a[4], b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a[j] = __ldg(base + i * slot_stride + lane + 32 * j);
      b[j] = __ldg(base + (i + kCombineWarps) * slot_stride + lane + 32 * j);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j].x = fmaf(w0, a[j].x, acc[j].x); acc[j].y = fmaf(w0, a[j].y, acc[j].y);
      acc[j].z = fmaf(w0, a[j].z, acc[j].z); acc[j].w = fmaf(w0, a[j].w, acc[j].w);
      acc[j].x = fmaf(w1, b[j].x, acc[j].x); acc[j].y = fmaf(w1, b[j].y, acc[j].y);
      acc[j].z = fmaf(w1, b[j].z, acc[j].z); acc[j].w = fmaf(w1, b[j].w, acc[j].w);
    }
  }
  if (i < n) {
    const float w0 = wgt[i];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 a = __ldg(base + i * slot_stride + lane + 32 * j);
      acc[j].x = fmaf(w0, a.x, acc[j].x); acc[j].y = fmaf(w0, a.y, acc[j].y);
      acc[j].z = fmaf(w0, a.z, acc[j].z); acc[j].w = fmaf(w0, a.w, acc[j].w);
    }
  }
  float4* my = reinterpret_cast<float4*>(sums + warp * kDc);
#pragma unroll
  for (int j = 0; j < 4; ++j) my[lane + 32 * j] = acc[j];
  __syncthreads();

  // Column c (t < 128 handles 4 columns): add the 8 warps' sums, round to bf16.
  if (t < kDc / 4) {
    float4 s = reinterpret_cast<const float4*>(sums)[t];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) {
      const float4 v = reinterpret_cast<const float4*>(sums + w * kDc)[t];
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    reinterpret_cast<uint2*>(p.out + orow * kDc)[t] = make_uint2(pack2(s.x, s.y), pack2(s.z, s.w));
  }
  if (t == 0) p.lse[orow] = total;
}

}  // namespace

cudaError_t combine_prepare_device() {
  const int max_smem = (kMaxCombineSlots + kCombineWarps * kDc) * 4;
  return cudaFuncSetAttribute(mla_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

cudaError_t launch_combine(const CombineParams& p, int num_items, int max_slots,
                           cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  if (max_slots < 1 || max_slots > kMaxCombineSlots) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(((max_slots + 3) & ~3) + kCombineWarps * kDc) * 4;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      dependent_launch(dim3(num_items, p.H, 1), dim3(kCombineThreads, 1, 1), smem, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
}

}  // namespace mla
