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
// One CTA of 128 threads per (request, head): thread t owns columns
// 4t .. 4t+3; the partials are read once with 16-byte loads (they are
// normally still in L2, written moments earlier by the decode kernel).
#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(128) mla_combine_kernel(const CombineParams p) {
  const CombineItem ci = p.items[blockIdx.x];
  const int h = blockIdx.y;
  const int t = threadIdx.x;
  float mx = -INFINITY;
  for (int i = 0; i < ci.n_slots; ++i)
    mx = fmaxf(mx, __ldg(&p.part_lse[static_cast<int64_t>(ci.first_slot + i) * p.H + h]));
  const int64_t orow = static_cast<int64_t>(ci.b) * p.H + h;
  uint2* out = reinterpret_cast<uint2*>(p.out + orow * kDc) + t;
  if (mx == -INFINITY) {
    *out = make_uint2(0u, 0u);
    if (t == 0) p.lse[orow] = -INFINITY;
    return;
  }
  float z = 0.0f;
  for (int i = 0; i < ci.n_slots; ++i)
    z += __expf(__ldg(&p.part_lse[static_cast<int64_t>(ci.first_slot + i) * p.H + h]) - mx);
  const float total = mx + __logf(z);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < ci.n_slots; ++i) {
    const int64_t slot = ci.first_slot + i;
    const float li = __ldg(&p.part_lse[slot * p.H + h]);
    if (li == -INFINITY) continue;
    const float wgt = __expf(li - total);
    const float4 o = __ldg(reinterpret_cast<const float4*>(p.part_o + (slot * p.H + h) * kDc) + t);
    acc.x = fmaf(wgt, o.x, acc.x);
    acc.y = fmaf(wgt, o.y, acc.y);
    acc.z = fmaf(wgt, o.z, acc.z);
    acc.w = fmaf(wgt, o.w, acc.w);
  }
  *out = make_uint2(pack2(acc.x, acc.y), pack2(acc.z, acc.w));
  if (t == 0) p.lse[orow] = total;
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int num_items, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  mla_combine_kernel<<<dim3(num_items, p.H, 1), dim3(128, 1, 1), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
