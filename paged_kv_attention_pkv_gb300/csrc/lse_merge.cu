// Merge of partial attention results over disjoint key sets.
//
// Under decode context parallelism every rank attends to its own share of
// the KV tokens and produces a partial output O_i with its log-sum-exp
// LSE_i; the partials are exchanged and combined with weights
// exp(LSE_i - LSE), LSE = ln sum_i exp(LSE_i) (page "vLLM Agentic 推理｜面向
// Agent 负载的推理优化", section 4.3.3, steps 3 and 4).  One warp merges one
// row: each lane owns 4 of the 128 head-dim values.
#include <math_constants.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(128)
    lse_merge_kernel(const float *__restrict__ parts_o, const float *__restrict__ parts_lse,
                     int num_parts, int64_t num_rows, __nv_bfloat16 *__restrict__ out,
                     float *__restrict__ lse) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= num_rows) return;
  float m = -CUDART_INF_F;
  for (int s = 0; s < num_parts; ++s) m = fmaxf(m, __ldg(parts_lse + s * num_rows + row));
  const float mu = m == -CUDART_INF_F ? 0.f : m;
  float l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < num_parts; ++s) {
    const float w = expf(__ldg(parts_lse + s * num_rows + row) - mu);
    const float4 o = __ldg(reinterpret_cast<const float4 *>(
                               parts_o + (s * num_rows + row) * kHeadDim) + lane);
    l += w;
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint2 v;
  v.x = pack_bf16(acc.x * inv, acc.y * inv);
  v.y = pack_bf16(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2 *>(out + row * kHeadDim)[lane] = v;
  if (lse != nullptr && lane == 0) lse[row] = l > 0.f ? mu + logf(l) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_lse_merge(const float *parts_o, const float *parts_lse, int num_parts,
                             int64_t num_rows, __nv_bfloat16 *out, float *lse,
                             cudaStream_t s) {
  if (num_rows == 0) return cudaSuccess;
  const int64_t blocks = (num_rows + 3) / 4;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), 128, 0, s>>>(parts_o, parts_lse, num_parts,
                                                                 num_rows, out, lse);
  return cudaGetLastError();
}

}  // namespace pkv
