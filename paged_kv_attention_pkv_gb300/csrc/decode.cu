// Split-KV decode attention over a paged KV cache.
//
// Decode is the memory-bound step: every token of every request's context is
// read once per step while only one (or a few) query tokens attend to it
// (page "AMPD：PD 分离遇上多轮推理，incremental prefill 到底该在哪跑", section 1;
// page "vLLM Agentic 推理｜面向 Agent 负载的推理优化", section 4.3.2).  A work
// item is (request, KV head, key range): the G query heads of the group (and
// up to 8 / G query tokens) form the 8 columns of one m16n8k16 MMA tile whose
// 16 rows are keys (S^T = K Q^T), so a KV head's rows are read once for the
// whole group (GQA, same page section 4.3.1).  Ranges of one (request, KV
// head) are merged through their log-sum-exp (same page, section 4.3.3 step
// 4; section 5.2 "Split Attention + Combine") by decode_merge_kernel, in
// range order, so results do not depend on timing.  (A merge by the last CTA
// to finish, inside this kernel, measured slower: it lengthened the tail and
// changed how the decode loop was compiled.)
//
// Data movement: each of the 4 warps owns a ring of 3 stages in shared
// memory.  Lane 0 fills a stage with 2D TMA tile copies of the (block, KV
// head) rows of K and V, 128-byte swizzled, completing on an mbarrier; the
// warp's lanes read it with conflict-free ldmatrix / ld.shared patterns.
// E4M3 pools: QK runs on FP8 MMAs over the stored K codes with the query
// split into two E4M3 parts (about bf16 precision); V codes are paired per
// head-dim column with byte permutes and converted exactly to f16 in
// hardware, PV runs in f16 with V's per-block scale folded into P.  K's
// per-block scale is folded into the fp32 scores.
#include "decode_nvfp4.cuh"

namespace pkv {
namespace {

// MASK: the masked context-parallel shard view (interleaves shorter than a
// stage), a separate instantiation so that the plain decode carries no test
// for it.
template <bool FP8, bool MASK>
__global__ void __launch_bounds__(kDecWarps * 32, FP8 ? 3 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  decode_item<FP8, kDecWarps, MASK>(kmap, vmap, p, p.items[blockIdx.x], smem, threadIdx.x, 0);
}

template <bool MASK>
__global__ void __launch_bounds__(kDecWarps * 32, kDecCtasNvfp4)
    decode_nvfp4_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  decode_item_nvfp4<kDecWarps, MASK>(kmap, vmap, p, p.items[blockIdx.x], smem, threadIdx.x, 0);
}

// Merges the key ranges of split decode items.  The first ranges of the
// split (request, KV head) pairs lead the item list; block b takes pair b,
// warp n its row n (up to kDecCols rows), lane l head dims 4l .. 4l + 3.
// Weights 2^(lse_s - max) / sum over the ranges (lanes striding over the
// ranges for the max and the sum), then the ranges' rows accumulated with
// independent loads.
__global__ void __launch_bounds__(kDecCols * 32) decode_merge_kernel(const DecodeParams p) {
  const pkv_work_item it = p.items[blockIdx.x];
  const int n = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (n >= it.n_rows) return;
  const int ns = it.n_split;
  const float *lse_p = p.part_lse + static_cast<int64_t>(it.pair) * kDecCols + n;
  const float *o_p = p.part_o + (static_cast<int64_t>(it.pair) * kDecCols + n) * kHeadDim;
  constexpr int64_t kSlotFloats = int64_t(kDecCols) * kHeadDim;
  // lane l holds the log-sum-exp of range l (the first 32 ranges: one load
  // serves the max, the sum and the weights of most merges)
  const float lse0 = lane < ns ? __ldcg(lse_p + lane * kDecCols) : -CUDART_INF_F;
  float M = lse0;
  for (int s2 = lane + 32; s2 < ns; s2 += 32) M = fmaxf(M, __ldcg(lse_p + s2 * kDecCols));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Mu = M == -CUDART_INF_F ? 0.f : M;
  float Ls = lane < ns ? exp2f(lse0 - Mu) : 0.f;
  for (int s2 = lane + 32; s2 < ns; s2 += 32) Ls += exp2f(__ldcg(lse_p + s2 * kDecCols) - Mu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  const float winv = Ls > 0.f ? 1.f / Ls : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const int s2 = s0 + lane;
    const float lse_s = s0 == 0 ? lse0 : (s2 < ns ? __ldcg(lse_p + s2 * kDecCols) : -CUDART_INF_F);
    const float w_l = s2 < ns ? exp2f(lse_s - Mu) * winv : 0.f;
    const int cnt = ns - s0 < 32 ? ns - s0 : 32;
#pragma unroll 8
    for (int k = 0; k < cnt; ++k) {
      const float w = __shfl_sync(0xffffffffu, w_l, k);
      const float4 x = __ldcg(reinterpret_cast<const float4 *>(o_p + (s0 + k) * kSlotFloats) + lane);
      acc.x += w * x.x;
      acc.y += w * x.y;
      acc.z += w * x.z;
      acc.w += w * x.w;
    }
  }
  const int r = it.row0 + n;
  const int64_t row = static_cast<int64_t>(it.tok0 + r / p.group) * p.hq +
                      it.kv_head * p.group + r % p.group;
  if (p.out_f32 != nullptr)
    reinterpret_cast<float4 *>(p.out_f32 + row * kHeadDim)[lane] = acc;
  else
    reinterpret_cast<uint2 *>(p.out + row * kHeadDim)[lane] =
        make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  if (lane == 0 && p.lse != nullptr)
    p.lse[row] = Ls > 0.f ? (Mu + log2f(Ls)) * kLn2 : -CUDART_INF_F;
}

// The same merge for steps whose pairs have more than 32 ranges (one long
// request split over the whole machine): walked by one warp, a row's ranges
// cost one dependent L2 round trip per 8 of them.  Here a CTA takes one row
// (blockIdx.y) of one pair and its 8 warps take contiguous runs of the
// ranges; the maximum, the weight sum and the per-warp sums are combined in
// a fixed order, so the result does not depend on timing.
constexpr int kWideMergeWarps = 8;

__global__ void __launch_bounds__(kWideMergeWarps * 32, 2)
    decode_merge_wide_kernel(const DecodeParams p) {
  const pkv_work_item it = p.items[blockIdx.x];
  const int n = blockIdx.y;
  if (n >= it.n_rows) return;   // the whole CTA
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns = it.n_split;
  const float *lse_p = p.part_lse + static_cast<int64_t>(it.pair) * kDecCols + n;
  const float *o_p = p.part_o + (static_cast<int64_t>(it.pair) * kDecCols + n) * kHeadDim;
  constexpr int64_t kSlotFloats = int64_t(kDecCols) * kHeadDim;
  constexpr int kThreads = kWideMergeWarps * 32;
  __shared__ float red[kWideMergeWarps];
  __shared__ float4 part[kWideMergeWarps][32];
  // largest log-sum-exp over the ranges
  float M = -CUDART_INF_F;
  for (int s2 = tid; s2 < ns; s2 += kThreads) M = fmaxf(M, __ldcg(lse_p + s2 * kDecCols));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kWideMergeWarps; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  const float Mu = M == -CUDART_INF_F ? 0.f : M;
  // sum of the weights 2^(lse_s - max)
  float Ls = 0.f;
  for (int s2 = tid; s2 < ns; s2 += kThreads) Ls += exp2f(__ldcg(lse_p + s2 * kDecCols) - Mu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  if (lane == 0) red[warp] = Ls;
  __syncthreads();
  Ls = 0.f;
#pragma unroll
  for (int w = 0; w < kWideMergeWarps; ++w) Ls += red[w];
  const float winv = Ls > 0.f ? 1.f / Ls : 0.f;
  // this warp's run of ranges, lane l holding head dims 4l .. 4l + 3
  const int per = (ns + kWideMergeWarps - 1) / kWideMergeWarps;
  const int s_lo = warp * per, s_hi = min(ns, s_lo + per);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = s_lo; s0 < s_hi; s0 += 32) {
    const int s2 = s0 + lane;
    const float w_l = s2 < s_hi ? exp2f(__ldcg(lse_p + s2 * kDecCols) - Mu) * winv : 0.f;
    const int cnt = s_hi - s0 < 32 ? s_hi - s0 : 32;
#pragma unroll 8
    for (int k = 0; k < cnt; ++k) {
      const float w = __shfl_sync(0xffffffffu, w_l, k);
      const float4 x = __ldcg(reinterpret_cast<const float4 *>(o_p + (s0 + k) * kSlotFloats) + lane);
      acc.x += w * x.x;
      acc.y += w * x.y;
      acc.z += w * x.z;
      acc.w += w * x.w;
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp != 0) return;
  acc = part[0][lane];
#pragma unroll
  for (int w = 1; w < kWideMergeWarps; ++w) {
    const float4 x = part[w][lane];
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
  const int r = it.row0 + n;
  const int64_t row = static_cast<int64_t>(it.tok0 + r / p.group) * p.hq +
                      it.kv_head * p.group + r % p.group;
  if (p.out_f32 != nullptr)
    reinterpret_cast<float4 *>(p.out_f32 + row * kHeadDim)[lane] = acc;
  else
    reinterpret_cast<uint2 *>(p.out + row * kHeadDim)[lane] =
        make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  if (lane == 0 && p.lse != nullptr)
    p.lse[row] = Ls > 0.f ? (Mu + log2f(Ls)) * kLn2 : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_decode_merge(const DecodeParams &p, int num_groups, int max_split,
                                cudaStream_t s) {
  if (num_groups == 0) return cudaSuccess;
  if (max_split > 32)
    decode_merge_wide_kernel<<<dim3(num_groups, kDecCols), kWideMergeWarps * 32, 0, s>>>(p);
  else
    decode_merge_kernel<<<num_groups, kDecCols * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap,
                          const DecodeParams &p, int num_items, int kv_dtype,
                          cudaStream_t s) {
  if (num_items == 0) return cudaSuccess;
  const bool fp8 = kv_dtype == PKV_KV_FP8_E4M3;
  const dim3 grid(num_items), block(kDecWarps * 32);
  if (kv_dtype == PKV_KV_NVFP4) {
    if (p.dcp_mask)
      decode_nvfp4_kernel<true><<<grid, block, kDecSmemBytesNvfp4, s>>>(kmap, vmap, p);
    else
      decode_nvfp4_kernel<false><<<grid, block, kDecSmemBytesNvfp4, s>>>(kmap, vmap, p);
  } else if (fp8) {
    if (p.dcp_mask)
      decode_kernel<true, true><<<grid, block, kDecSmemBytesFp8, s>>>(kmap, vmap, p);
    else
      decode_kernel<true, false><<<grid, block, kDecSmemBytesFp8, s>>>(kmap, vmap, p);
  } else {
    if (p.dcp_mask)
      decode_kernel<false, true><<<grid, block, kDecSmemBytes, s>>>(kmap, vmap, p);
    else
      decode_kernel<false, false><<<grid, block, kDecSmemBytes, s>>>(kmap, vmap, p);
  }
  return cudaGetLastError();
}

cudaError_t configure_decode() {
  const void *kernels[] = {
      reinterpret_cast<const void *>(decode_nvfp4_kernel<false>),
      reinterpret_cast<const void *>(decode_nvfp4_kernel<true>),
      reinterpret_cast<const void *>(decode_kernel<true, false>),
      reinterpret_cast<const void *>(decode_kernel<true, true>),
      reinterpret_cast<const void *>(decode_kernel<false, false>),
      reinterpret_cast<const void *>(decode_kernel<false, true>)};
  const int bytes[] = {kDecSmemBytesNvfp4, kDecSmemBytesNvfp4, kDecSmemBytesFp8,
                       kDecSmemBytesFp8,   kDecSmemBytes,      kDecSmemBytes};
  for (int k = 0; k < 6; ++k) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernels[k], cudaFuncAttributeMaxDynamicSharedMemorySize, bytes[k]);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pkv
