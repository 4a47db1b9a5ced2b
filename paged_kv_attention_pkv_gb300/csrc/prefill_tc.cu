// Incremental-prefill attention on the 5th-generation tensor cores (tcgen05,
// accumulators and P in TMEM).
//
// l_incr new query tokens attend to l_hist cached tokens plus themselves
// (page "AMPD：PD 分离遇上多轮推理，incremental prefill 到底该在哪跑",
// sections 1 and 3).  A work item is (request, KV head, up to 256 query
// rows), where row r = t * G + g packs the G query heads of the KV head's
// group (GQA, page "vLLM Agentic 推理｜面向 Agent 负载的推理优化", section
// 4.3.1).  The rows form two 128-row Q tiles that share every 128-key K/V
// tile, so each byte brought into shared memory feeds 256 rows.
//
// Roles (384 threads, one CTA per SM; warp 11 only completes the third
// warpgroup, whose registers move to the softmax warpgroups):
//   warps 9-10  TMA producers, warp 9 for the Q tiles (one 3D box per
//               64-column half) and a 2-stage K ring, warp 10 for a 3-stage
//               V ring, tiles of 128 keys laid out [half][128 rows][64],
//               128-byte swizzled, one 2D box per block and half (16 copies
//               per tile for 16-token blocks: one issuing thread cannot keep
//               up with both rings); K of tile j is released once both QKs
//               of tile j are done, V once both PVs are done.
//   warp 8      one thread issues tcgen05.mma in the order
//                 PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1), ...
//               so the tensor core works on one Q tile while the softmax of
//               the other runs.  S_t = Q_t K^T lands in TMEM; P_t overwrites
//               S_t there (bf16 pairs) and is read back as the A operand of
//               O_t += P_t V (V an MN-major shared-memory operand).  Work is
//               signalled with tcgen05.commit on mbarriers.
//   warps 0-3   softmax of Q tile 0, warps 4-7 of Q tile 1: thread r owns row
//               r (TMEM lane r), loads its 128 scores with one tcgen05.ld,
//               masks causally on diagonal tiles, keeps a
//               running max in log2 units that only moves when it grows by
//               more than 8 (O is rescaled rarely), writes P, and finally
//               normalises O.
//
// A step with few items has their key ranges split into runs of whole tiles
// (one item per run); each run writes O / l and its log-sum-exp as a partial
// and prefill_merge_kernel combines the runs of each item, the log-sum-exp
// merge of split attention (page "vLLM Agentic 推理｜面向 Agent 负载的推理
// 优化", section 4.3.3).
#include "prefill_tc_body.cuh"

namespace pkv {
namespace {

template <int FMT>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  prefill_tc_item<FMT>(qmap, kmap, vmap, p, p.items[blockIdx.x], smem);
}

// Merges the key-range partials of prefill items split over key ranges
// (online-softmax combine: weights 2^(lse_s - max) over the ranges).  The
// first ranges of the split items lead the item list; block b takes 8 rows
// of group b / 32, one warp per row, lane l holding head dims 4l .. 4l + 3
// and the log-sum-exp of range l (at most kPfMaxSplits ranges).
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillParams p) {
  const pkv_work_item it = p.items[blockIdx.x >> 5];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int prow = (blockIdx.x & 31) * 8 + warp;   // line in a partial slot
  const int t = prow >> 7, r = prow & 127;
  const int G = p.group, R = pf_tile_rows(G);
  const int n0 = it.n_rows < R ? it.n_rows : R;
  if (r >= (t == 0 ? n0 : it.n_rows - n0)) return;
  const int rowg = it.row0 + R * t + r;
  const int64_t orow = static_cast<int64_t>(it.tok0 + rowg / G) * p.hq +
                       it.kv_head * G + rowg % G;
  const int ns = it.n_split;
  auto slot = [&](int s2) {
    return (static_cast<int64_t>(it.pair) + int64_t(s2) * kPfPartSlots) * kDecCols + prow;
  };
  const float lse_l = lane < ns ? __ldcg(p.part_lse + slot(lane)) : -CUDART_INF_F;
  float M = lse_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Mu = M == -CUDART_INF_F ? 0.f : M;
  float w_l = lane < ns ? exp2f(lse_l - Mu) : 0.f;
  float wsum = w_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  w_l *= wsum > 0.f ? 1.f / wsum : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s2 = 0; s2 < ns; ++s2) {
    const float w = __shfl_sync(0xffffffffu, w_l, s2);
    const float4 x = __ldcg(reinterpret_cast<const float4 *>(p.part_o + slot(s2) * kHeadDim) + lane);
    acc.x += w * x.x;
    acc.y += w * x.y;
    acc.z += w * x.z;
    acc.w += w * x.w;
  }
  reinterpret_cast<uint2 *>(p.out + orow * kHeadDim)[lane] =
      make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  if (lane == 0 && p.lse != nullptr)
    p.lse[orow] = wsum > 0.f ? (Mu + log2f(wsum)) * kLn2 : -CUDART_INF_F;
}

template <int FMT>
cudaError_t configure_one() {
  // setmaxnreg moves registers within the CTA's launch allotment: the split
  // must not ask for more than the kernel was compiled (and launched) with
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<FMT>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kTcThreads < static_cast<int>(2 * 128 * kRegsSoftmax + 128 * kRegsCtl))
    return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(prefill_tc_kernel<FMT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &qmap, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, const PrefillParams &p,
                              int num_items, int kv_dtype, cudaStream_t s) {
  if (num_items == 0) return cudaSuccess;
  if (kv_dtype == kFmtStaged)
    prefill_tc_kernel<kFmtStaged><<<num_items, kTcThreads, kTcSmemBytes, s>>>(qmap, kmap,
                                                                              vmap, p);
  else if (kv_dtype == kFmtStagedV)
    prefill_tc_kernel<kFmtStagedV><<<num_items, kTcThreads, kTcSmemBytes, s>>>(qmap, kmap,
                                                                               vmap, p);
  else if (kv_dtype == PKV_KV_NVFP4)
    prefill_tc_kernel<PKV_KV_NVFP4><<<num_items, kTcThreads, kTcSmemBytes, s>>>(qmap, kmap,
                                                                               vmap, p);
  else if (kv_dtype == PKV_KV_FP8_E4M3)
    prefill_tc_kernel<PKV_KV_FP8_E4M3><<<num_items, kTcThreads, kTcSmemBytes, s>>>(qmap, kmap,
                                                                                  vmap, p);
  else
    prefill_tc_kernel<PKV_KV_BF16><<<num_items, kTcThreads, kTcSmemBytes, s>>>(qmap, kmap,
                                                                              vmap, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_merge(const PrefillParams &p, int num_groups, cudaStream_t s) {
  if (num_groups == 0) return cudaSuccess;
  prefill_merge_kernel<<<num_groups * 32, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t configure_prefill_tc() {
  cudaError_t e = configure_one<PKV_KV_BF16>();
  if (e == cudaSuccess) e = configure_one<PKV_KV_FP8_E4M3>();
  if (e == cudaSuccess) e = configure_one<kFmtStaged>();
  if (e == cudaSuccess) e = configure_one<kFmtStagedV>();
  return e != cudaSuccess ? e : configure_one<PKV_KV_NVFP4>();
}

}  // namespace pkv
