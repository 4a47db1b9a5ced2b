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
  if (kv_dtype == PKV_KV_NVFP4)
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

cudaError_t configure_prefill_tc() {
  cudaError_t e = configure_one<PKV_KV_BF16>();
  if (e == cudaSuccess) e = configure_one<PKV_KV_FP8_E4M3>();
  return e != cudaSuccess ? e : configure_one<PKV_KV_NVFP4>();
}

}  // namespace pkv
