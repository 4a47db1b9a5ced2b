// One-launch mixed step: a batch holding both incremental-prefill chunks and
// decodes, as the V1 scheduler composes a step under its token budget (page
// "vLLM/V1 推理调度器", section 处理流程), runs as a single kernel launch
// instead of one launch per kind.
//
// The grid is the prefill tiles (longest first) followed by the split-KV
// decode items (longest first).  A CTA whose index falls on a prefill tile
// runs the tcgen05 prefill item with all 12 warps; a CTA on a decode item
// runs the decode item with 8 warps (8 rings of 3 stages in the same shared
// memory, so an SM keeps as many K/V bytes in flight as two 4-warp decode
// CTAs) and lets the other 4 warps exit.  Decode CTAs are scheduled last and
// fill the SMs that prefill tiles free at different times, so the tail of
// the prefill work overlaps the memory-bound decode work.  Split decode
// ranges (and prefill ranges) are merged by the merge kernels launched after
// this one.
#include "decode_body.cuh"
#include "prefill_tc_body.cuh"

namespace pkv {
namespace {

constexpr int kMixedDecWarps = 8;
static_assert(kMixedDecWarps * kDecStages * kDecStageBytes + 256 <= kTcSmemBytes - 1024,
              "decode rings must fit the prefill shared memory");

__global__ void __launch_bounds__(kTcThreads, 1)
    mixed_kernel(const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap kmap_pf,
                 const __grid_constant__ CUtensorMap vmap_pf,
                 const __grid_constant__ CUtensorMap kmap_dec,
                 const __grid_constant__ CUtensorMap vmap_dec, const PrefillParams pp,
                 const DecodeParams dp, const int n_prefill) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  if (static_cast<int>(blockIdx.x) < n_prefill) {
    prefill_tc_item<PKV_KV_BF16>(qmap, kmap_pf, vmap_pf, pp, pp.items[blockIdx.x], smem);
  } else {
    if (threadIdx.x >= kMixedDecWarps * 32) return;
    decode_item<false, kMixedDecWarps>(kmap_dec, vmap_dec, dp,
                                       dp.items[blockIdx.x - n_prefill], smem,
                                       threadIdx.x, 1);
  }
}

}  // namespace

cudaError_t launch_mixed(const CUtensorMap &qmap, const CUtensorMap &kmap_pf,
                         const CUtensorMap &vmap_pf, const CUtensorMap &kmap_dec,
                         const CUtensorMap &vmap_dec, const PrefillParams &pp,
                         const DecodeParams &dp, int n_prefill, int n_decode,
                         cudaStream_t s) {
  if (n_prefill + n_decode == 0) return cudaSuccess;
  mixed_kernel<<<n_prefill + n_decode, kTcThreads, kTcSmemBytes, s>>>(
      qmap, kmap_pf, vmap_pf, kmap_dec, vmap_dec, pp, dp, n_prefill);
  return cudaGetLastError();
}

cudaError_t configure_mixed() {
  // setmaxnreg moves registers within the CTA's launch allotment: the split
  // must not ask for more than the kernel was compiled (and launched) with
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, mixed_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kTcThreads < static_cast<int>(2 * 128 * kRegsSoftmax + 128 * kRegsCtl))
    return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(mixed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kTcSmemBytes);
}

}  // namespace pkv
