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
// 4; section 5.2 "Split Attention + Combine"): the last CTA to finish a range
// does the merge, in range order, so results do not depend on timing.
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

template <bool FP8>
__global__ void __launch_bounds__(kDecWarps * 32, FP8 ? 3 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  decode_item<FP8, kDecWarps>(kmap, vmap, p, p.items[blockIdx.x], smem, threadIdx.x, 0);
}

__global__ void __launch_bounds__(kDecWarps * 32, kDecCtasNvfp4)
    decode_nvfp4_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  decode_item_nvfp4<kDecWarps>(kmap, vmap, p, p.items[blockIdx.x], smem, threadIdx.x, 0);
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap,
                          const DecodeParams &p, int num_items, int kv_dtype,
                          cudaStream_t s) {
  if (num_items == 0) return cudaSuccess;
  const bool fp8 = kv_dtype == PKV_KV_FP8_E4M3;
  if (kv_dtype == PKV_KV_NVFP4)
    decode_nvfp4_kernel<<<num_items, kDecWarps * 32, kDecSmemBytesNvfp4, s>>>(kmap, vmap, p);
  else if (fp8)
    decode_kernel<true><<<num_items, kDecWarps * 32, kDecSmemBytesFp8, s>>>(kmap, vmap, p);
  else
    decode_kernel<false><<<num_items, kDecWarps * 32, kDecSmemBytes, s>>>(kmap, vmap, p);
  return cudaGetLastError();
}

cudaError_t configure_decode() {
  cudaError_t e = cudaFuncSetAttribute(decode_nvfp4_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kDecSmemBytesNvfp4);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kDecSmemBytesFp8);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kDecSmemBytes);
}

}  // namespace pkv
