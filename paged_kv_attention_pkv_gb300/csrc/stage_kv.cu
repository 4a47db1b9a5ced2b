// K/V staging for the tensor-core prefill over E4M3 and NVFP4 pools.
//
// The incremental prefill is compute-bound, and a request's whole context is
// read once per 256-row prefill item (a post-tool-call session of l_incr new
// tokens with query group G has l_incr * G / 256 items per KV head, each
// walking the same l_hist + l_incr keys; page "AMPD：PD 分离遇上多轮推理，
// incremental prefill 到底该在哪跑", sections 1 and 3).  Converting the
// quantised codes inside the prefill kernel therefore repeats the same
// conversion once per item, on two converter warps that cannot keep up with
// the tensor cores.  Staging converts each context block once per step
// instead, into staging pools laid out like a bf16 pool (page "vLLM 优化
// DeepSeek-V4.1-Flash：智能体吞吐提升 5 倍", section Kernels: the FP8 and NVFP4
// KV formats).
//
// NVFP4 pools stage K and V.  K keeps its exact code values,
// e2m1(code) * e4m3(micro scale) (at most 6 significant bits: exact in
// bf16), and its block scale goes to a staging scale array, applied to the
// fp32 scores per 16-key group as over the quantised pools (rounding K times
// its scale, even to f16, moves the scores of peaked queries by up to 1e-2).
// E4M3 pools stage V alone: the prefill reads E4M3 K from the pool with FP8
// MMAs, which need no conversion.  V becomes its value times the block
// scale, rounded once to nearest even.  The tensor-core prefill then reads
// the staged tiles with bf16 MMAs.
//
// Staged blocks of one request are consecutive: request r's block j is
// staging block first_r + j.  Rows past the request's context are written as
// zeros.  A block id outside the pool is recorded (kErrBadBlock) and staged
// as zeros.
#include "pkv_device.cuh"

namespace pkv {
namespace {

// Staged request of staging block sb: the last entry whose first block is
// <= sb (entries ascend by first block).
__device__ __forceinline__ int staged_request(const StageParams &p, int sb) {
  int lo = 0, hi = p.n_reqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.reqs[3 * mid + 1] <= sb)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// One CTA per staging block: every KV head, K (NVFP4) and V.  A thread
// takes one 16-byte load of codes per unit (16 E4M3 or 32 E2M1 elements)
// and writes its 2 or 4 16-byte bf16 chunks; units run in row order, so a
// warp reads and writes contiguous spans.
template <int FMT>
__global__ void __launch_bounds__(256) stage_kv_kernel(const StageParams p) {
  const int sb = blockIdx.x;
  __shared__ int s_info[3];
  if (threadIdx.x == 0) {
    const int r = staged_request(p, sb);
    const int seq = p.reqs[3 * r], first = p.reqs[3 * r + 1], len = p.reqs[3 * r + 2];
    const int j = sb - first;
    int32_t blk = p.block_tables[static_cast<int64_t>(seq) * p.bt_stride + j];
    if (blk < 0 || blk >= p.num_blocks) {
      record_error(p.err, kErrBadBlock);
      blk = -1;
    }
    s_info[0] = blk;
    s_info[1] = len - j * p.bs;   // valid rows of this block (may exceed bs)
  }
  __syncthreads();
  const int32_t blk = s_info[0];
  const int valid = s_info[1];
  const int bs = p.bs, hkv = p.hkv;
  const int bs_sh = 31 - __clz(bs);   // block sizes are powers of two
  constexpr bool V_ONLY = FMT == PKV_KV_FP8_E4M3;
  constexpr int kUnitSh = V_ONLY ? 3 : 2;        // units per 128-element row: 8 or 4
  constexpr int kOut = (kHeadDim >> kUnitSh) / 8;   // 16-byte bf16 chunks per unit
  if constexpr (!V_ONLY)
    for (int h = threadIdx.x; h < hkv; h += blockDim.x)
      p.k_stage_scale[static_cast<int64_t>(sb) * hkv + h] =
          blk >= 0 ? __ldg(p.k_scale + static_cast<int64_t>(blk) * hkv + h) : 0.f;
  const int per_kv = (hkv << bs_sh) << kUnitSh;   // units of one of K / V
  for (int c = threadIdx.x; c < (V_ONLY ? 1 : 2) * per_kv; c += blockDim.x) {
    const bool is_v = V_ONLY || c >= per_kv;
    const int cc = is_v && !V_ONLY ? c - per_kv : c;
    const int q = cc & ((1 << kUnitSh) - 1);    // unit of the row
    const int r = (cc >> kUnitSh) & (bs - 1);   // row in the block
    const int h = (cc >> kUnitSh) >> bs_sh;     // KV head
    uint32_t o[4 * kOut];
#pragma unroll
    for (int k = 0; k < 4 * kOut; ++k) o[k] = 0u;
    if (blk >= 0 && r < valid) {
      const int64_t tile = static_cast<int64_t>(blk) * hkv + h;
      const float sc = is_v ? __ldg(p.v_scale + tile) : 1.f;   // K: exact codes
      const uint8_t *pool = is_v ? p.v_pool : p.k_pool;
      if constexpr (FMT == PKV_KV_FP8_E4M3) {
        // elements 16q .. 16q + 15
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(pool + ((tile << bs_sh) + r) * 128) + q);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 a = e4m3x2_to_f32(ww[u] & 0xFFFFu);
          const float2 b = e4m3x2_to_f32(ww[u] >> 16);
          o[2 * u] = pack_bf16(a.x * sc, a.y * sc);
          o[2 * u + 1] = pack_bf16(b.x * sc, b.y * sc);
        }
      } else {
        // NVFP4 tile: rows in groups of min(bs, 64), a group's code rows
        // (64 bytes) then its micro-scale rows (8 bytes); elements
        // 32q .. 32q + 31 are micro blocks 2q and 2q + 1
        const int gs_sh = bs_sh < 6 ? bs_sh : 6;
        const int gs = 1 << gs_sh;
        const int rg = r & (gs - 1);
        const uint8_t *grp = pool + ((tile << bs_sh) + ((r >> gs_sh) << gs_sh)) * kNvfp4RowBytes;
        const uint4 codes = __ldg(reinterpret_cast<const uint4 *>(grp + rg * 64) + q);
        const uint16_t mus =
            __ldg(reinterpret_cast<const uint16_t *>(grp + gs * 64 + rg * 8) + q);
        const float2 mu = e4m3x2_to_f32(mus);
        const float ms[2] = {mu.x * sc, mu.y * sc};
        const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {   // 8 elements of micro block 2q + u / 2
          uint32_t f[4];
          e2m1x8_to_f16x2(cw[u], f);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&f[k]));
            o[4 * u + k] = pack_bf16(v.x * ms[u >> 1], v.y * ms[u >> 1]);
          }
        }
      }
    }
    uint4 *dst = reinterpret_cast<uint4 *>((is_v ? p.v_stage : p.k_stage) +
                                           (((static_cast<int64_t>(sb) * hkv + h) << bs_sh) + r) *
                                               kHeadDim) +
                 q * kOut;
#pragma unroll
    for (int k = 0; k < kOut; ++k)
      dst[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
  }
}

}  // namespace

cudaError_t launch_stage_kv(const StageParams &p, int num_stage_blocks, int kv_dtype,
                            cudaStream_t s) {
  if (num_stage_blocks == 0) return cudaSuccess;
  if (kv_dtype == PKV_KV_NVFP4)
    stage_kv_kernel<PKV_KV_NVFP4><<<num_stage_blocks, 256, 0, s>>>(p);
  else
    stage_kv_kernel<PKV_KV_FP8_E4M3><<<num_stage_blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
