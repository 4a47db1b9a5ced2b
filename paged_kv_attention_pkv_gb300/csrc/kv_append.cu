// KV append ("KV 写入") and the validate-mode metadata check.
//
// The append stores each new token's K and V rows at the slot the scheduler
// assigned it (page "vLLM Agentic 推理｜面向 Agent 负载的推理优化", section
// 5.2: the KV write of K1).  It is a pure HBM scatter: every thread moves one
// 16-byte chunk of one (token, KV head) row of K and of V.  Slots point into
// [num_blocks][Hkv][block_size][128] pools.
#include "pkv_device.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  // first source -> upper byte, second -> lower byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

// 8 bf16 (one uint4) -> 8 E4M3 codes of x / scale (one uint2).
__device__ __forceinline__ uint2 quantize8(uint4 v, float scale) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint16_t a = cvt_e4m3x2(__fdiv_rn(bf16_lo(w[2 * i]), scale),
                                  __fdiv_rn(bf16_hi(w[2 * i]), scale));
    const uint16_t b = cvt_e4m3x2(__fdiv_rn(bf16_lo(w[2 * i + 1]), scale),
                                  __fdiv_rn(bf16_hi(w[2 * i + 1]), scale));
    out[i] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
  }
  return make_uint2(out[0], out[1]);
}

template <bool FP8>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendParams p) {
  constexpr int kChunks = kHeadDim / 8;  // 16-byte chunks of a bf16 row
  const int64_t total = p.num_tokens * p.hkv * kChunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < total; i += stride) {
    const int64_t row = i / kChunks;  // token * hkv + head
    const int c = static_cast<int>(i % kChunks);
    const int64_t t = row / p.hkv;
    const int h = static_cast<int>(row % p.hkv);
    const int64_t slot = p.slots[t];
    if (slot < 0) continue;  // padding token
    const int64_t blk = slot / p.bs;
    if (blk >= p.num_blocks) {  // never write outside the pool
      record_error(p.err, kErrBadSlot);
      continue;
    }
    const size_t dst = (static_cast<size_t>(blk) * p.hkv + h) * p.bs + slot % p.bs;
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(p.k_new) + row * kChunks + c);
    const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(p.v_new) + row * kChunks + c);
    if constexpr (!FP8) {
      reinterpret_cast<uint4 *>(p.k_cache)[dst * kChunks + c] = kv;
      reinterpret_cast<uint4 *>(p.v_cache)[dst * kChunks + c] = vv;
    } else {
      const size_t si = static_cast<size_t>(blk) * p.hkv + h;
      const float sk = __ldg(p.k_scale + si);
      const float sv = __ldg(p.v_scale + si);
      reinterpret_cast<uint2 *>(p.k_cache)[dst * kChunks + c] = quantize8(kv, sk);
      reinterpret_cast<uint2 *>(p.v_cache)[dst * kChunks + c] = quantize8(vv, sv);
    }
  }
}

// Validate mode: the device metadata must equal the host mirrors the plan
// was built from, and every block-table entry in use must be in the pool.
__global__ void __launch_bounds__(256) check_kernel(CheckParams p) {
  const int i = blockIdx.x;
  if (i >= p.num_seqs) return;
  if (threadIdx.x == 0) {
    if (p.seq_lens[i] != p.seq_lens_expect[i] || p.qsl[i] != p.qsl_expect[i] ||
        p.qsl[i + 1] != p.qsl_expect[i + 1])
      record_error(p.err, kErrMismatch);
  }
  const int64_t L = p.seq_lens_expect[i];
  const int64_t nb = (L + p.bs - 1) / p.bs;
  for (int64_t j = threadIdx.x; j < nb; j += blockDim.x) {
    const int32_t b = p.block_tables[static_cast<int64_t>(i) * p.bt_stride + j];
    if (b < 0 || b >= p.num_blocks) record_error(p.err, kErrBadBlock);
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, bool fp8, cudaStream_t s) {
  const int64_t total = p.num_tokens * p.hkv * (kHeadDim / 8);
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + 255) / 256;
  const int blocks = static_cast<int>(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
  if (fp8)
    kv_append_kernel<true><<<blocks, 256, 0, s>>>(p);
  else
    kv_append_kernel<false><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_check(const CheckParams &p, cudaStream_t s) {
  if (p.num_seqs == 0) return cudaSuccess;
  check_kernel<<<p.num_seqs, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
