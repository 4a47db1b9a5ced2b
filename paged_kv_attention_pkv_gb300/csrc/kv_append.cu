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

// ---- NVFP4 -------------------------------------------------------------------
// E2M1 code of an fp32 value: nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 by its
// magnitude, ties to the even code, saturating at 6; the sign bit is copied
// (NaN gives 0).  Each comparison adds one step of the grid; the midpoints
// that are ties use > when the lower code is even and >= when it is odd.
__device__ __forceinline__ uint32_t e2m1_code(float q) {
  const float a = fabsf(q);
  const uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
                     (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return c | ((__float_as_uint(q) >> 28) & 8u);
}

// Value of an E4M3 code (exact).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  return e4m3x2_to_f32(code & 0xFFu).x;
}

// Micro scale of 16 values with largest magnitude amax under the (block, KV
// head) scale: E4M3(amax / (6 scale)), product and quotient in fp32.
__device__ __forceinline__ uint32_t nvfp4_micro_scale(float amax, float scale) {
  return e4m3x2_from_f32(__fdiv_rn(amax, __fmul_rn(6.f, scale)), 0.f) & 0xFFu;
}

// Codes of 8 values (element 2j in the low nibble of byte j) for the
// quantisation step `step` = scale * micro scale (0: all codes 0).
__device__ __forceinline__ uint32_t nvfp4_codes8(const float (&x)[8], float step) {
  uint32_t w = 0;
  if (step != 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= e2m1_code(__fdiv_rn(x[i], step)) << (4 * i);
  }
  return w;
}

// One micro block (16 bf16 values, two uint4) -> 8 code bytes; *ms gets its
// micro-scale code.
__device__ __forceinline__ uint2 nvfp4_quantize16(uint4 a, uint4 b, float scale, uint32_t *ms) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[2][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[i >> 2][2 * (i & 3)] = bf16_lo(w[i]);
    x[i >> 2][2 * (i & 3) + 1] = bf16_hi(w[i]);
    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  }
  *ms = nvfp4_micro_scale(amax, scale);
  const float step = __fmul_rn(scale, e4m3_value(*ms));
  return make_uint2(nvfp4_codes8(x[0], step), nvfp4_codes8(x[1], step));
}

// Byte offsets inside a (block, KV head) tile of row `off`'s codes and micro
// scales: rows in groups of min(bs, 64), each group its codes then scales.
__device__ __forceinline__ void nvfp4_row_offsets(int bs, int64_t off, int64_t *codes,
                                                  int64_t *mscale) {
  const int gs = bs < kNvfp4Group ? bs : kNvfp4Group;
  const int64_t group = (off / gs) * gs * kNvfp4RowBytes;
  const int64_t r = off % gs;
  *codes = group + r * (kHeadDim / 2);
  *mscale = group + gs * (kHeadDim / 2) + r * (kHeadDim / 16);
}

// NVFP4 append: one thread per micro block (16 elements) of a (token, KV
// head) row of K and of V; 8 threads cover a row.
__global__ void __launch_bounds__(256) kv_append_nvfp4_kernel(AppendParams p) {
  constexpr int kBlocks = kHeadDim / 16;
  const int64_t total = p.num_tokens * p.hkv * kBlocks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < total; i += stride) {
    const int64_t row = i / kBlocks;  // token * hkv + head
    const int b = static_cast<int>(i % kBlocks);
    const int64_t t = row / p.hkv;
    const int h = static_cast<int>(row % p.hkv);
    const int64_t slot = p.slots[t];
    if (slot < 0) continue;
    const int64_t blk = slot / p.bs;
    if (blk >= p.num_blocks) {
      record_error(p.err, kErrBadSlot);
      continue;
    }
    const int64_t tile = (blk * p.hkv + h) * p.bs * kNvfp4RowBytes;
    int64_t co, mo;
    nvfp4_row_offsets(p.bs, slot % p.bs, &co, &mo);
    const size_t si = static_cast<size_t>(blk) * p.hkv + h;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const uint4 *src = reinterpret_cast<const uint4 *>(kv ? p.v_new : p.k_new) +
                         row * (kHeadDim / 8) + 2 * b;
      uint32_t ms;
      const uint2 c = nvfp4_quantize16(__ldg(src), __ldg(src + 1),
                                       __ldg((kv ? p.v_scale : p.k_scale) + si), &ms);
      uint8_t *pool = static_cast<uint8_t *>(kv ? p.v_cache : p.k_cache) + tile;
      *reinterpret_cast<uint2 *>(pool + co + 8 * b) = c;
      pool[mo + b] = static_cast<uint8_t>(ms);
    }
  }
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

// Rotary position embedding fused with the append (the KV write and RoPE
// run in one kernel in the pages' first per-layer kernel: page "vLLM
// Agentic 推理｜面向 Agent 负载的推理优化", section 5.2, K1).  A CTA handles one
// token; each warp handles whole 128-element rows (q heads, then K heads,
// then V heads), 4 elements per lane.  Pairs rotate by the angle of the
// token's position: NEOX pairs element i with i + 64, otherwise 2i with
// 2i + 1 (pair index i in 0..63 either way).  Rotation runs in fp32 and is
// rounded to bf16, which is also what an FP8 pool quantises.
__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <int FMT, bool NEOX>
__global__ void __launch_bounds__(256) rope_append_kernel(RopeAppendParams rp) {
  const AppendParams &p = rp.a;
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pos = __ldg(rp.positions + t);
  if (pos < 0 || pos >= rp.max_pos) {
    if (threadIdx.x == 0) record_error(p.err, kErrBadPosition);
    return;
  }
  const int64_t slot = p.slots[t];
  const int64_t blk = slot >= 0 ? slot / p.bs : -1;
  if (slot >= 0 && blk >= p.num_blocks && threadIdx.x == 0) record_error(p.err, kErrBadSlot);
  const bool write_kv = slot >= 0 && blk < p.num_blocks;
  // this lane's 4 elements e = 4 lane + j and their pair indices
  const float *cs = rp.cos_sin + pos * kHeadDim;
  float c[4], sn[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * lane + j;
    const int i = NEOX ? (e & 63) : (e >> 1);
    c[j] = __ldg(cs + i);
    sn[j] = __ldg(cs + 64 + i);
  }
  auto rotate = [&](uint2 w, float (&y)[4]) {
    float x[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
    float xp[4];
    if (NEOX) {   // partner of element e is e ^ 64: lane ^ 16, same j
#pragma unroll
      for (int j = 0; j < 4; ++j) xp[j] = __shfl_xor_sync(0xffffffffu, x[j], 16);
    } else {
      xp[0] = x[1]; xp[1] = x[0]; xp[2] = x[3]; xp[3] = x[2];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * lane + j;
      const bool second = NEOX ? (e >= 64) : (e & 1);
      // first of a pair: x cos - x' sin; second: x cos + x' sin
      y[j] = fmaf(x[j], c[j], second ? xp[j] * sn[j] : -(xp[j] * sn[j]));
    }
  };
  const int rows = rp.hq + 2 * p.hkv;
  for (int r = warp; r < rows; r += blockDim.x >> 5) {
    if (r < rp.hq) {
      uint2 *qrow = reinterpret_cast<uint2 *>(rp.q + (t * rp.hq + r) * kHeadDim);
      float y[4];
      rotate(qrow[lane], y);
      qrow[lane] = make_uint2(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]));
      continue;
    }
    const bool is_k = r < rp.hq + p.hkv;
    const int h = is_k ? r - rp.hq : r - rp.hq - p.hkv;
    const int64_t row = t * p.hkv + h;
    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(is_k ? p.k_new : p.v_new) +
                          row * (kHeadDim / 4) + lane);
    float y[4];
    if (is_k) {
      rotate(w, y);   // whole warp (the shuffle needs every lane)
    } else {
      y[0] = bf16_lo(w.x); y[1] = bf16_hi(w.x); y[2] = bf16_lo(w.y); y[3] = bf16_hi(w.y);
    }
    if constexpr (FMT == PKV_KV_NVFP4) {
      // a micro block is 4 lanes (16 elements); the amax reduction needs
      // every lane of the warp, so it runs before the write_kv exit
      float xr[4];
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xr[j] = bf16_round(y[j]);
        amax = fmaxf(amax, fabsf(xr[j]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      if (!write_kv) continue;
      const float sc = __ldg((is_k ? p.k_scale : p.v_scale) + static_cast<size_t>(blk) * p.hkv + h);
      const uint32_t ms = nvfp4_micro_scale(amax, sc);
      const float step = __fmul_rn(sc, e4m3_value(ms));
      uint32_t w = 0;
      if (step != 0.f) {
#pragma unroll
        for (int j = 0; j < 4; ++j) w |= e2m1_code(__fdiv_rn(xr[j], step)) << (4 * j);
      }
      int64_t co, mo;
      nvfp4_row_offsets(p.bs, slot % p.bs, &co, &mo);
      uint8_t *pool = static_cast<uint8_t *>(is_k ? p.k_cache : p.v_cache) +
                      (blk * p.hkv + h) * p.bs * kNvfp4RowBytes;
      *reinterpret_cast<uint16_t *>(pool + co + 2 * lane) = static_cast<uint16_t>(w);
      if ((lane & 3) == 0) pool[mo + (lane >> 2)] = static_cast<uint8_t>(ms);
      continue;
    }
    if (!write_kv) continue;
    const size_t dst = (static_cast<size_t>(blk) * p.hkv + h) * p.bs + slot % p.bs;
    void *pool = is_k ? p.k_cache : p.v_cache;
    if constexpr (FMT == PKV_KV_BF16) {
      reinterpret_cast<uint2 *>(pool)[dst * (kHeadDim / 4) + lane] =
          make_uint2(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]));
    } else {
      const float sc = __ldg((is_k ? p.k_scale : p.v_scale) + static_cast<size_t>(blk) * p.hkv + h);
      const uint16_t a = cvt_e4m3x2(__fdiv_rn(bf16_round(y[0]), sc), __fdiv_rn(bf16_round(y[1]), sc));
      const uint16_t b = cvt_e4m3x2(__fdiv_rn(bf16_round(y[2]), sc), __fdiv_rn(bf16_round(y[3]), sc));
      reinterpret_cast<uint32_t *>(pool)[dst * (kHeadDim / 4) + lane] =
          static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
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
    if (b < 0 || b >= p.num_blocks) {
      record_error(p.err, kErrBadBlock);
    } else if (p.k_scale != nullptr) {
      for (int h = 0; h < p.hkv; ++h) {
        const int64_t si = static_cast<int64_t>(b) * p.hkv + h;
        if (!(p.k_scale[si] <= kQuantScaleMax) || !(p.v_scale[si] <= kQuantScaleMax))
          record_error(p.err, kErrBadScale);
      }
    }
  }
}

// Self-test of the bounded waits: one thread waits, through mbar_wait, on
// an mbarrier that nothing arrives at and no copy or MMA completes, so the
// wait runs out after limit_ns and the timeout is recorded like any other.
__global__ void wait_selftest_kernel(int32_t *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  fence_mbar_init();
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) record_error(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t *err, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_rope_append(const RopeAppendParams &p, int kv_dtype, bool neox,
                               cudaStream_t s) {
  if (p.a.num_tokens == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(p.a.num_tokens);
  switch (kv_dtype * 2 + (neox ? 1 : 0)) {
    case 0: rope_append_kernel<PKV_KV_BF16, false><<<grid, 256, 0, s>>>(p); break;
    case 1: rope_append_kernel<PKV_KV_BF16, true><<<grid, 256, 0, s>>>(p); break;
    case 2: rope_append_kernel<PKV_KV_FP8_E4M3, false><<<grid, 256, 0, s>>>(p); break;
    case 3: rope_append_kernel<PKV_KV_FP8_E4M3, true><<<grid, 256, 0, s>>>(p); break;
    case 4: rope_append_kernel<PKV_KV_NVFP4, false><<<grid, 256, 0, s>>>(p); break;
    default: rope_append_kernel<PKV_KV_NVFP4, true><<<grid, 256, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams &p, int kv_dtype, cudaStream_t s) {
  const bool nvfp4 = kv_dtype == PKV_KV_NVFP4;
  const bool fp8 = kv_dtype == PKV_KV_FP8_E4M3;
  const int64_t total = p.num_tokens * p.hkv * (kHeadDim / (nvfp4 ? 16 : 8));
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + 255) / 256;
  const int blocks = static_cast<int>(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
  if (nvfp4)
    kv_append_nvfp4_kernel<<<blocks, 256, 0, s>>>(p);
  else if (fp8)
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
