// Incremental-prefill attention over a paged KV cache (warp-MMA version).
//
// l_incr new query tokens of a request attend to its l_hist cached tokens and
// to themselves (page "AMPD：PD 分离遇上多轮推理，incremental prefill 到底该在哪跑",
// sections 1 and 3): query token t sits at position l_hist + t and sees keys
// 0 .. l_hist + t.  A work item is (request, KV head, 64 query rows), where
// row r = t * G + g packs the G query heads sharing the KV head (GQA, page
// "vLLM Agentic 推理｜面向 Agent 负载的推理优化", section 4.3.1), so each K/V
// tile is read once for the whole group.  One producer warp streams 64-key
// K/V tiles through a 3-stage shared-memory ring with TMA (one 2D box per
// block and 64-column half, 128-byte swizzled); four consumer warps each own
// 16 rows and run S = Q K^T and O += P V as m16n8k16 bf16 MMAs with an
// online softmax in registers.  The causal mask is applied only on tiles
// that reach past a row's position.
#include <math_constants.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr float kLn2f = 0.6931471805599453f;
constexpr int kPfConsumers = 4;
constexpr int kPfThreads = (kPfConsumers + 1) * 32;
constexpr int kPfHalfBytes = kPfKeys * 128;   // one 64-column half of a tile
constexpr int kPfTileBytes = 2 * kPfHalfBytes;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kPfThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap,
                   const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kPfStages * kPfStageBytes);
  uint64_t *empty = full + kPfStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const pkv_work_item it = p.items[blockIdx.x];
  const int kv_end = it.k_end;
  const int n_tiles = (kv_end + kPfKeys - 1) / kPfKeys;

  if (threadIdx.x < kPfStages) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], kPfConsumers);
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  fence_mbar_init();
  __syncthreads();

  if (warp == kPfConsumers) {
    // ---------------- producer warp: TMA loads of K/V tiles ----------------
    if (lane != 0) return;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride;
    const int br = p.bs < kPfKeys ? p.bs : kPfKeys;
    for (int i = 0; i < n_tiles; ++i) {
      const int slot = i % kPfStages;
      if (i >= kPfStages) {
        if (!mbar_wait(&empty[slot], ((i / kPfStages) - 1) & 1)) {
          record_error(p.err, kErrTimeout);
          return;
        }
      }
      uint8_t *kdst = smem + slot * kPfStageBytes;
      uint8_t *vdst = kdst + kPfTileBytes;
      const int key0 = i * kPfKeys;
      int boxes = 0;
      for (int r = 0; r < kPfKeys; r += br)
        if (key0 + r < kv_end) ++boxes;
      mbar_arrive_expect_tx(&full[slot], boxes * br * 128 * 4);
      for (int r = 0; r < kPfKeys; r += br) {
        const int key = key0 + r;
        if (key >= kv_end) break;
        const int32_t blk = __ldg(bt + key / p.bs);
        int32_t y = p.rows_total;
        if (blk >= 0 && blk < p.num_blocks)
          y = (blk * p.hkv + it.kv_head) * p.bs + key % p.bs;
        else
          record_error(p.err, kErrBadBlock);
        tma_load_2d(kdst + r * 128, &kmap, 0, y, &full[slot]);
        tma_load_2d(kdst + kPfHalfBytes + r * 128, &kmap, 64, y, &full[slot]);
        tma_load_2d(vdst + r * 128, &vmap, 0, y, &full[slot]);
        tma_load_2d(vdst + kPfHalfBytes + r * 128, &vmap, 64, y, &full[slot]);
      }
    }
    return;
  }

  // ---------------- consumer warps: 16 query rows each ----------------
  const int g = lane >> 2;
  const int t = lane & 3;
  const int group = p.group;
  const int rb = it.row0 + 16 * warp;         // first row of this warp
  const int row_end = it.row0 + it.n_rows;
  const int rA = rb + g, rB = rb + g + 8;
  const bool okA = rA < row_end, okB = rB < row_end;
  auto qrow = [&](int r) {
    return p.q + (static_cast<int64_t>(it.tok0 + r / group) * p.hq +
                  it.kv_head * group + r % group) * kHeadDim;
  };
  uint32_t qa[8][4];
  {
    const __nv_bfloat16 *qA = qrow(okA ? rA : it.row0);
    const __nv_bfloat16 *qB = qrow(okB ? rB : it.row0);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d = 16 * ks + 2 * t;
      qa[ks][0] = okA ? __ldg(reinterpret_cast<const uint32_t *>(qA + d)) : 0u;
      qa[ks][1] = okB ? __ldg(reinterpret_cast<const uint32_t *>(qB + d)) : 0u;
      qa[ks][2] = okA ? __ldg(reinterpret_cast<const uint32_t *>(qA + d + 8)) : 0u;
      qa[ks][3] = okB ? __ldg(reinterpret_cast<const uint32_t *>(qB + d + 8)) : 0u;
    }
  }
  // positions; padded rows see every key (their output is never written)
  const int posA = okA ? it.hist + rA / group : 0x7fffffff;
  const int posB = okB ? it.hist + rB / group : 0x7fffffff;
  const int pos_min = posA < posB ? posA : posB;

  float mA = -CUDART_INF_F, mB = -CUDART_INF_F, lA = 0.f, lB = 0.f;
  float acc[16][4];
#pragma unroll
  for (int dn = 0; dn < 16; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;
  const float sc = p.scale_log2;
  const int mi = lane >> 3;
  const int lr = lane & 7;

  for (int i = 0; i < n_tiles; ++i) {
    const int slot = i % kPfStages;
    const bool ok = mbar_wait(&full[slot], (i / kPfStages) & 1);
    if (!__all_sync(0xffffffffu, ok)) {
      record_error(p.err, kErrTimeout);
      return;
    }
    const uint32_t kbase = smem_addr(smem + slot * kPfStageBytes);
    const uint32_t vbase = kbase + kPfTileBytes;
    const int key0 = i * kPfKeys;

    // ---- S = Q K^T : 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        // matrices: (ks=2kp, d lo), (2kp, d hi), (2kp+1, lo), (2kp+1, hi)
        const int d = 32 * kp + 8 * mi;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + (d >> 6) * kPfHalfBytes + swz128(nt * 8 + lr, (d & 63) >> 3),
                b0, b1, b2, b3);
        mma_bf16(s[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
        mma_bf16(s[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2],
                 qa[2 * kp + 1][3], b2, b3);
      }
    }
    // ---- scale + causal mask (only where the tile reaches past a position)
    const bool need_mask = key0 + kPfKeys - 1 > pos_min || key0 + kPfKeys > kv_end;
    float tmA = -CUDART_INF_F, tmB = -CUDART_INF_F;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v = s[nt][c] * sc;
        if (need_mask) {
          const int key = key0 + nt * 8 + 2 * t + (c & 1);
          const int pos = (c < 2) ? posA : posB;
          if (key > pos || key >= kv_end) v = -CUDART_INF_F;
        }
        s[nt][c] = v;
      }
      tmA = fmaxf(tmA, fmaxf(s[nt][0], s[nt][1]));
      tmB = fmaxf(tmB, fmaxf(s[nt][2], s[nt][3]));
    }
    tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 1));
    tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 2));
    tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 1));
    tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 2));
    const float mnA = fmaxf(mA, tmA), mnB = fmaxf(mB, tmB);
    const float muA = mnA == -CUDART_INF_F ? 0.f : mnA;
    const float muB = mnB == -CUDART_INF_F ? 0.f : mnB;
    const float alA = ex2(mA - muA), alB = ex2(mB - muB);
    mA = mnA;
    mB = mnB;
    float sumA = 0.f, sumB = 0.f;
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = ex2(s[nt][0] - muA), p1 = ex2(s[nt][1] - muA);
      const float p2 = ex2(s[nt][2] - muB), p3 = ex2(s[nt][3] - muB);
      sumA += p0 + p1;
      sumB += p2 + p3;
      // A fragment of P for keys 16*(nt/2) .. : nt even -> a0/a1, odd -> a2/a3
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    lA = lA * alA + sumA;
    lB = lB * alB + sumB;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      acc[dn][0] *= alA;
      acc[dn][1] *= alA;
      acc[dn][2] *= alB;
      acc[dn][3] *= alB;
    }
    // ---- O += P V  (V rows of keys past kv_end may hold anything: zero them)
    const bool tail = key0 + kPfKeys > kv_end;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
      if (tail) {
        const int ka = key0 + 16 * kk + 2 * t;
        mlo = (ka < kv_end ? 0x0000FFFFu : 0u) | (ka + 1 < kv_end ? 0xFFFF0000u : 0u);
        mhi = (ka + 8 < kv_end ? 0x0000FFFFu : 0u) | (ka + 9 < kv_end ? 0xFFFF0000u : 0u);
      }
      const int key = 16 * kk + (mi & 1) * 8 + lr;
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        // matrices: (keys lo, d-tile 2dp), (keys hi, 2dp), (lo, 2dp+1), (hi, 2dp+1)
        const int d = 8 * (2 * dp + (mi >> 1));
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vbase + (d >> 6) * kPfHalfBytes + swz128(key, (d & 63) >> 3),
                      v0, v1, v2, v3);
        // a0/a1 = rows g / g+8 keys 2t.., a2/a3 = keys 2t+8..
        mma_bf16(acc[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], v0 & mlo, v1 & mhi);
        mma_bf16(acc[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], v2 & mlo,
                 v3 & mhi);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // ---- normalise and write
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const float invA = lA > 0.f ? 1.f / lA : 0.f;
  const float invB = lB > 0.f ? 1.f / lB : 0.f;
  if (okA) {
    const int64_t row = static_cast<int64_t>(it.tok0 + rA / group) * p.hq +
                        it.kv_head * group + rA % group;
    uint32_t *o = reinterpret_cast<uint32_t *>(p.out + row * kHeadDim);
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
      o[(8 * dn + 2 * t) >> 1] = pack_bf16(acc[dn][0] * invA, acc[dn][1] * invA);
    if (t == 0 && p.lse != nullptr)
      p.lse[row] = lA > 0.f ? (mA + log2f(lA)) * kLn2f : -CUDART_INF_F;
  }
  if (okB) {
    const int64_t row = static_cast<int64_t>(it.tok0 + rB / group) * p.hq +
                        it.kv_head * group + rB % group;
    uint32_t *o = reinterpret_cast<uint32_t *>(p.out + row * kHeadDim);
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
      o[(8 * dn + 2 * t) >> 1] = pack_bf16(acc[dn][2] * invB, acc[dn][3] * invB);
    if (t == 0 && p.lse != nullptr)
      p.lse[row] = lB > 0.f ? (mB + log2f(lB)) * kLn2f : -CUDART_INF_F;
  }
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const PrefillParams &p, int num_items, cudaStream_t s) {
  if (num_items == 0) return cudaSuccess;
  prefill_kernel<<<num_items, kPfThreads, kPfSmemBytes, s>>>(kmap, vmap, p);
  return cudaGetLastError();
}

cudaError_t configure_prefill() {
  return cudaFuncSetAttribute(prefill_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kPfSmemBytes);
}

}  // namespace pkv
