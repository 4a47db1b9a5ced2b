// Incremental-prefill attention on the 5th-generation tensor cores (tcgen05,
// accumulators in TMEM).
//
// l_incr new query tokens attend to l_hist cached tokens plus themselves
// (page "AMPD：PD 分离遇上多轮推理，incremental prefill 到底该在哪跑",
// sections 1 and 3).  A work item is (request, KV head, 128 query rows),
// where row r = t * G + g packs the G query heads of the KV head's group
// (GQA, page "vLLM Agentic 推理｜面向 Agent 负载的推理优化", section 4.3.1),
// so each 128-key K/V tile feeds all of them.
//
// Roles (192 threads, one CTA per SM):
//   warp 5      TMA producer: the Q tile (one 3D box per 64-column half) and
//               K/V tiles of 128 keys (one 2D box per block and half) into a
//               2-stage ring, 128-byte swizzled.
//   warp 4      one thread issues tcgen05.mma: S_j = Q K_j^T into one of two
//               TMEM S buffers (128 x 128 fp32), then O += P_{j-1} V_{j-1}
//               into the TMEM O accumulator; completion is signalled with
//               tcgen05.commit on mbarriers.  QK of tile j overlaps the
//               softmax of tile j-1.
//   warps 0-3   softmax: thread r owns row r (TMEM lane r), reads its 128
//               scores with tcgen05.ld, masks causally on diagonal tiles,
//               keeps a running max in log2 units that is only moved when it
//               grows by more than 8 (so O is rescaled rarely), writes P as
//               bf16 into swizzled shared memory, and finally normalises O.
#include <math_constants.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kTcThreads = 192;
constexpr uint32_t kHalf = 128 * 128;             // one 64-column half of a 128-row tile
constexpr uint32_t kTile = 2 * kHalf;             // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kTile;                // 2 stages of K then V
constexpr uint32_t kStage = 2 * kTile;
constexpr uint32_t kOffP = kOffKV + 2 * kStage;   // 2 P buffers
constexpr uint32_t kOffBar = kOffP + 2 * kTile;   // 229376
constexpr uint32_t kTmemCols = 512;               // S0, S1, O (+ spare)
constexpr uint32_t kIdescQK = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 0, 1);
constexpr float kRescaleThreshold = 8.f;          // log2 units
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b,
                                       uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *q_full = bars + 0;
  uint64_t *kv_full = bars + 1;   // [2]
  uint64_t *kv_empty = bars + 3;  // [2]
  uint64_t *s_full = bars + 5;    // [2]
  uint64_t *s_free = bars + 7;    // [2]
  uint64_t *p_full = bars + 9;    // [2]
  uint64_t *o_done = bars + 11;   // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 13);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const pkv_work_item it = p.items[blockIdx.x];
  const int G = p.group;
  const int k_end = it.k_end;
  const int n_tiles = (k_end + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  if (warp == 4) tmem_alloc(tmem_slot, kTmemCols);
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 5) {
    // ---------------- TMA producer (whole warp) ----------------
    // Lane i holds the block id of box i of the next tile, loaded one tile
    // ahead so table reads never sit between TMA issues; lane 0 issues.
    const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride;
    const int br = p.bs < 128 ? p.bs : 128;
    const int nbox = 128 / br;  // <= 8
    auto load_ids = [&](int j) {
      const int key = j * 128 + lane * br;
      return (lane < nbox && j < n_tiles && key < k_end) ? __ldg(bt + key / p.bs) : -1;
    };
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, kTile);
      const int t0 = it.tok0 + it.row0 / G;
      tma_load_3d(smem + kOffQ, &qmap, 0, it.kv_head * G, t0, q_full);
      tma_load_3d(smem + kOffQ + kHalf, &qmap, 64, it.kv_head * G, t0, q_full);
    }
    int32_t ids = load_ids(0);
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j & 1;
      const int32_t next_ids = load_ids(j + 1);
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&kv_empty[s], ((j >> 1) - 1) & 1))) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      const int key0 = j * 128;
      int32_t yv = p.rows_total;
      if (lane < nbox && key0 + lane * br < k_end) {
        if (ids >= 0 && ids < p.num_blocks)
          yv = (ids * p.hkv + it.kv_head) * p.bs + (key0 + lane * br) % p.bs;
        else
          record_error(p.err, kErrBadBlock);
      }
      int boxes = 0;
      for (int r = 0; r < 128; r += br)
        if (key0 + r < k_end) ++boxes;
      uint8_t *kdst = smem + kOffKV + s * kStage;
      uint8_t *vdst = kdst + kTile;
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[s], boxes * br * 128 * 4);
      for (int bx = 0; bx < boxes; ++bx) {
        const int32_t y = __shfl_sync(0xffffffffu, yv, bx);
        if (lane == 0) {
          const int r = bx * br;
          tma_load_2d(kdst + r * 128, &kmap, 0, y, &kv_full[s]);
          tma_load_2d(kdst + kHalf + r * 128, &kmap, 64, y, &kv_full[s]);
          tma_load_2d(vdst + r * 128, &vmap, 0, y, &kv_full[s]);
          tma_load_2d(vdst + kHalf + r * 128, &vmap, 64, y, &kv_full[s]);
        }
      }
      ids = next_ids;
    }
  } else if (warp == 4) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0) {
      const uint32_t qa = smem_addr(smem + kOffQ);
      bool ok = mbar_wait(q_full, 0);
      auto issue_pv = [&](int i) {
        const int b = i & 1;
        if (!mbar_wait(&p_full[b], (i >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t pa = smem_addr(smem + kOffP + b * kTile);
        const uint32_t va = smem_addr(smem + kOffKV + b * kStage + kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc_sw128(pa + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(va + kk * 2048, kHalf, 1024);
          tc_mma(tmem + 256, ad, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&o_done[b]);
        tc_commit(&kv_empty[b]);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j & 1;
        ok = mbar_wait(&kv_full[s], (j >> 1) & 1);
        if (ok && j >= 2) ok = mbar_wait(&s_free[s], ((j >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = smem_addr(smem + kOffKV + s * kStage);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
          tc_mma(tmem + s * 128, smem_desc_sw128(qa + off, 16, 1024),
                 smem_desc_sw128(ka + off, 16, 1024), kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[s]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) record_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- softmax / epilogue: thread r owns row r ----------------
    const int r = threadIdx.x;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int rowg = it.row0 + r;
    const bool row_ok = r < it.n_rows;
    const int pos = it.hist + rowg / G;   // padded rows see every key
    const float c = p.scale_log2;
    float m = -CUDART_INF_F;              // running max, log2 units
    float l = 0.f;
    bool ok = true;
    // TMEM loads and stores are .sync.aligned: every decision that guards
    // one is made warp-uniform (__all_sync / __any_sync).
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[32];
        tmem_ld32(lane_addr + b * 128 + 32 * q, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * q + i] = v[i];
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);

      const int key0 = j * 128;
      if (key0 + 127 > pos) {
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (key0 + k > pos) s[k] = -CUDART_INF_F;
      }
      float mt = s[0];
#pragma unroll
      for (int k = 1; k < 128; ++k) mt = fmaxf(mt, s[k]);
      const float mt2 = mt * c;
      float alpha = 1.f;
      bool rescale = false;
      if (mt2 > m + kRescaleThreshold) {
        alpha = ex2(m - mt2);
        rescale = j > 0;
        m = mt2;
      }
      // P buffer b is free once PV of tile j-2 has completed
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&o_done[b], ((j >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      const uint32_t pbase = smem_addr(smem + kOffP + b * kTile);
      float sum = 0.f;
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        float e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          e[i] = ex2(fmaf(s[8 * cc + i], c, -m));
          sum += e[i];
        }
        sts128(pbase + (cc >> 3) * kHalf + swz128(r, cc & 7), pack_bf16(e[0], e[1]),
               pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]), pack_bf16(e[6], e[7]));
      }
      l = l * alpha + sum;
      if (__any_sync(0xffffffffu, rescale)) {
        // the whole warp rescales (alpha is 1 on rows whose max held); O
        // must not be written by PV of tile j-1 meanwhile
        if (!rescale) alpha = 1.f;
        if (!__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[32];
          tmem_ld32(lane_addr + 256 + 32 * q, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(lane_addr + 256 + 32 * q, v);
        }
        tmem_wait_st();
      }
      if (j == n_tiles - 1) {
        // V rows past the last key may hold anything: zero them for PV
        const int vvalid = k_end - key0;
        if (r >= vvalid) {
          const uint32_t vrow = smem_addr(smem + kOffKV + b * kStage + kTile) + r * 128;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 8; ++q) sts128(vrow + h * kHalf + 16 * q, 0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    // ---- epilogue: O / l -> bf16
    const int J = n_tiles - 1;
    if (__all_sync(0xffffffffu, ok && mbar_wait(&o_done[J & 1], (J >> 1) & 1))) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow = static_cast<int64_t>(it.tok0 + rowg / G) * p.hq +
                           it.kv_head * G + rowg % G;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[32];
        tmem_ld32(lane_addr + 256 + 32 * q, v);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[4 * q + i] = make_uint4(pack_bf16(v[8 * i] * inv, v[8 * i + 1] * inv),
                                        pack_bf16(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                        pack_bf16(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                        pack_bf16(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
        }
      }
      if (row_ok && p.lse != nullptr)
        p.lse[orow] = l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
    } else {
      record_error(p.err, kErrTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

constexpr uint32_t kTcSmemBytes = kOffBar + 256 + 1024;

cudaError_t launch_prefill_tc(const CUtensorMap &qmap, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, const PrefillParams &p,
                              int num_items, cudaStream_t s) {
  if (num_items == 0) return cudaSuccess;
  prefill_tc_kernel<<<num_items, kTcThreads, kTcSmemBytes, s>>>(qmap, kmap, vmap, p);
  return cudaGetLastError();
}

cudaError_t configure_prefill_tc() {
  return cudaFuncSetAttribute(prefill_tc_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kTcSmemBytes);
}

}  // namespace pkv
