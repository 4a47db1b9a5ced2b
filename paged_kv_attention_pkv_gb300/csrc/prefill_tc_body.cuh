// Incremental-prefill work item on tcgen05 (device code shared by the
// prefill kernel and the one-launch mixed-step kernel).  See prefill_tc.cu
// for what it computes and how the roles divide the work.
#pragma once

#include <math_constants.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {


// 12 warps: softmax warpgroups 0-1 (warps 0-7), then warp 8 (MMA issue,
// TMEM owner), warp 9 (TMA producer) and two idle warps completing
// warpgroup 2, so registers can move between warpgroups (setmaxnreg): the
// launch gives every thread 168; warpgroup 2 drops to kRegsCtl and the
// softmax warpgroups rise to kRegsSoftmax (2 x 128 x 216 + 128 x 72 =
// 384 x 168, the registers the CTA was launched with; neither side spills).
constexpr int kTcThreads = 384;
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsCtl = 72;
constexpr uint32_t kRegsSoftmax = 216;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsCtl == kTcThreads * kRegsLaunch,
              "register split must use exactly the launch's registers");
constexpr int kKst = 2;                           // K ring depth
constexpr int kVst = 3;                           // V ring depth
constexpr uint32_t kHalf = 128 * 128;             // one 64-column half of a 128-row tile
constexpr uint32_t kTile = 2 * kHalf;             // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kOffQ = 0;                     // 2 Q tiles
constexpr uint32_t kOffK = 2 * kTile;             // kKst K tiles
constexpr uint32_t kOffV = kOffK + kKst * kTile;  // kVst V tiles
constexpr uint32_t kOffBar = kOffV + kVst * kTile;   // 229376
static_assert(kOffBar == 229376, "Q, K and V tiles fill 224 KB");
// E4M3 pools: K tiles stay E4M3 (16 KB: 128 keys x 128 bytes) and feed FP8
// MMAs; V tiles arrive as E4M3 in a 2-deep staging ring and are converted to
// f16 (times their block scale) into the same 32 KB V ring.
constexpr uint32_t kTile8 = 128 * 128;
constexpr uint32_t kOffK8 = 2 * kTile;
constexpr uint32_t kOffVs8 = kOffK8 + kKst * kTile8;
constexpr uint32_t kOffV8 = kOffVs8 + 2 * kTile8;
static_assert(kOffV8 + kVst * kTile == kOffBar, "the E4M3 layout fills the same 224 KB");
// NVFP4 pools: K and V tiles arrive as NVFP4 (codes then micro scales per
// group of rows, 9 KB a tile), K into a 2-deep and V into a 1-deep staging
// ring, and are converted to f16 into 2-stage f16 K and V rings.
constexpr uint32_t kStgN = 128 * kNvfp4RowBytes;   // 9216
constexpr uint32_t kOffKn = 2 * kTile;
constexpr uint32_t kOffVn = kOffKn + kKst * kTile;
constexpr int kVstN = 2;
constexpr uint32_t kOffKsN = kOffVn + kVstN * kTile;
constexpr uint32_t kOffVsN = kOffKsN + 2 * kStgN;
static_assert(kOffVsN + kStgN <= kOffBar, "the NVFP4 layout fits the same 224 KB");
// per-tile block scales (K of 8 key groups of 16, then V), a ring of 8 tiles
constexpr uint32_t kOffScales = kOffBar + 512;
constexpr int kScaleRing = 8;
constexpr uint32_t kTmemCols = 512;               // S0, S1, O0, O1
constexpr uint32_t kIdescQK = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 0, 1);
constexpr uint32_t kIdescQK8 = idesc_e4m3(128, 128);
constexpr uint32_t kIdescPV16 = idesc_f16(128, 128, 0, 1);
constexpr uint32_t kIdescQK16 = idesc_f16(128, 128, 0, 0);
constexpr float kRescaleThreshold = 8.f;          // log2 units

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (d0, d1) = (a0 b + c, a1 b + c) and (d0, d1) += (a0, a1) as packed f32x2
// operations (each lane rounds like fmaf / a plain add).
__device__ __forceinline__ void fma2_bc(float &d0, float &d1, float a0, float a1, float b,
                                        float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
      "add.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b,
                                       uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// 64 consecutive fp32 TMEM columns of this thread's lane (one load, wait
// included).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  tmem_ld64x(taddr, v);
}

// One prefill work item processed by all kTcThreads threads of the CTA;
// `smem` is 1024-byte aligned (kTcSmemBytes - 1024 bytes).  FMT is the pool
// format (pkv_kv_dtype): bf16, E4M3 or NVFP4 codes with one fp32 scale per
// (block, KV head); or kFmtStaged, NVFP4 K and V staged as bf16
// (stage_kv.cu): the bf16 data path, with K's block scales (K holds exact
// code values) applied per 16-key group as for the quantised pools; or
// kFmtStagedV, E4M3 K from the pool (FP8 QK as for FMT = E4M3) and V staged
// as bf16 (bf16 PV), no converter warps.
template <int FMT>
__device__ __forceinline__ void prefill_tc_item(const CUtensorMap &qmap,
                                                const CUtensorMap &kmap,
                                                const CUtensorMap &vmap,
                                                const PrefillParams &p,
                                                const pkv_work_item it, uint8_t *smem) {
  constexpr bool FP8 = FMT == PKV_KV_FP8_E4M3;
  constexpr bool NV = FMT == PKV_KV_NVFP4;
  constexpr bool CONV = FP8 || NV;    // converter warps, scale ring, Q converted
  constexpr bool STG = FMT == kFmtStaged;
  constexpr bool HYB = FMT == kFmtStagedV;
  constexpr bool K8 = FP8 || HYB;            // E4M3 K tiles, FP8 QK
  constexpr bool SV = STG || HYB;            // V from the staging pool
  constexpr bool KSC = CONV || STG || HYB;   // K block scales per 16-key group (scale ring)
  constexpr bool QCV = CONV || HYB;          // the softmax warps convert Q first (q_ready)
  constexpr bool QF16 = NV;                  // ... into f16 (QK in f16), else E4M3 hi + lo
  constexpr int VST = NV ? kVstN : kVst;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *q_full = bars + 0;
  uint64_t *k_full = bars + 1;               // [kKst]
  uint64_t *k_empty = k_full + kKst;         // [kKst]
  uint64_t *v_full = k_empty + kKst;         // [kVst]
  uint64_t *v_empty = v_full + kVst;         // [kVst]
  uint64_t *s_full = v_empty + kVst;         // [2] per Q tile
  uint64_t *p_full = s_full + 2;             // [2]
  uint64_t *o_done = p_full + 2;             // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(o_done + 2);
  // E4M3 and NVFP4 pools only
  uint64_t *q_ready = o_done + 3;            // [2] Q tile t converted
  uint64_t *vs_full = q_ready + 2;           // [2] V staging loaded
  uint64_t *vs_empty = vs_full + 2;          // [2] ... and converted
  uint64_t *sc_ready = vs_empty + 2;         // [kScaleRing] tile scales written
  uint64_t *ks_full = sc_ready + kScaleRing; // [2] NVFP4 K staging loaded
  uint64_t *ks_empty = ks_full + 2;          // [2] ... and converted
  float *scales = reinterpret_cast<float *>(smem + kOffScales);   // [ring][16]
  static_assert(8 * (17 + 1 + 2 + 2 + 2 + kScaleRing + 4) <= 512, "barriers fit their 512 bytes");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  // Q tile t holds rows [row0 + 128 t, +n_t) and reaches keys [0, kend_t)
  // a Q tile holds R = G * floor(128 / G) rows (whole tokens); TMEM lanes
  // R .. 127 compute on stale rows that are never stored
  const int R = pf_tile_rows(G);
  const int n0 = it.n_rows < R ? it.n_rows : R;
  const int n1 = it.n_rows - n0;
  const bool two = n1 > 0;
  // This item covers keys [kb, k_end): the whole causal range, or one range
  // of a split item (kb a multiple of 128 and of the block size, at or below
  // every row's position, so each row sees at least one key here).  Local
  // tile j holds keys kb + 128 j ...; the producers and converters count keys
  // from kb (kspan of them) and read the block table from block kb / bs.
  const int kb = it.k_begin;
  const int k_end = it.k_end;
  const int kspan = k_end - kb;
  const int kend0 = min(it.hist + (it.row0 + n0 - 1) / G + 1, k_end);
  const int kend1 = two ? min(it.hist + (it.row0 + R + n1 - 1) / G + 1, k_end) : kend0;
  const int nt0 = (kend0 - kb + 127) / 128;
  const int nt1 = two ? (kend1 - kb + 127) / 128 : 0;
  const int n_tiles = (k_end - kb + 127) / 128;   // = max(nt0, nt1)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kKst; ++i) {
      mbar_init(&k_full[i], NV ? 2 : 1);    // NVFP4: the two converter warps
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kVst; ++i) {
      mbar_init(&v_full[i], CONV ? 2 : 1);  // the two converter warps
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    if (QCV)
      for (int i = 0; i < 2; ++i) mbar_init(&q_ready[i], 128);
    if (CONV) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&vs_full[i], 1);
        mbar_init(&vs_empty[i], 2);
        mbar_init(&ks_full[i], 1);
        mbar_init(&ks_empty[i], 2);
      }
    }
    if (KSC)
      for (int i = 0; i < kScaleRing; ++i) mbar_init(&sc_ready[i], 1);
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  if (warp == 8) tmem_alloc(tmem_slot, kTmemCols);
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
   setmaxnreg_dec<kRegsCtl>();
   if ((!CONV && !HYB && (warp == 9 || warp == 10)) || (HYB && warp == 10)) {
    // ---------------- TMA producers: warp 9 loads Q and K, warp 10 V (only
    // V over E4M3 K, which warp 9 loads as for E4M3 pools) ----
    // Each ring is filled in tile order; K_j waits for the QKs of tile
    // j - kKst, V_j for the PVs of tile j - kVst.  Small blocks take one box
    // per block and 64-column half (16 copies per 128-key tile for 16-token
    // blocks), so K and V are issued by separate warps.  Lane b holds the
    // row of box b of a tile (block ids are read one tile ahead, so table
    // reads never sit between copies); lane 0 issues the copies.
    const bool is_k = warp == 9;
    const CUtensorMap *map = is_k ? &kmap : &vmap;
    const int nst = is_k ? kKst : kVst;
    uint8_t *ring = smem + (is_k ? kOffK : HYB ? kOffV8 : kOffV);
    uint64_t *full = is_k ? k_full : v_full;
    uint64_t *empty = is_k ? k_empty : v_empty;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride + kb / p.bs;
    const int br = p.bs < 128 ? p.bs : 128;
    const int nbox = 128 / br;  // <= 8
    // staged K/V: a request's blocks are consecutive in the staging pool
    const int32_t sbase = SV ? __ldg(p.stage_base + it.seq) + kb / p.bs : -1;
    const int64_t nblk = SV ? p.stage_blocks : p.num_blocks;
    auto tile_rows = [&](int j) {
      const int key = j * 128 + lane * br;
      int32_t y = SV ? p.stage_rows : p.rows_total;
      if (lane < nbox && j < n_tiles && key < kspan) {
        const int32_t blk = SV ? sbase + key / p.bs : __ldg(bt + key / p.bs);
        if (blk >= 0 && blk < nblk)
          y = (blk * p.hkv + it.kv_head) * p.bs + key % p.bs;
        else if (is_k)
          record_error(p.err, kErrBadBlock);
      }
      return y;
    };
    if (is_k && lane == 0) {
      // each box carries R rows of 128 bytes per 64-column half
      mbar_arrive_expect_tx(q_full, (two ? 2 : 1) * 2 * R * 128);
      const int t0 = it.tok0 + it.row0 / G;
      tma_load_3d(smem + kOffQ, &qmap, 0, it.kv_head * G, t0, q_full);
      tma_load_3d(smem + kOffQ + kHalf, &qmap, 64, it.kv_head * G, t0, q_full);
      if (two) {
        const int t1 = t0 + 128 / G;
        tma_load_3d(smem + kOffQ + kTile, &qmap, 0, it.kv_head * G, t1, q_full);
        tma_load_3d(smem + kOffQ + kTile + kHalf, &qmap, 64, it.kv_head * G, t1, q_full);
      }
    }
    // staged K: lane g < 8 holds the block scale of key group g of a tile,
    // loaded one tile ahead (like the box rows) so that no global load sits
    // between the copies
    auto tile_scale = [&](int j) {
      const int key = j * 128 + 16 * lane;
      return (STG && is_k && lane < 8 && j < n_tiles && key < kspan)
                 ? __ldg(p.k_scale + static_cast<int64_t>(sbase + key / p.bs) * p.hkv + it.kv_head)
                 : 1.f;
    };
    float sk_cur = tile_scale(0);
    int32_t y_cur = tile_rows(0);
    for (int j = 0; j < n_tiles; ++j) {
      const int32_t y_next = tile_rows(j + 1);
      const float sk_next = tile_scale(j + 1);
      if (STG && is_k) {
        // tile j's K block scales for the softmax (the ring is 8 tiles deep;
        // this warp runs at most kKst tiles ahead of it)
        if (lane < 8) scales[(j % kScaleRing) * 16 + lane] = sk_cur;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc_ready[j % kScaleRing]);
      }
      sk_cur = sk_next;
      const int s = j % nst;
      if (j >= nst &&
          !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((j / nst) - 1) & 1))) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      uint8_t *dst = ring + s * kTile;
      // boxes holding keys of this item; staged V over E4M3 K takes every
      // box (those past the item's keys start past the pool's last row and
      // arrive as zeros, and the staged rows past a request's context are
      // zeros)
      int n = 0;
      for (int r = 0; r < 128; r += br)
        if ((HYB && !is_k) || j * 128 + r < kspan) ++n;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], n * br * 128 * 2);
      for (int bx = 0; bx < n; ++bx) {
        const int32_t y = __shfl_sync(0xffffffffu, y_cur, bx);
        if (lane == 0) {
          tma_load_2d(dst + bx * br * 128, map, 0, y, &full[s]);
          tma_load_2d(dst + kHalf + bx * br * 128, map, 64, y, &full[s]);
        }
      }
      y_cur = y_next;
    }
   } else if (K8 && warp == 9) {
    // ---------------- TMA producer, E4M3 pools: Q, the E4M3 K ring, the
    // E4M3 V staging ring (one box per block, no column halves), and each
    // tile's block scales for the softmax and the converters; over staged V
    // (warp 10 loads it) Q, K and the K scales ----
    const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride + kb / p.bs;
    const int br = p.bs < 128 ? p.bs : 128;
    const int nbox = 128 / br;  // <= 8
    // lane b < nbox: pool row of box b of tile j, and its block's scales
    auto tile_info = [&](int j, float &sk, float &sv) {
      const int key = j * 128 + lane * br;
      int32_t y = p.rows_total;
      sk = sv = 1.f;
      if (lane < nbox && j < n_tiles && key < kspan) {
        const int32_t blk = __ldg(bt + key / p.bs);
        if (blk >= 0 && blk < p.num_blocks) {
          y = (blk * p.hkv + it.kv_head) * p.bs + key % p.bs;
          const int64_t si = static_cast<int64_t>(blk) * p.hkv + it.kv_head;
          sk = __ldg(p.k_scale + si);
          sv = HYB ? 1.f : __ldg(p.v_scale + si);   // staged V is already scaled
        } else {
          record_error(p.err, kErrBadBlock);
        }
      }
      return y;
    };
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, (two ? 2 : 1) * 2 * R * 128);
      const int t0 = it.tok0 + it.row0 / G;
      tma_load_3d(smem + kOffQ, &qmap, 0, it.kv_head * G, t0, q_full);
      tma_load_3d(smem + kOffQ + kHalf, &qmap, 64, it.kv_head * G, t0, q_full);
      if (two) {
        const int t1 = t0 + 128 / G;
        tma_load_3d(smem + kOffQ + kTile, &qmap, 0, it.kv_head * G, t1, q_full);
        tma_load_3d(smem + kOffQ + kTile + kHalf, &qmap, 64, it.kv_head * G, t1, q_full);
      }
    }
    float sk_cur, sv_cur;
    int32_t y_cur = tile_info(0, sk_cur, sv_cur);
    for (int j = 0; j < n_tiles; ++j) {
      float sk_nxt, sv_nxt;
      const int32_t y_next = tile_info(j + 1, sk_nxt, sv_nxt);
      // scales of the tile's 8 key groups of 16 (group g lies in box g*16/br)
      const int gb = (lane * 16 / br) & 31;
      const float gk = __shfl_sync(0xffffffffu, sk_cur, gb);
      const float gv = __shfl_sync(0xffffffffu, sv_cur, gb);
      if (lane < 8) {
        scales[(j % kScaleRing) * 16 + lane] = gk;
        scales[(j % kScaleRing) * 16 + 8 + lane] = gv;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc_ready[j % kScaleRing]);
      int n = 0;
      for (int r = 0; r < 128; r += br)
        if (j * 128 + r < kspan) ++n;
      // K tile j once the QKs of tile j - kKst are done
      const int s = j % kKst;
      if (j >= kKst &&
          !__all_sync(0xffffffffu, mbar_wait(&k_empty[s], ((j / kKst) - 1) & 1))) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&k_full[s], n * br * 128);
      for (int bx = 0; bx < n; ++bx) {
        const int32_t y = __shfl_sync(0xffffffffu, y_cur, bx);
        if (lane == 0)
          tma_load_2d(smem + kOffK8 + s * kTile8 + bx * br * 128, &kmap, 0, y, &k_full[s]);
      }
      if constexpr (!HYB) {
        // V tile j into staging j & 1 once the converters are done with j - 2
        const int v2 = j & 1;
        if (j >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(&vs_empty[v2], ((j >> 1) - 1) & 1))) {
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&vs_full[v2], n * br * 128);
        for (int bx = 0; bx < n; ++bx) {
          const int32_t y = __shfl_sync(0xffffffffu, y_cur, bx);
          if (lane == 0)
            tma_load_2d(smem + kOffVs8 + v2 * kTile8 + bx * br * 128, &vmap, 0, y, &vs_full[v2]);
        }
      }
      y_cur = y_next;
      sk_cur = sk_nxt;
      sv_cur = sv_nxt;
    }
   } else if (FP8 && warp >= 10) {
    // ---------------- V converters, E4M3 pools: staging -> f16 V ring ----
    // Warp 10 converts key rows 0-63 of a tile, warp 11 rows 64-127; lane l
    // takes rows l and l + 32 of its half (8 consecutive rows per 8-lane
    // phase, which the 128-byte swizzle spreads over all banks).  Codes
    // become f16 exactly; the multiply by the block scale rounds once.
    // Rows past the item's last key are written as zeros (PV multiplies them
    // by P = 0, and stale bytes could be NaN).
    const int rbase = (warp - 10) * 64;
    for (int j = 0; j < n_tiles; ++j) {
      const int v2 = j & 1;
      const int s = j % kVst;
      bool wok = mbar_wait(&vs_full[v2], (j >> 1) & 1);
      if (wok && j >= kVst) wok = mbar_wait(&v_empty[s], ((j / kVst) - 1) & 1);
      if (wok) wok = mbar_wait(&sc_ready[j % kScaleRing], (j / kScaleRing) & 1);
      if (!__all_sync(0xffffffffu, wok)) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      const uint32_t src = smem_addr(smem + kOffVs8 + v2 * kTile8);
      const uint32_t dst = smem_addr(smem + kOffV8 + s * kTile);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = rbase + lane + 32 * i;   // key row in the tile
        const uint32_t sw = k & 7;
        if (j * 128 + k >= kspan) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              sts128(dst + h * kHalf + k * 128 + ((c ^ sw) << 4), 0u, 0u, 0u, 0u);
          continue;
        }
        const float sv = scales[(j % kScaleRing) * 16 + 8 + (k >> 4)];
        const uint32_t sv2 = pack_f16(sv, sv);
#pragma unroll
        for (int oc = 0; oc < 8; ++oc) {   // head dims 16 oc .. 16 oc + 15
          const uint4 x = lds128(src + k * 128 + ((oc ^ sw) << 4));
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            o[2 * q] = hmul2(e4m3x2lo_to_f16x2(w[q]), sv2);
            o[2 * q + 1] = hmul2(e4m3x2hi_to_f16x2(w[q]), sv2);
          }
          // f16 chunks 2(oc & 3) and 2(oc & 3) + 1 of column half oc >> 2
          const uint32_t hb = dst + (oc >> 2) * kHalf + k * 128;
          const uint32_t c0 = 2 * (oc & 3);
          sts128(hb + ((c0 ^ sw) << 4), o[0], o[1], o[2], o[3]);
          sts128(hb + (((c0 + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&v_full[s]);
        mbar_arrive(&vs_empty[v2]);
      }
    }
   } else if (NV && warp == 9) {
    // ---------------- TMA producer, NVFP4 pools: Q, the NVFP4 K staging
    // ring (2 deep), the NVFP4 V staging tile (1 deep), and each tile's block
    // scales.  A group of min(bs, 64) rows is contiguous in the pool (codes
    // then micro scales), so one box of 9/8 rows per row brings both ----
    const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride + kb / p.bs;
    const int gs = p.bs < kNvfp4Group ? p.bs : kNvfp4Group;
    const int ngrp = 128 / gs;  // <= 8
    const int tile_rows = p.bs / 8 * 9, group_rows = gs / 8 * 9;
    // lane b < ngrp: first pool row of group b of tile j, and its scales
    auto tile_info = [&](int j, float &sk, float &sv) {
      const int key = j * 128 + lane * gs;
      int32_t y = p.rows_total;
      sk = sv = 1.f;
      if (lane < ngrp && j < n_tiles && key < kspan) {
        const int32_t blk = __ldg(bt + key / p.bs);
        if (blk >= 0 && blk < p.num_blocks) {
          y = (blk * p.hkv + it.kv_head) * tile_rows + (key % p.bs) / gs * group_rows;
          const int64_t si = static_cast<int64_t>(blk) * p.hkv + it.kv_head;
          sk = __ldg(p.k_scale + si);
          sv = __ldg(p.v_scale + si);
        } else {
          record_error(p.err, kErrBadBlock);
        }
      }
      return y;
    };
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, (two ? 2 : 1) * 2 * R * 128);
      const int t0 = it.tok0 + it.row0 / G;
      tma_load_3d(smem + kOffQ, &qmap, 0, it.kv_head * G, t0, q_full);
      tma_load_3d(smem + kOffQ + kHalf, &qmap, 64, it.kv_head * G, t0, q_full);
      if (two) {
        const int t1 = t0 + 128 / G;
        tma_load_3d(smem + kOffQ + kTile, &qmap, 0, it.kv_head * G, t1, q_full);
        tma_load_3d(smem + kOffQ + kTile + kHalf, &qmap, 64, it.kv_head * G, t1, q_full);
      }
    }
    float sk_cur, sv_cur;
    int32_t y_cur = tile_info(0, sk_cur, sv_cur);
    for (int j = 0; j < n_tiles; ++j) {
      float sk_nxt, sv_nxt;
      const int32_t y_next = tile_info(j + 1, sk_nxt, sv_nxt);
      const int gb = (lane * 16 / gs) & 31;   // group of key group `lane`
      const float gk = __shfl_sync(0xffffffffu, sk_cur, gb);
      const float gv = __shfl_sync(0xffffffffu, sv_cur, gb);
      if (lane < 8) {
        scales[(j % kScaleRing) * 16 + lane] = gk;
        scales[(j % kScaleRing) * 16 + 8 + lane] = gv;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc_ready[j % kScaleRing]);
      int n = 0;
      for (int r = 0; r < 128; r += gs)
        if (j * 128 + r < kspan) ++n;
      // K tile j into staging j & 1 once the converters are done with j - 2
      const int k2 = j & 1;
      if (j >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&ks_empty[k2], ((j >> 1) - 1) & 1))) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&ks_full[k2], n * gs * kNvfp4RowBytes);
      for (int bx = 0; bx < n; ++bx) {
        const int32_t y = __shfl_sync(0xffffffffu, y_cur, bx);
        if (lane == 0)
          tma_load_2d(smem + kOffKsN + k2 * kStgN + bx * gs * kNvfp4RowBytes, &kmap, 0, y,
                      &ks_full[k2]);
      }
      // V tile j into the staging tile once the converters are done with j - 1
      if (j >= 1 &&
          !__all_sync(0xffffffffu, mbar_wait(&vs_empty[0], (j - 1) & 1))) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&vs_full[0], n * gs * kNvfp4RowBytes);
      for (int bx = 0; bx < n; ++bx) {
        const int32_t y = __shfl_sync(0xffffffffu, y_cur, bx);
        if (lane == 0)
          tma_load_2d(smem + kOffVsN + bx * gs * kNvfp4RowBytes, &vmap, 0, y, &vs_full[0]);
      }
      y_cur = y_next;
      sk_cur = sk_nxt;
      sv_cur = sv_nxt;
    }
   } else if (NV && warp >= 10) {
    // ---------------- converters, NVFP4 pools: staging -> f16 K and V rings ----
    // Four lanes share a key row, lane c taking head dims 32c .. 32c + 31 (16
    // code bytes: micro blocks 2c and 2c + 1); warp 10 converts rows 0-63 of
    // a tile, warp 11 rows 64-127, eight rows per pass.  K becomes f16 code x
    // micro scale, exactly (a 2-bit by 4-bit significand product); V becomes
    // f16 code x (micro scale x block scale), rounded once.  Rows past the
    // item's last key are written as zeros.
    const int gs = p.bs < kNvfp4Group ? p.bs : kNvfp4Group;
    const int c = lane & 3;
    const int rbase = (warp - 10) * 64 + (lane >> 2);
    auto convert = [&](uint32_t stg, uint32_t dst, int j, bool is_v) {
#pragma unroll 2
      for (int ps = 0; ps < 8; ++ps) {
        const int k = rbase + 8 * ps;   // key row in the tile
        const uint32_t sw = k & 7;
        uint32_t o[16];
        if (j * 128 + k >= kspan) {
#pragma unroll
          for (int q = 0; q < 16; ++q) o[q] = 0u;
        } else {
          const uint32_t grp = stg + (k / gs) * gs * kNvfp4RowBytes;
          const int r = k % gs;
          const uint4 x = lds128(grp + r * 64 + 16 * c);
          const uint32_t msb = lds16(grp + gs * 64 + r * 8 + 2 * c);
          uint32_t m0, m1;   // (s, s) f16 pairs for micro blocks 2c and 2c + 1
          if (is_v) {
            const float2 ms = e4m3x2_to_f32(msb);
            const float sv = scales[(j % kScaleRing) * 16 + 8 + (k >> 4)];
            m0 = pack_f16(ms.x * sv, ms.x * sv);
            m1 = pack_f16(ms.y * sv, ms.y * sv);
          } else {
            const uint32_t mh = e4m3x2lo_to_f16x2(msb);
            m0 = __byte_perm(mh, 0, 0x1010);
            m1 = __byte_perm(mh, 0, 0x3232);
          }
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t f[4];
            e2m1x8_to_f16x2(w[q], f);
#pragma unroll
            for (int u = 0; u < 4; ++u) o[4 * q + u] = hmul2(f[u], q < 2 ? m0 : m1);
          }
        }
        // f16 row: column half c >> 1, chunks 4 (c & 1) .. + 3
        const uint32_t hb = dst + (c >> 1) * kHalf + k * 128;
        const uint32_t c0 = 4 * (c & 1);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          sts128(hb + (((c0 + q) ^ sw) << 4), o[4 * q], o[4 * q + 1], o[4 * q + 2],
                 o[4 * q + 3]);
      }
    };
    for (int j = 0; j < n_tiles; ++j) {
      const int k2 = j & 1, s = j % kKst, vs = j % kVstN;
      bool wok = mbar_wait(&ks_full[k2], (j >> 1) & 1);
      if (wok && j >= kKst) wok = mbar_wait(&k_empty[s], ((j / kKst) - 1) & 1);
      if (wok) wok = mbar_wait(&sc_ready[j % kScaleRing], (j / kScaleRing) & 1);
      if (!__all_sync(0xffffffffu, wok)) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      convert(smem_addr(smem + kOffKsN + k2 * kStgN), smem_addr(smem + kOffKn + s * kTile), j,
              false);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&k_full[s]);
        mbar_arrive(&ks_empty[k2]);
      }
      wok = mbar_wait(&vs_full[0], j & 1);
      if (wok && j >= kVstN) wok = mbar_wait(&v_empty[vs], ((j / kVstN) - 1) & 1);
      if (!__all_sync(0xffffffffu, wok)) {
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      convert(smem_addr(smem + kOffVsN), smem_addr(smem + kOffVn + vs * kTile), j, true);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&v_full[vs]);
        mbar_arrive(&vs_empty[0]);
      }
    }
   } else if (warp == 8) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0) {
      // E4M3 / NVFP4 pools: the softmax warps first turn Q tile t into E4M3
      // hi/lo parts / scaled f16
      bool ok = QCV ? mbar_wait(&q_ready[0], 0) : mbar_wait(q_full, 0);
      if (QCV) tc_fence_after();
      // Descriptors are built once; tiles, stages and k-steps add constant
      // offsets to the start-address field (addresses stay < 256 KB, so the
      // 14-bit field never carries).  The issuing warp shares its SM
      // sub-partition with two softmax warps: every instruction it issues
      // between MMA groups is time the tensor pipe may sit idle.
      constexpr uint64_t kTileDesc = kTile >> 4;
      const uint64_t qd0 = smem_desc_sw128(smem_addr(smem + kOffQ), 16, 1024);
      const uint64_t kd0 =
          smem_desc_sw128(smem_addr(smem + (NV ? kOffKn : K8 ? kOffK8 : kOffK)), 16, 1024);
      const uint64_t vd0 =
          smem_desc_sw128(smem_addr(smem + (NV ? kOffVn : K8 ? kOffV8 : kOffV)), kHalf, 1024);
      auto qk = [&](int t, int j) {   // S_t = Q_t K_j^T
        const int s = j & (kKst - 1);
        // K arrives by TMA (async proxy, like the MMA): the mbarrier alone
        // orders it; NVFP4 K is written by the converter warps
        if (!mbar_wait(&k_full[s], (j / kKst) & 1)) return false;
        if (NV) tc_fence_after();
        const uint64_t a0 = qd0 + t * kTileDesc;
        const uint32_t d = tmem + t * 128;
        if constexpr (K8) {
          // S = (Q_hi + Q_lo) K^T: E4M3 K codes, four 32-byte k-steps per part
          // (Q_hi in the tile's first half, Q_lo in its second)
          const uint64_t b0 = kd0 + s * (kTile8 >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t off = (ks * 32) >> 4;
            if (ks == 0)
              tc_mma8_first(d, a0, b0, kIdescQK8);
            else
              tc_mma8_acc(d, a0 + off, b0 + off, kIdescQK8);
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t off = (ks * 32) >> 4;
            tc_mma8_acc(d, a0 + (kHalf >> 4) + off, b0 + off, kIdescQK8);
          }
        } else {
          const uint64_t b0 = kd0 + s * kTileDesc;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t off = ((ks >> 2) * kHalf + (ks & 3) * 32) >> 4;
            if (ks == 0)
              tc_mma_first(d, a0, b0, QF16 ? kIdescQK16 : kIdescQK);
            else
              tc_mma_acc(d, a0 + off, b0 + off, QF16 ? kIdescQK16 : kIdescQK);
          }
        }
        tc_commit(&s_full[t]);
        return true;
      };
      auto pv = [&](int t, int j, int s, int vpar) {   // O_t += P_t V_j, V_j in stage s
        if (!mbar_wait(&p_full[t], j & 1)) return false;
        if (!mbar_wait(&v_full[s], vpar)) return false;
        tc_fence_after();
        const uint64_t b0 = vd0 + s * kTileDesc;
        const uint32_t dO = tmem + 256 + t * 128, aP = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = b0 + ((kk * 2048) >> 4);
          if (kk > 0)
            tc_mma_tmem_a_acc(dO, aP + kk * 8, bd, CONV ? kIdescPV16 : kIdescPV);
          else
            tc_mma_tmem_a(dO, aP, bd, CONV ? kIdescPV16 : kIdescPV, j > 0 ? 1u : 0u);
        }
        tc_commit(&o_done[t]);
        return true;
      };
      // prologue: QK of tile 0 for both Q tiles
      if (ok) ok = qk(0, 0);
      if (QCV && ok && two) {
        ok = mbar_wait(&q_ready[1], 0);
        tc_fence_after();
      }
      if (ok && two) ok = qk(1, 0);
      if (ok) tc_commit(&k_empty[0]);
      // P_t(j) lives where QK_t(j+1) writes: QK_t(j+1) is issued after
      // PV_t(j) (tcgen05.mma of one thread execute in order).
      // V_j is released as soon as its last PV is issued, K_{j+1} after its
      // last QK.
      static_assert((kKst & (kKst - 1)) == 0, "K ring depth: a power of two");
      int vs = 0, vpar = 0;   // V_j's stage and its phase parity
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j < nt0) {
          ok = pv(0, j, vs, vpar);
          if (ok && j + 1 < nt0) ok = qk(0, j + 1);
        }
        const bool t1 = two && j < nt1;
        if (ok && t1) ok = pv(1, j, vs, vpar);
        if (!ok) break;
        tc_commit(&v_empty[vs]);
        if (++vs == VST) {
          vs = 0;
          vpar ^= 1;
        }
        if (t1 && j + 1 < nt1) ok = qk(1, j + 1);
        if (!ok) break;
        if (j + 1 < n_tiles) tc_commit(&k_empty[(j + 1) & (kKst - 1)]);
      }
      if (!ok) record_error(p.err, kErrTimeout);
    }
   }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ---------------- softmax / epilogue: thread r of tile t owns row r ----
    const int t = warp >> 2;                   // Q tile of this warpgroup
    const int r = threadIdx.x & 127;
    const int nrow = t == 0 ? n0 : n1;
    const int ntl = t == 0 ? nt0 : nt1;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t col_s = t * 128, col_o = 256 + t * 128;
    const int rowg = it.row0 + R * t + r;
    const bool row_ok = r < nrow;
    // this row's position relative to the item's first key (padded rows
    // see every key)
    const int pos = it.hist + rowg / G - kb;
    float c = p.scale_log2;
    float m = -CUDART_INF_F;              // running max, log2 units
    float l = 0.f;
    bool ok = true;
    if (QCV && ntl > 0) {
      // E4M3 pools: this thread's Q row, scaled by a power of two sq (largest
      // |q sq| in [128, 256)), becomes hi + lo, both E4M3 (about bf16
      // precision), written in place over the row: hi into the tile's first
      // 128-byte half, lo into its second (each the 128B-swizzled K-major
      // layout of a 128 x 128 E4M3 tile); likewise with E4M3 K over staged V.
      // NVFP4 pools: the row becomes f16 in place (largest |q sq| in
      // [2^14, 2^15), the bf16 layout).  1/sq goes into this row's scale.
      ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0));
      if (ok) {
        const uint32_t qt = smem_addr(smem + kOffQ + t * kTile);
        const uint32_t sw = r & 7;
        uint32_t w[64];   // bf16 pairs: dims 2i, 2i + 1 in w[i]
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const uint4 v = lds128(qt + h * kHalf + r * 128 + ((cc ^ sw) << 4));
            w[32 * h + 4 * cc] = v.x;
            w[32 * h + 4 * cc + 1] = v.y;
            w[32 * h + 4 * cc + 2] = v.z;
            w[32 * h + 4 * cc + 3] = v.w;
          }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          amax = fmax3(amax, fabsf(__uint_as_float(w[i] << 16)),
                       fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
        const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
        const int top = QF16 ? 14 : 7;
        const int k2 = top - e < 126 ? top - e : 126;
        const float sq = __uint_as_float(static_cast<uint32_t>(127 + k2) << 23);
        c *= __uint_as_float(static_cast<uint32_t>(127 - k2) << 23);
        if constexpr (QF16) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              uint32_t o[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t wv = w[32 * h + 4 * cc + u];
                o[u] = pack_f16(__uint_as_float(wv << 16) * sq,
                                __uint_as_float(wv & 0xFFFF0000u) * sq);
              }
              sts128(qt + h * kHalf + r * 128 + ((cc ^ sw) << 4), o[0], o[1], o[2], o[3]);
            }
        }
#pragma unroll
        for (int oc = 0; oc < (QF16 ? 0 : 8); ++oc) {   // 16 dims: words 8 oc .. 8 oc + 7
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t hc[2], lc[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t wv = w[8 * oc + 2 * q + u];
              const float x0 = __uint_as_float(wv << 16) * sq;
              const float x1 = __uint_as_float(wv & 0xFFFF0000u) * sq;
              hc[u] = e4m3x2_from_f32(x0, x1);
              const float2 back = e4m3x2_to_f32(hc[u]);
              lc[u] = e4m3x2_from_f32(x0 - back.x, x1 - back.y);
            }
            hi[q] = hc[0] | (hc[1] << 16);
            lo[q] = lc[0] | (lc[1] << 16);
          }
          sts128(qt + r * 128 + ((oc ^ sw) << 4), hi[0], hi[1], hi[2], hi[3]);
          sts128(qt + kHalf + r * 128 + ((oc ^ sw) << 4), lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async();
      }
      mbar_arrive(&q_ready[t]);
    }
    // TMEM loads and stores are .sync.aligned: every decision that guards
    // one is warp-uniform (__all_sync / __any_sync).
    for (int j = 0; j < ntl; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = j * 128;   // relative to kb, like pos
      // one pass: the whole S row in registers (one TMEM load)
      float s[128];
      tmem_ld128(lane_addr + col_s, s);
      if (key0 + 127 > pos) {   // diagonal tile: causal mask
#pragma unroll
        for (int k = 0; k < 128; ++k) {
          const int key = key0 + k;
          s[k] = key > pos ? -CUDART_INF_F : s[k];
        }
      }
      // E4M3 and NVFP4 pools: key group g (16 keys, one block) has its own
      // score scale c * k_scale (positive), so maxima are taken per group
      float cg[8];
      float mt2;
      if constexpr (KSC) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&sc_ready[j % kScaleRing], (j / kScaleRing) & 1))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) cg[g] = c * scales[(j % kScaleRing) * 16 + g];
        mt2 = -CUDART_INF_F;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float* sg = s + 16 * g;
          float a = fmax3(sg[0], sg[1], sg[2]);
          a = fmax3(a, sg[3], sg[4]);
          a = fmax3(a, sg[5], sg[6]);
          a = fmax3(a, sg[7], sg[8]);
          a = fmax3(a, sg[9], sg[10]);
          a = fmax3(a, sg[11], sg[12]);
          a = fmax3(a, sg[13], sg[14]);
          a = fmaxf(a, sg[15]);
          mt2 = fmaxf(mt2, a * cg[g]);
        }
      } else {
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[8 + i]);
#pragma unroll
        for (int k = 16; k < 128; k += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[k + i], s[k + 8 + i]);
        const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                               fmaxf(mx[6], mx[7]));
        mt2 = mt * c;
      }
      float alpha = 1.f;
      bool rescale = false;
      if (mt2 > m + kRescaleThreshold) {
        alpha = ex2(m - mt2);
        rescale = j > 0;
        m = mt2;
      }
      // P = 2^(s c - m) as bf16 pairs over the S columns, in two 64-column
      // chunks (chunk 0's P lands on S columns 0-31, already in registers)
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          float x0, x1;
          fma2_bc(x0, x1, s[64 * hh + 2 * k], s[64 * hh + 2 * k + 1],
                  KSC ? cg[(64 * hh + 2 * k) >> 4] : c, -m);
          const float e0 = ex2(x0), e1 = ex2(x1);
          add2(acc[(2 * k) & 7], acc[(2 * k + 1) & 7], e0, e1);
          // E4M3 and NVFP4 pools run PV in f16 (V converted to f16)
          pk[k] = CONV ? pack_f16(e0, e1) : pack_bf16(e0, e1);
        }
        tmem_st32u(lane_addr + col_s + 32 * hh, pk);
      }
      const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) +
                        ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      l = l * alpha + sum;
      if (__any_sync(0xffffffffu, rescale)) {
        // the whole warp rescales (alpha is 1 on rows whose max held); O
        // must not be written by PV of tile j-1 meanwhile
        if (!rescale) alpha = 1.f;
        if (!__all_sync(0xffffffffu, mbar_wait(&o_done[t], (j - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld128(lane_addr + col_o, s);
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] *= alpha;
        tmem_st128(lane_addr + col_o, s);
      }
      // The last K/V tile may carry V rows past the item's last key (rows
      // of other requests or never loaded): zero them before any PV reads
      // them.  Q tile 0 does it when it reaches that tile (its PV comes
      // first), otherwise Q tile 1.  (E4M3 and NVFP4 pools: the converters write
      // those rows as zeros; staged V over E4M3 K: they arrive as zeros.)
      if (!CONV && !HYB && j == n_tiles - 1 && kspan - key0 < 128 &&
          (t == 0 || nt0 < n_tiles)) {
        const int vvalid = kspan - key0;
        const int vs = j % kVst;
        if (!__all_sync(0xffffffffu, mbar_wait(&v_full[vs], (j / kVst) & 1))) {
          ok = false;
          break;
        }
        if (r >= vvalid) {   // thread r clears the V row of tile-local key r
          const uint32_t vt = smem_addr(smem + kOffV + vs * kTile);
          const uint32_t vrow = vt + r * 128;
          const uint32_t hstep = kHalf;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 8; ++q)   // rotate chunks across rows: no bank conflicts
              sts128(vrow + h * hstep + 16 * ((q + r) & 7), 0u, 0u, 0u, 0u);
        }
        fence_proxy_async();
      }
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    // ---- epilogue: O / l -> bf16; an item split over key ranges writes
    // this range's partial (O / l in fp32, log-sum-exp in log2 units) for
    // prefill_merge_kernel instead
    if (ntl > 0) {
      const int J = ntl - 1;
      if (__all_sync(0xffffffffu, ok && mbar_wait(&o_done[t], J & 1))) {
        tc_fence_after();
        const bool split = it.part >= 0;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t orow = static_cast<int64_t>(it.tok0 + rowg / G) * p.hq +
                             it.kv_head * G + rowg % G;
        // this row's line in the range's partial slot
        const int64_t pline = static_cast<int64_t>(split ? it.part : 0) * kDecCols + t * 128 + r;
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim);
        float4 *pdst = reinterpret_cast<float4 *>(p.part_o + pline * kHeadDim);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[64];
          tmem_ld64(lane_addr + col_o + 64 * hh, v);
          if (row_ok && split) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pdst[16 * hh + i] = make_float4(v[4 * i] * inv, v[4 * i + 1] * inv,
                                              v[4 * i + 2] * inv, v[4 * i + 3] * inv);
          } else if (row_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[8 * hh + i] = make_uint4(pack_bf16(v[8 * i] * inv, v[8 * i + 1] * inv),
                                           pack_bf16(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                           pack_bf16(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                           pack_bf16(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
          }
        }
        const float lse2 = l > 0.f ? m + log2f(l) : -CUDART_INF_F;
        if (row_ok && split)
          p.part_lse[pline] = lse2;
        else if (row_ok && p.lse != nullptr)
          p.lse[orow] = lse2 * kLn2;
      } else {
        record_error(p.err, kErrTimeout);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, kTmemCols);
}


// barriers (256 B), the E4M3 scale ring (8 tiles x 16 fp32), alignment slack
constexpr uint32_t kTcSmemBytes = kOffScales + kScaleRing * 16 * 4 + 1024;
static_assert(kTcSmemBytes <= 232448, "within the 227 KB a CTA may have");

}  // namespace
}  // namespace pkv
