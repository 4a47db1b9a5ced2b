// Split-KV decode work item (device code shared by the decode kernel and the
// one-launch mixed-step kernel).  See decode.cu for what it computes.
#pragma once

#include <type_traits>

#include <math_constants.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {


template <bool FP8>
struct DecTile {
  static constexpr int kKeys = FP8 ? kDecKeysFp8 : kDecKeysBf16;  // per stage
  static constexpr int kSubs = kKeys / 16;
  static constexpr int kKBytes = kKeys * kHeadDim * (FP8 ? 1 : 2);  // 4096
  static_assert(kKBytes * 2 == kDecStageBytes, "stage layout");
};

// log2 of the block size (a power of two).
__device__ __forceinline__ int bs_shift(const DecodeParams &p) { return 31 - __clz(p.bs); }

// Row of the pool maps holding key `key` of KV head `kvh` of a request, or
// rows_total (entirely outside the map: TMA fills zeros) for a bad block id.
__device__ __forceinline__ int32_t pool_row(const int32_t *bt, int32_t key,
                                            int32_t kvh, const DecodeParams &p,
                                            int32_t *blk_out) {
  const int32_t blk = __ldg(bt + (key >> bs_shift(p)));
  *blk_out = blk;
  if (blk < 0 || blk >= p.num_blocks) {
    record_error(p.err, kErrBadBlock);
    return p.rows_total;
  }
  return (blk * p.hkv + kvh) * p.bs + (key & (p.bs - 1));
}

// E4M3 pools: key of MMA key slot r (0..15) of a 16-key sub-tile.  The V^T
// fragments come from an 8-bit transposing ldmatrix, which gives lane
// (g, t) keys 4t .. 4t+3 of a head dim: slots 2t, 2t+1 hold keys 4t, 4t+1
// and slots 2t+8, 2t+9 keys 4t+2, 4t+3, so the QK MMA reads its K rows in
// that order too (slot r of S^T is key fp8_key(r)).
__device__ __forceinline__ int fp8_key(int r) {
  return 4 * ((r & 7) >> 1) + 2 * (r >> 3) + (r & 1);
}

// Global key of an item-local key: the identity, or the shard view (see
// DecodeParams).  Keys of one stage stay consecutive.
__device__ __forceinline__ int32_t global_key(const DecodeParams &p, int32_t x) {
  if (p.dcp_n <= 1 || p.dcp_mask) return x;
  return ((x / p.dcp_k) * p.dcp_n + p.dcp_r) * p.dcp_k + x % p.dcp_k;
}

// Masked shard view: does this shard own global key gk?
__device__ __forceinline__ bool shard_owns(const DecodeParams &p, int32_t gk) {
  return (gk / p.dcp_k) % p.dcp_n == p.dcp_r;
}

// Quantised pools fold V's block scale s_v into P before P is rounded to
// f16 for the PV MMAs.  Block scales of real KV are small (E4M3: amax / 448,
// often 1e-3 .. 1e-5), which would push P * s_v into f16 subnormals.  So P is
// computed as 2^(s - m + kPExp) instead of 2^(s - m): a constant offset on
// the online-softmax running max (the row sums carry the same 2^kPExp, so
// O / l is unchanged, and the log-sum-exp is taken against m - kPExp).  With
// block scales at most kQuantScaleMax = 16, P * s_v <= 2^11 * 16 = 2^15 stays
// a finite f16, and scales down to 1e-7 keep P * s_v normal for P >= 3e-4
// (smaller weights lose relative precision, and matter less in proportion).
constexpr float kPExp = 11.f;

// End of a decode item, shared by the storage formats: merge the NW warps'
// (max, sum, O) through shared memory, normalise, and write the rows, or
// this range's partial (O / l and the log-sum-exp), which decode_merge_kernel
// combines with the other ranges of the (request, KV head).
// `dmap(mt, dr)` is the head-dim index of row dr of m-tile mt of the O^T
// accumulator; `acc_scale` undoes a power-of-two factor carried in acc.
template <int NW, typename DMap>
__device__ __forceinline__ void decode_finish(const DecodeParams &p, const pkv_work_item &it,
                                              uint8_t *smem, const int tid,
                                              const int bar, float m0, float m1, float l0,
                                              float l1, const float (&acc)[8][4],
                                              const float acc_scale, DMap dmap) {
  constexpr int kDecWarps = NW;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int group = p.group;
  auto sync = [&]() { named_barrier(bar, NW * 32); };
  // ---- per-warp row sums, then merge the 4 warps through shared memory
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  sync();  // rings are free now
  float *red_o = reinterpret_cast<float *>(smem);           // [NW][8][128]
  float *red_m = red_o + kDecWarps * kDecCols * kHeadDim;   // [NW][8]
  float *red_l = red_m + kDecWarps * kDecCols;              // [NW][8]
  if (g == 0) {
    red_m[warp * kDecCols + 2 * t] = m0;
    red_m[warp * kDecCols + 2 * t + 1] = m1;
    red_l[warp * kDecCols + 2 * t] = l0;
    red_l[warp * kDecCols + 2 * t + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int n = 2 * t + (c & 1);
      const int dr = g + 8 * (c >> 1);
      red_o[(warp * kDecCols + n) * kHeadDim + dmap(mt, dr)] = acc[mt][c] * acc_scale;
    }
  }
  sync();

  // one head-dim element per thread; NW/4 groups of 128 threads split the rows
  const int d = tid & 127;
  const int n_first = tid >> 7, n_step = NW / 4;
  auto write_row = [&](int n, float o, float lse2) {
    const int r = it.row0 + n;
    const int64_t row = static_cast<int64_t>(it.tok0 + r / group) * p.hq +
                        it.kv_head * group + r % group;
    if (p.out_f32 != nullptr)
      p.out_f32[row * kHeadDim + d] = o;
    else
      p.out[row * kHeadDim + d] = __float2bfloat16_rn(o);
    if (d == 0 && p.lse != nullptr) p.lse[row] = lse2 * kLn2;
  };
  for (int n = n_first; n < it.n_rows; n += n_step) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red_m[w * kDecCols + n]);
    const float Mu = M == -CUDART_INF_F ? 0.f : M;
    float Ls = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float sw = exp2f(red_m[w * kDecCols + n] - Mu);
      Ls += red_l[w * kDecCols + n] * sw;
      o += red_o[(w * kDecCols + n) * kHeadDim + d] * sw;
    }
    const float lse2 = Ls > 0.f ? Mu + log2f(Ls) : -CUDART_INF_F;
    o = Ls > 0.f ? o / Ls : 0.f;
    if (it.part < 0) {
      write_row(n, o, lse2);
    } else {
      p.part_o[(static_cast<int64_t>(it.part) * kDecCols + n) * kHeadDim + d] = o;
      if (d == 0) p.part_lse[static_cast<int64_t>(it.part) * kDecCols + n] = lse2;
    }
  }
}

// One decode work item processed by NW warps (threads tid = 0 .. 32 NW - 1
// of the CTA); `smem` is 1024-byte aligned and holds NW rings plus their
// mbarriers; `bar` is the named barrier these warps synchronise on.  MASK:
// the masked context-parallel shard view (DecodeParams::dcp_mask), compiled
// only into the kernels that serve it.
template <bool FP8, int NW, bool MASK = false>
__device__ __forceinline__ void decode_item(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                            const DecodeParams &p, const pkv_work_item it,
                                            uint8_t *smem, const int tid, const int bar) {
  using Tile = DecTile<FP8>;
  constexpr int KS = Tile::kKeys;
  constexpr int kDecStages = FP8 ? kDecStagesFp8 : pkv::kDecStages;  // ring depth
  constexpr int kDecWarps = NW;
  uint64_t *bars = reinterpret_cast<uint64_t *>(
      smem + kDecWarps * kDecStages * kDecStageBytes);
  auto sync = [&]() { named_barrier(bar, NW * 32); };

  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;
  const int t = lane & 3;

  if (tid < kDecWarps * kDecStages) mbar_init(&bars[tid], 1);
  if (tid == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  fence_mbar_init();
  sync();
  const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride;

  const int kb = it.k_begin;
  const int ke = it.k_end;
  const int n_total = (ke - kb + KS - 1) / KS;
  const int my_n = n_total > warp ? (n_total - warp + kDecWarps - 1) / kDecWarps : 0;
  uint8_t *ring = smem + warp * kDecStages * kDecStageBytes;
  uint64_t *full = bars + warp * kDecStages;
  const int br = p.bs < KS ? p.bs : KS;  // rows per TMA box

  // Fill ring slot for this warp's i-th stage (lane 0 only).
  auto issue = [&](int i) {
    const int key0 = kb + (warp + i * kDecWarps) * KS;
    const int slot = i % kDecStages;
    uint8_t *kdst = ring + slot * kDecStageBytes;
    uint8_t *vdst = kdst + Tile::kKBytes;
    const int gkey0 = global_key(p, key0);
    int boxes = 0;
    for (int r = 0; r < KS; r += br)
      if (key0 + r < ke) ++boxes;
    mbar_arrive_expect_tx(&full[slot], boxes * br * 128 * 2 * (FP8 ? 1 : 2));
    for (int r = 0; r < KS; r += br) {
      if (key0 + r >= ke) break;
      int32_t blk;
      const int32_t y = pool_row(bt, gkey0 + r, it.kv_head, p, &blk);
      if constexpr (FP8) {
        tma_load_2d(kdst + r * 128, &kmap, 0, y, &full[slot]);
        tma_load_2d(vdst + r * 128, &vmap, 0, y, &full[slot]);
      } else {
        tma_load_2d(kdst + r * 128, &kmap, 0, y, &full[slot]);
        tma_load_2d(kdst + KS * 128 + r * 128, &kmap, 64, y, &full[slot]);
        tma_load_2d(vdst + r * 128, &vmap, 0, y, &full[slot]);
        tma_load_2d(vdst + KS * 128 + r * 128, &vmap, 64, y, &full[slot]);
      }
    }
  };

  if (lane == 0) {
    const int pre = my_n < kDecStages ? my_n : kDecStages;
    for (int i = 0; i < pre; ++i) issue(i);
  }

  // Query fragments (B operand, column n = g) with the head-dim order that
  // matches how this thread reads K rows.
  const int group = p.group;
  const bool col_ok = g < it.n_rows;
  uint32_t qf[8][2];
  // E4M3 pools: QK runs on FP8 MMAs over the stored K codes.  Each query
  // column is scaled by a power of two sq (max |q sq| <= 448) and split into
  // q sq = hi + lo, both E4M3 (about bf16 precision); 1/sq is folded into
  // the score scale of that column.
  float inv_sq0 = 1.f, inv_sq1 = 1.f;
  if constexpr (FP8) {
    const int r = it.row0 + g;
    const __nv_bfloat16 *qrow =
        p.q + (static_cast<int64_t>(it.tok0 + r / group) * p.hq +
               it.kv_head * group + r % group) * kHeadDim + 32 * t;
    float qv[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (col_ok) w = __ldg(reinterpret_cast<const uint4 *>(qrow) + i);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        qv[8 * i + 2 * k] = __uint_as_float(ww[k] << 16);
        qv[8 * i + 2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qv[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float sq = amax > 0.f ? exp2f(floorf(log2f(448.f / amax))) : 1.f;
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t hcode[2], lcode[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float x0 = qv[4 * k + 2 * h2] * sq, x1 = qv[4 * k + 2 * h2 + 1] * sq;
        hcode[h2] = e4m3x2_from_f32(x0, x1);
        const float2 back = e4m3x2_to_f32(hcode[h2]);
        lcode[h2] = e4m3x2_from_f32(x0 - back.x, x1 - back.y);
      }
      hw[k] = hcode[0] | (hcode[1] << 16);
      lw[k] = lcode[0] | (lcode[1] << 16);
    }
    // step s (32 head-dim values): b0 = word 4(s>>1) + 2(s&1), b1 = next
#pragma unroll
    for (int st = 0; st < 4; ++st) {
      const int w0 = 4 * (st >> 1) + 2 * (st & 1);
      qf[st][0] = hw[w0];
      qf[st][1] = hw[w0 + 1];
      qf[4 + st][0] = lw[w0];
      qf[4 + st][1] = lw[w0 + 1];
    }
    const float inv = 1.f / sq;
    inv_sq0 = __shfl_sync(0xffffffffu, inv, (2 * t) * 4);
    inv_sq1 = __shfl_sync(0xffffffffu, inv, (2 * t + 1) * 4);
  } else {
    const int r = it.row0 + g;
    const __nv_bfloat16 *qrow =
        p.q + (static_cast<int64_t>(it.tok0 + r / group) * p.hq +
               it.kv_head * group + r % group) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d0 = 64 * (ks >> 2) + 16 * t + 8 * ((ks >> 1) & 1) + 4 * (ks & 1);
      uint2 v = make_uint2(0u, 0u);
      if (col_ok) v = __ldg(reinterpret_cast<const uint2 *>(qrow + d0));
      qf[ks][0] = v.x;
      qf[ks][1] = v.y;
    }
  }
  // the keys of this thread's two S^T rows (g, g+8) within a sub-tile
  const int krow0 = FP8 ? fp8_key(g) : g, krow1 = FP8 ? fp8_key(g + 8) : g + 8;
  // causal limit of this thread's two columns (2t, 2t+1)
  const int c0 = it.row0 + 2 * t;
  const int pos0 = (2 * t < it.n_rows) ? it.hist + c0 / group : 0x7fffffff;
  const int pos1 = (2 * t + 1 < it.n_rows) ? it.hist + (c0 + 1) / group : 0x7fffffff;

  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
    acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // E4M3 pools: the per-block scales of a stage's sub-tiles are loaded
  // before its wait (block ids one stage ahead), so their latency hides
  // behind the copy instead of sitting between the MMAs and the softmax
  // (a stage, KS keys from a multiple of KS in one run of a shard, lies in
  // one block when blocks hold at least KS keys)
  const bool one_block = p.bs >= KS;
  const int bs_sh = bs_shift(p);
  auto stage_blocks = [&](int i, int32_t (&blk)[Tile::kSubs]) {
#pragma unroll
    for (int sub = 0; sub < Tile::kSubs; ++sub) {
      const int k16 = kb + (warp + i * kDecWarps) * KS + 16 * sub;
      if (sub > 0 && one_block)
        blk[sub] = k16 < ke ? blk[0] : -1;
      else
        blk[sub] = (FP8 && i < my_n && k16 < ke) ? __ldg(bt + (global_key(p, k16) >> bs_sh)) : -1;
    }
  };
  // smallest position of the item's rows: a stage whose keys all lie at or
  // below it and before ke needs no mask
  const int pos_lo = it.hist + it.row0 / p.group;
  // running maxima as used for P (E4M3: m - kPExp; 0 before any key)
  float mp0 = FP8 ? -kPExp : 0.f, mp1 = mp0;
  int32_t blk_next[Tile::kSubs];
  stage_blocks(0, blk_next);


  int consumed = 0;
  bool timed_out = false;
  for (int i = 0; i < my_n; ++i) {
    const int slot = i % kDecStages;
    float sk_sub[Tile::kSubs], sv_sub[Tile::kSubs];
    if constexpr (FP8) {
#pragma unroll
      for (int sub = 0; sub < Tile::kSubs; ++sub) {
        const int32_t blk = blk_next[sub];
        sk_sub[sub] = sv_sub[sub] = 0.f;
        if (sub > 0 && one_block) {   // the same block's scales (sub-tiles past ke: unused)
          sk_sub[sub] = sk_sub[0];
          sv_sub[sub] = sv_sub[0];
        } else if (blk >= 0 && blk < p.num_blocks) {
          const int64_t si = static_cast<int64_t>(blk) * p.hkv + it.kv_head;
          sk_sub[sub] = __ldg(p.k_scale + si);
          sv_sub[sub] = __ldg(p.v_scale + si);
        }
      }
      stage_blocks(i + 1, blk_next);
    }
    const bool ok = mbar_wait(&full[slot], (i / kDecStages) & 1);
    if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform way out
      timed_out = true;
      break;
    }
    const int key0 = kb + (warp + i * kDecWarps) * KS;
    const int gkey0 = global_key(p, key0);
    const uint32_t kbase = smem_addr(ring + slot * kDecStageBytes);
    const uint32_t vbase = kbase + Tile::kKBytes;
    // ---- S^T = K Q^T, 16 keys x 8 columns per sub-tile; the sub-tiles'
    // MMA chains are independent, then one softmax step covers the stage
    float s[Tile::kSubs][4];
#pragma unroll
    for (int sub = 0; sub < Tile::kSubs; ++sub) {
      s[sub][0] = s[sub][1] = s[sub][2] = s[sub][3] = 0.f;
      if (key0 + 16 * sub >= ke) continue;
      if constexpr (FP8) {
        // raw K codes straight into FP8 MMAs: thread t's 16 bytes of a row
        // are steps 2h, 2h+1 (words 0,1 -> a0,a2 of step 2h; 2,3 of 2h+1)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 x = lds128(kbase + swz128(16 * sub + krow0, 2 * t + h));
          const uint4 y = lds128(kbase + swz128(16 * sub + krow1, 2 * t + h));
          mma_e4m3(s[sub], x.x, y.x, x.y, y.y, qf[2 * h][0], qf[2 * h][1]);
          mma_e4m3(s[sub], x.x, y.x, x.y, y.y, qf[4 + 2 * h][0], qf[4 + 2 * h][1]);
          mma_e4m3(s[sub], x.z, y.z, x.w, y.w, qf[2 * h + 1][0], qf[2 * h + 1][1]);
          mma_e4m3(s[sub], x.z, y.z, x.w, y.w, qf[4 + 2 * h + 1][0], qf[4 + 2 * h + 1][1]);
        }
      } else {
#pragma unroll
        for (int L = 0; L < 4; ++L) {
          const uint32_t off = (L >> 1) * (KS * 128);
          const uint32_t ch = 2 * t + (L & 1);
          const uint4 x = lds128(kbase + off + swz128(g, ch));
          const uint4 y = lds128(kbase + off + swz128(g + 8, ch));
          mma_bf16(s[sub], x.x, y.x, x.y, y.y, qf[2 * L][0], qf[2 * L][1]);
          mma_bf16(s[sub], x.z, y.z, x.w, y.w, qf[2 * L + 1][0], qf[2 * L + 1][1]);
        }
      }
    }
    // ---- scale, mask (validity on item-local keys, causality on global
    // positions), online softmax per column over the stage
    float tm0 = -CUDART_INF_F, tm1 = -CUDART_INF_F;
    const bool unmasked = !MASK && key0 + KS <= ke && gkey0 + KS - 1 <= pos_lo;
#pragma unroll
    for (int sub = 0; sub < Tile::kSubs; ++sub) {
      float sc0 = p.scale_log2, sc1 = p.scale_log2;
      if constexpr (FP8) {
        sc0 *= sk_sub[sub] * inv_sq0;
        sc1 *= sk_sub[sub] * inv_sq1;
      }
      if (unmasked) {
        s[sub][0] *= sc0;
        s[sub][1] *= sc1;
        s[sub][2] *= sc0;
        s[sub][3] *= sc1;
      } else {
        const int kr0 = key0 + 16 * sub + krow0, kr1 = key0 + 16 * sub + krow1;
        const int gr0 = gkey0 + 16 * sub + krow0, gr1 = gkey0 + 16 * sub + krow1;
        s[sub][0] = (kr0 < ke && gr0 <= pos0) ? s[sub][0] * sc0 : -CUDART_INF_F;
        s[sub][1] = (kr0 < ke && gr0 <= pos1) ? s[sub][1] * sc1 : -CUDART_INF_F;
        s[sub][2] = (kr1 < ke && gr1 <= pos0) ? s[sub][2] * sc0 : -CUDART_INF_F;
        s[sub][3] = (kr1 < ke && gr1 <= pos1) ? s[sub][3] * sc1 : -CUDART_INF_F;
        if constexpr (MASK) {   // masked shard view: keys another shard owns
          if (!shard_owns(p, gr0)) s[sub][0] = s[sub][1] = -CUDART_INF_F;
          if (!shard_owns(p, gr1)) s[sub][2] = s[sub][3] = -CUDART_INF_F;
        }
      }
      tm0 = fmaxf(tm0, fmaxf(s[sub][0], s[sub][2]));
      tm1 = fmaxf(tm1, fmaxf(s[sub][1], s[sub][3]));
    }
    // a column's maximum grows only if one of its scores lies above it: only
    // then reduce the stage maxima over the column's threads and rescale
    // (otherwise every factor is exactly 1)
    if (__any_sync(0xffffffffu, tm0 > m0 || tm1 > m1)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, o));
        tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, o));
      }
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      const float mu0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
      const float mu1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
      const float al0 = ex2(m0 - mu0), al1 = ex2(m1 - mu1);
      mp0 = FP8 ? mu0 - kPExp : mu0;
      mp1 = FP8 ? mu1 - kPExp : mu1;
      m0 = mn0;
      m1 = mn1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
    }
#pragma unroll
    for (int sub = 0; sub < Tile::kSubs; ++sub) {
      const int k16 = key0 + 16 * sub;
      if (k16 >= ke) break;
      const float p0 = ex2(s[sub][0] - mp0), p1 = ex2(s[sub][1] - mp1);
      const float p2 = ex2(s[sub][2] - mp0), p3 = ex2(s[sub][3] - mp1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      const float pv_scale = FP8 ? sv_sub[sub] : 1.f;
      // ---- P^T as the B operand: transpose the two 8x8 halves in registers
      // (f16 for E4M3 pools, whose V is unpacked to f16; bf16 otherwise)
      const uint32_t b0 = movmatrix_trans(FP8 ? pack_f16(p0 * pv_scale, p1 * pv_scale)
                                              : pack_bf16(p0 * pv_scale, p1 * pv_scale));
      const uint32_t b1 = movmatrix_trans(FP8 ? pack_f16(p2 * pv_scale, p3 * pv_scale)
                                              : pack_bf16(p2 * pv_scale, p3 * pv_scale));
      // keys of this thread's V^T fragment halves
      const bool tail = k16 + 16 > ke;
      const int ka = k16 + 2 * t;
      const uint32_t mlo = tail ? ((ka < ke ? 0x0000FFFFu : 0u) | (ka + 1 < ke ? 0xFFFF0000u : 0u))
                                : 0xFFFFFFFFu;
      const uint32_t mhi = tail ? ((ka + 8 < ke ? 0x0000FFFFu : 0u) | (ka + 9 < ke ? 0xFFFF0000u : 0u))
                                : 0xFFFFFFFFu;
      // ---- O^T += V^T P^T
      if constexpr (FP8) {
        // V^T fragments straight from the E4M3 tile: one 8-bit transposing
        // ldmatrix gives two m-tiles (16 head dims each, lanes 0-15 address
        // the sub-tile's 16 key rows in the first one's 16-byte chunk, lanes
        // 16-31 in the second's); each register holds keys 4t .. 4t+3 of one
        // head dim, converted exactly to f16 pairs for key slots (2t, 2t+1)
        // and (2t+8, 2t+9) (see fp8_key).  Masks only on the item's last,
        // partial sub-tile.
        const uint32_t vrow = 16 * sub + (lane & 15);
        auto pv8 = [&](auto masked) {
          uint32_t qlo = 0xFFFFFFFFu, qhi = 0xFFFFFFFFu;
          if (decltype(masked)::value) {
            const int kq = k16 + 4 * t;
            qlo = (kq < ke ? 0x0000FFFFu : 0u) | (kq + 1 < ke ? 0xFFFF0000u : 0u);
            qhi = (kq + 2 < ke ? 0x0000FFFFu : 0u) | (kq + 3 < ke ? 0xFFFF0000u : 0u);
          }
#pragma unroll
          for (int mp = 0; mp < 4; ++mp) {
            uint32_t r[4];
            ldsm_b8_x2_trans(vbase + swz128(vrow, 2 * mp + (lane >> 4)), r[0], r[1], r[2],
                             r[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a0 = e4m3x2lo_to_f16x2(r[2 * h]), a2 = e4m3x2hi_to_f16x2(r[2 * h]);
              uint32_t a1 = e4m3x2lo_to_f16x2(r[2 * h + 1]), a3 = e4m3x2hi_to_f16x2(r[2 * h + 1]);
              if (decltype(masked)::value) {
                a0 &= qlo;
                a1 &= qlo;
                a2 &= qhi;
                a3 &= qhi;
              }
              mma_f16(acc[2 * mp + h], a0, a1, a2, a3, b0, b1);
            }
          }
        };
        if (tail)
          pv8(std::true_type{});
        else
          pv8(std::false_type{});
      } else {
        const int mi = lane >> 3;
        const int key = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const uint32_t ch = 2 * (mt & 3) + (mi & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(vbase + (mt >> 2) * (KS * 128) + swz128(key, ch), a0, a1,
                        a2, a3);
          mma_bf16(acc[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, b0, b1);
        }
      }
    }
    __syncwarp();
    ++consumed;
    if (lane == 0 && i + kDecStages < my_n) {
      fence_proxy_async();
      issue(i + kDecStages);
    }
  }
  if (timed_out) {
    record_error(p.err, kErrTimeout);
    // let copies already in flight land before the shared memory is reused
    const int issued = my_n < consumed + kDecStages ? my_n : consumed + kDecStages;
    for (int i = consumed; i < issued; ++i)
      mbar_wait(&full[i % kDecStages], (i / kDecStages) & 1);
  }

  // P carried 2^kPExp: the effective running maxima are m - kPExp
  decode_finish<NW>(p, it, smem, tid, bar, FP8 ? m0 - kPExp : m0, FP8 ? m1 - kPExp : m1, l0,
                    l1, acc, 1.f, [](int mt, int dr) { return 16 * mt + dr; });
}


}  // namespace
}  // namespace pkv
