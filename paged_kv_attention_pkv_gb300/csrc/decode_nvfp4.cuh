// Split-KV decode over NVFP4 pools (device code).  Same work item, key
// split, online softmax and combine as the bf16 / E4M3 decode
// (decode_body.cuh); what differs is how a stage of keys reaches the MMAs.
//
// NVFP4 KV is the compressed KV format of page "vLLM 优化
// DeepSeek-V4.1-Flash：智能体吞吐提升 5 倍", section Kernels (MegaAttention
// reads NVFP4 KV, nearly half the bytes of FP8).  Element value =
// e2m1(code) * e4m3(micro scale of its 16 elements) * fp32 (block, KV head)
// scale.
//
// A stage is kDecKeysNvfp4 keys: their code rows (64 bytes each) arrive by
// TMA into a 64-byte-swizzled tile, their micro scales (8 bytes each) by a
// bulk copy.
// Codes are converted to f16 in hardware and multiplied by their micro scale
// in f16, which is exact (a 2-bit by 4-bit significand product), so the MMAs
// see e2m1 * e4m3 exactly; the fp32 block scales are folded into the score
// scale (K) and into P (V, with P's exponent offset kPExp), as for E4M3
// pools.  Queries enter the f16 MMAs
// scaled by a power of two per column (largest |q| in [2^14, 2^15)), undone
// in the score scale.
//
// Inside each 16-key sub-tile the MMA's key index k reads physical row
// nv_key(k).  With the 64-byte swizzle this keeps both the QK reads (two
// rows per 8-lane phase) and the V^T fragment reads (four rows per 16-lane
// phase, 8 bytes each) free of shared-memory bank conflicts.
#pragma once

#include "decode_body.cuh"

namespace pkv {
namespace {

constexpr int kNvKeys = kDecKeysNvfp4;            // keys per stage
constexpr int kNvCodeBytes = kNvKeys * 64;        // code rows of one of K / V
constexpr int kNvScaleBytes = kNvKeys * 8;        // micro scales of one of K / V
static_assert(2 * (kNvCodeBytes + kNvScaleBytes) == kDecStageBytesNvfp4, "stage layout");

// Byte offset in a tile of 64-byte rows written by TMA with
// CU_TENSOR_MAP_SWIZZLE_64B (16-byte chunk bits 4-5 XOR address bits 7-8);
// the tile starts 512-byte aligned.
__device__ __forceinline__ uint32_t swz64(uint32_t o) { return o ^ ((o >> 3) & 0x30u); }

// Physical row of MMA key index k (0..15) in a 16-key sub-tile:
// 0 3 1 2 4 7 5 6, then the same plus 8.
__device__ __forceinline__ int nv_key(int k) {
  return (k & 12) | ((0x9C >> (2 * (k & 3))) & 3);
}

// Head-dim index of row dr of m-tile mt of the O^T accumulator: thread g
// holds the 16 elements of micro block g; m-tile 4w + j takes element
// 8w + 2j (rows g) and 8w + 2j + 1 (rows g + 8) of it.
__device__ __forceinline__ int nvfp4_dmap(int mt, int dr) {
  return 16 * (dr & 7) + 8 * (mt >> 2) + 2 * (mt & 3) + (dr >> 3);
}

template <int NW, bool MASK = false>
__device__ __forceinline__ void decode_item_nvfp4(const CUtensorMap &kmap,
                                                  const CUtensorMap &vmap,
                                                  const DecodeParams &p,
                                                  const pkv_work_item it, uint8_t *smem,
                                                  const int tid, const int bar) {
  constexpr int KS = kNvKeys;
  constexpr int S = kDecStagesNvfp4;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * S * kDecStageBytesNvfp4);
  auto sync = [&]() { named_barrier(bar, NW * 32); };
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2;
  const int t = lane & 3;

  if (tid < NW * S) mbar_init(&bars[tid], 1);
  if (tid == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  fence_mbar_init();
  sync();

  const int kb = it.k_begin;
  const int ke = it.k_end;
  const int n_total = (ke - kb + KS - 1) / KS;
  const int my_n = n_total > warp ? (n_total - warp + NW - 1) / NW : 0;
  uint8_t *ring = smem + warp * S * kDecStageBytesNvfp4;
  uint64_t *full = bars + warp * S;
  const int32_t *bt = p.block_tables + static_cast<int64_t>(it.seq) * p.bt_stride;
  // block sizes are powers of two: keys map to blocks and row groups by shifts
  const int bs_sh = 31 - __clz(p.bs);
  const int gs_sh = bs_sh < 6 ? bs_sh : 6;                  // kNvfp4Group = 64 rows
  const int gs = 1 << gs_sh;                                // rows per group
  const int br = gs < KS ? gs : KS;                         // keys per copy
  const int tile_rows = p.bs / 8 * 9;                       // 64-byte rows per tile
  const int group_rows = gs / 8 * 9;
  // a stage (KS keys from a multiple of KS, in one run of a shard) lies in
  // one block when blocks hold at least KS keys
  const bool one_block = p.bs >= KS;

  // Fill ring slot i % S with stage i (lane 0 only): per run of br keys
  // inside one group, the code rows by TMA and the micro scales by a bulk
  // copy.
  auto issue = [&](int i) {
    const int key0 = kb + (warp + i * NW) * KS;
    const int slot = i % S;
    uint8_t *st = ring + slot * kDecStageBytesNvfp4;
    const int gkey0 = global_key(p, key0);
    int runs = 0;
    for (int r = 0; r < KS; r += br)
      if (key0 + r < ke) ++runs;
    mbar_arrive_expect_tx(&full[slot], runs * br * 2 * kNvfp4RowBytes);
    for (int r = 0; r < KS; r += br) {
      if (key0 + r >= ke) break;
      const int gk = gkey0 + r;
      const int32_t blk = __ldg(bt + (gk >> bs_sh));
      int32_t row = p.rows_total;   // outside the map: TMA fills zeros
      int64_t sbyte = 0;            // (a flagged bad block reads scales from offset 0)
      if (blk < 0 || blk >= p.num_blocks) {
        record_error(p.err, kErrBadBlock);
      } else {
        const int in_blk = gk & (p.bs - 1);
        const int grp0 = (blk * p.hkv + it.kv_head) * tile_rows + (in_blk >> gs_sh) * group_rows;
        row = grp0 + (in_blk & (gs - 1));
        sbyte = static_cast<int64_t>(grp0 + gs) * 64 + (in_blk & (gs - 1)) * 8;
      }
      tma_load_2d(st + r * 64, &kmap, 0, row, &full[slot]);
      tma_load_2d(st + kNvCodeBytes + r * 64, &vmap, 0, row, &full[slot]);
      bulk_load(st + 2 * kNvCodeBytes + r * 8, p.k_pool + sbyte, br * 8, &full[slot]);
      bulk_load(st + 2 * kNvCodeBytes + kNvScaleBytes + r * 8, p.v_pool + sbyte, br * 8,
                &full[slot]);
    }
  };

  if (lane == 0) {
    const int pre = my_n < S ? my_n : S;
    for (int i = 0; i < pre; ++i) issue(i);
  }

  // Query fragments: thread (g, t) holds head dims 32t .. 32t+31 of column
  // g; k-step ks takes dims 4ks, 4ks+1 (b0) and 4ks+2, 4ks+3 (b1) of them,
  // matching code bytes 2ks and 2ks+1 of the thread's 16-byte K chunk.
  const int group = p.group;
  const bool col_ok = g < it.n_rows;
  uint32_t qf[8][2];
  float inv_sq0, inv_sq1;
  {
    const int r = it.row0 + g;
    const __nv_bfloat16 *qrow =
        p.q + (static_cast<int64_t>(it.tok0 + r / group) * p.hq + it.kv_head * group +
               r % group) * kHeadDim + 32 * t;
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
    // sq = 2^(14 - e) for amax = m 2^e (m in [1, 2)): |q sq| < 2^15
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
    const int k2 = 14 - e < 126 ? 14 - e : 126;
    const float sq = __uint_as_float(static_cast<uint32_t>(127 + k2) << 23);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[ks][0] = pack_f16(qv[4 * ks] * sq, qv[4 * ks + 1] * sq);
      qf[ks][1] = pack_f16(qv[4 * ks + 2] * sq, qv[4 * ks + 3] * sq);
    }
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - k2) << 23);
    inv_sq0 = __shfl_sync(0xffffffffu, inv, (2 * t) * 4);
    inv_sq1 = __shfl_sync(0xffffffffu, inv, (2 * t + 1) * 4);
  }
  // causal limit of this thread's two columns (2t, 2t+1)
  const int c0 = it.row0 + 2 * t;
  const int pos0 = (2 * t < it.n_rows) ? it.hist + c0 / group : 0x7fffffff;
  const int pos1 = (2 * t + 1 < it.n_rows) ? it.hist + (c0 + 1) / group : 0x7fffffff;

  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
    acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // block ids of a stage's sub-tiles, one stage ahead (their scales are
  // loaded before the stage's wait)
  constexpr int kSubs = KS / 16;
  auto stage_blocks = [&](int i, int32_t (&blk)[kSubs]) {
#pragma unroll
    for (int sub = 0; sub < kSubs; ++sub) {
      const int k16 = kb + (warp + i * NW) * KS + 16 * sub;
      if (sub > 0 && one_block)
        blk[sub] = k16 < ke ? blk[0] : -1;
      else
        blk[sub] = (i < my_n && k16 < ke) ? __ldg(bt + (global_key(p, k16) >> bs_sh)) : -1;
    }
  };
  int32_t blk_next[kSubs];
  stage_blocks(0, blk_next);

  // rows this thread reads: QK rows nv_key(g) and nv_key(g) + 8; V^T rows for
  // MMA keys 2t, 2t+1 (A/B) and 2t+8, 2t+9 (C/D).  Offsets in sub-tile 0;
  // sub-tile sub adds 1024 sub to the code offsets (the swizzle acts on
  // address bits 4-8 only) and 128 sub to the micro-scale offsets.
  const int qk_row = nv_key(g);
  const int pv_a = nv_key(2 * t), pv_b = nv_key(2 * t + 1);
  const uint32_t o_ka = swz64(qk_row * 64 + 16 * t), o_kb = swz64((qk_row + 8) * 64 + 16 * t);
  const uint32_t o_ksa = qk_row * 8 + 2 * t, o_ksb = o_ksa + 64;
  const uint32_t o_va = swz64(pv_a * 64 + 8 * g), o_vb = swz64(pv_b * 64 + 8 * g);
  const uint32_t o_vc = swz64((pv_a + 8) * 64 + 8 * g), o_vd = swz64((pv_b + 8) * 64 + 8 * g);
  const uint32_t o_vsa = pv_a * 8 + g, o_vsb = pv_b * 8 + g;
  // smallest position of the item's rows: a stage whose keys all lie at or
  // below it and before ke needs no mask
  const int pos_lo = it.hist + it.row0 / group;
  // running maxima as used for P (m - kPExp, 0 before any key)
  float mp0 = -kPExp, mp1 = -kPExp;

  int consumed = 0;
  bool timed_out = false;
  for (int i = 0; i < my_n; ++i) {
    const int slot = i % S;
    float sk_sub[kSubs], sv_sub[kSubs];
#pragma unroll
    for (int sub = 0; sub < kSubs; ++sub) {
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
    const bool ok = mbar_wait(&full[slot], (i / S) & 1);
    if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform way out
      timed_out = true;
      break;
    }
    const int key0 = kb + (warp + i * NW) * KS;
    const int gkey0 = global_key(p, key0);
    const uint32_t kc = smem_addr(ring + slot * kDecStageBytesNvfp4);
    const uint32_t vc = kc + kNvCodeBytes;
    const uint32_t ksc = kc + 2 * kNvCodeBytes;
    const uint32_t vsc = ksc + kNvScaleBytes;
    // ---- S^T = K Q^T for the stage's sub-tiles (16 keys x 8 columns each):
    // independent MMA chains, then one softmax step for all 64 keys
    float s[kSubs][4];
#pragma unroll
    for (int sub = 0; sub < kSubs; ++sub) {
      s[sub][0] = s[sub][1] = s[sub][2] = s[sub][3] = 0.f;
      if (key0 + 16 * sub >= ke) continue;
      const uint4 x = lds128(kc + 1024 * sub + o_ka);
      const uint4 y = lds128(kc + 1024 * sub + o_kb);
      // micro scales of micro blocks 2t, 2t+1 of both rows, as f16 pairs
      const uint32_t sa = e4m3x2lo_to_f16x2(lds16(ksc + 128 * sub + o_ksa));
      const uint32_t sb = e4m3x2lo_to_f16x2(lds16(ksc + 128 * sub + o_ksb));
      const uint32_t sa0 = __byte_perm(sa, 0, 0x1010), sa1 = __byte_perm(sa, 0, 0x3232);
      const uint32_t sb0 = __byte_perm(sb, 0, 0x1010), sb1 = __byte_perm(sb, 0, 0x3232);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
      const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t ca[4], cb[4];
        e2m1x8_to_f16x2(xw[w], ca);
        e2m1x8_to_f16x2(yw[w], cb);
        const uint32_t ma = w < 2 ? sa0 : sa1, mb = w < 2 ? sb0 : sb1;
        mma_f16(s[sub], hmul2(ca[0], ma), hmul2(cb[0], mb), hmul2(ca[1], ma),
                hmul2(cb[1], mb), qf[2 * w][0], qf[2 * w][1]);
        mma_f16(s[sub], hmul2(ca[2], ma), hmul2(cb[2], mb), hmul2(ca[3], ma),
                hmul2(cb[3], mb), qf[2 * w + 1][0], qf[2 * w + 1][1]);
      }
    }
    // ---- scale, mask (validity on item-local keys, causality on global
    // positions), online softmax per column over the whole stage
    float tm0 = -CUDART_INF_F, tm1 = -CUDART_INF_F;
    const bool unmasked = !MASK && key0 + KS <= ke && gkey0 + KS - 1 <= pos_lo;
#pragma unroll
    for (int sub = 0; sub < kSubs; ++sub) {
      const float sc0 = p.scale_log2 * sk_sub[sub] * inv_sq0;
      const float sc1 = p.scale_log2 * sk_sub[sub] * inv_sq1;
      if (unmasked) {
        s[sub][0] *= sc0;
        s[sub][1] *= sc1;
        s[sub][2] *= sc0;
        s[sub][3] *= sc1;
      } else {
        const int kr0 = key0 + 16 * sub + qk_row, kr1 = kr0 + 8;
        const int gr0 = gkey0 + 16 * sub + qk_row, gr1 = gr0 + 8;
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
      mp0 = mu0 - kPExp;
      mp1 = mu1 - kPExp;
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
    for (int sub = 0; sub < kSubs; ++sub) {
      const int k16 = key0 + 16 * sub;
      if (k16 >= ke) break;
      const float p0 = ex2(s[sub][0] - mp0), p1 = ex2(s[sub][1] - mp1);
      const float p2 = ex2(s[sub][2] - mp0), p3 = ex2(s[sub][3] - mp1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      // ---- P^T as the B operand (f16, V's block scale folded in)
      const float pv_scale = sv_sub[sub];
      const uint32_t b0 = movmatrix_trans(pack_f16(p0 * pv_scale, p1 * pv_scale));
      const uint32_t b1 = movmatrix_trans(pack_f16(p2 * pv_scale, p3 * pv_scale));
      // ---- O^T += V^T P^T: this thread's micro block g of rows A, B, C, D
      const int rA = 16 * sub + pv_a, rB = 16 * sub + pv_b, rC = rA + 8, rD = rB + 8;
      const uint2 uA = lds64(vc + 1024 * sub + o_va);
      const uint2 uB = lds64(vc + 1024 * sub + o_vb);
      const uint2 uC = lds64(vc + 1024 * sub + o_vc);
      const uint2 uD = lds64(vc + 1024 * sub + o_vd);
      const uint32_t vs = vsc + 128 * sub;
      uint32_t sab = e4m3x2lo_to_f16x2(lds8(vs + o_vsa) | (lds8(vs + o_vsb) << 8));
      uint32_t scd = e4m3x2lo_to_f16x2(lds8(vs + o_vsa + 64) | (lds8(vs + o_vsb + 64) << 8));
      if (k16 + 16 > ke) {
        // the item's last, partial sub-tile: keys past ke get micro scale 0
        // (their rows may hold stale bytes; codes are always finite, a stale
        // micro scale may not be, and P is 0 there)
        sab &= (key0 + rA < ke ? 0x0000FFFFu : 0u) | (key0 + rB < ke ? 0xFFFF0000u : 0u);
        scd &= (key0 + rC < ke ? 0x0000FFFFu : 0u) | (key0 + rD < ke ? 0xFFFF0000u : 0u);
      }
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t a = w ? uA.y : uA.x, b = w ? uB.y : uB.x;
        const uint32_t c = w ? uC.y : uC.x, d = w ? uD.y : uD.x;
        // pair the two keys' nibbles per head dim: even dims, odd dims
        uint32_t ae[4], ao[4], ce[4], co[4];
        e2m1x8_to_f16x2((a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u), ae);
        e2m1x8_to_f16x2(((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u), ao);
        e2m1x8_to_f16x2((c & 0x0F0F0F0Fu) | ((d << 4) & 0xF0F0F0F0u), ce);
        e2m1x8_to_f16x2(((c >> 4) & 0x0F0F0F0Fu) | (d & 0xF0F0F0F0u), co);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_f16(acc[4 * w + j], hmul2(ae[j], sab), hmul2(ao[j], sab), hmul2(ce[j], scd),
                  hmul2(co[j], scd), b0, b1);
      }
    }
    __syncwarp();
    ++consumed;
    if (lane == 0 && i + S < my_n) {
      fence_proxy_async();
      issue(i + S);
    }
  }
  if (timed_out) {
    record_error(p.err, kErrTimeout);
    // let copies already in flight land before the shared memory is reused
    const int issued = my_n < consumed + S ? my_n : consumed + S;
    for (int i = consumed; i < issued; ++i) mbar_wait(&full[i % S], (i / S) & 1);
  }
  // P carried 2^kPExp: the effective running maxima are m - kPExp
  decode_finish<NW>(p, it, smem, tid, bar, m0 - kPExp, m1 - kPExp, l0, l1, acc, 1.f,
                    [](int mt, int dr) { return nvfp4_dmap(mt, dr); });
}

}  // namespace
}  // namespace pkv
