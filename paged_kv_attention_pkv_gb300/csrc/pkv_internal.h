// Internal definitions shared by the libpkv host code and kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kHeadDim = 128;

// Device error word bits (validate mode and bounded waits).
enum : int32_t {
  kErrBadBlock = 1,     // a block-table entry in use is outside the pool
  kErrBadSlot = 2,      // a slot_mapping entry is outside the pool
  kErrTimeout = 4,      // a bounded wait gave up
  kErrMismatch = 8,     // device metadata differs from the host mirrors
  kErrBadPosition = 16, // a rotary position is outside the cos/sin cache
  kErrBadScale = 32,    // a quantised pool's block scale in use is above the cap (or NaN)
};

// Block scales of E4M3 and NVFP4 pools must not exceed this: the kernels
// round values times block scales to f16 (decode: P * s_v <= 2^11 * 16; the
// prefill's V conversion: at most 448 * 16 or 6 * 448 * 16 = 43008, all
// below 65504).
constexpr float kQuantScaleMax = 16.f;

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// ---- decode (split-KV) kernel geometry ---------------------------------------
constexpr int kDecWarps = 4;              // consumer warps, each its own ring
constexpr int kDecStages = 3;             // ring depth per warp
constexpr int kDecStageBytes = 8192;      // K 4 KB + V 4 KB per stage
constexpr int kDecCols = 8;               // query rows per item (MMA N)
constexpr int kDecKeysBf16 = 16;          // keys per stage, bf16 pools
constexpr int kDecKeysFp8 = 32;           // keys per stage, E4M3 pools
constexpr int kDecSmemBytes =
    kDecWarps * kDecStages * kDecStageBytes + 1024 /* align */ + 256;
// E4M3 pools: shorter rings and three CTAs per SM (same bytes in flight, more
// warps to hide the latency of the longer per-key instruction stream).
constexpr int kDecStagesFp8 = 2;
constexpr int kDecSmemBytesFp8 =
    kDecWarps * kDecStagesFp8 * kDecStageBytes + 1024 + 256;
// NVFP4 pools: 64 code bytes + 8 micro-scale bytes per 128-element row;
// rows of a (block, KV head) tile in groups of min(block_size, 64).  Decode
// stages hold kDecKeysNvfp4 keys (K and V codes 64 bytes a key, micro scales
// 8), kDecStagesNvfp4 per warp ring, kDecCtasNvfp4 CTAs per SM.
constexpr int kNvfp4RowBytes = kHeadDim / 2 + kHeadDim / 16;   // 72
constexpr int kNvfp4Group = 64;
constexpr int kDecKeysNvfp4 = 64;
constexpr int kDecStagesNvfp4 = 2;
constexpr int kDecCtasNvfp4 = 3;
constexpr int kDecStageBytesNvfp4 = 2 * kDecKeysNvfp4 * kNvfp4RowBytes;   // 9216
constexpr int kDecSmemBytesNvfp4 =
    kDecWarps * kDecStagesNvfp4 * kDecStageBytesNvfp4 + 1024 + 256;
constexpr int kSplitAlign = 256;          // split ranges start at multiples

// ---- prefill kernel geometry ---------------------------------------------------

struct DecodeParams {
  const pkv_work_item *items;
  const __nv_bfloat16 *q;
  const int32_t *block_tables;
  int32_t bt_stride;
  const float *k_scale;
  const float *v_scale;
  __nv_bfloat16 *out;
  float *lse;
  float *part_o;     // [slots][kDecCols][128]
  float *part_lse;   // [slots][kDecCols], log2 domain
  int32_t *err;
  int32_t hq, hkv, group, bs;
  int32_t rows_total;   // num_blocks * hkv * bs (rows of the pool maps)
  int64_t num_blocks;
  float scale_log2;     // softmax_scale * log2(e)
  int32_t validate;
  // Context-parallel shard view (dcp_n > 1): shard dcp_r of dcp_n owns the
  // runs j of dcp_k keys with j % dcp_n == dcp_r.  When dcp_k is a multiple
  // of the stage's key count, items walk the shard's own keys (item-local
  // key x is global key ((x / dcp_k) * dcp_n + dcp_r) * dcp_k + x % dcp_k);
  // otherwise (dcp_mask) items walk every key and the scores of keys the
  // shard does not own are masked.  Results go to out_f32 (fp32,
  // normalised) instead of out when out_f32 is set.
  int32_t dcp_n, dcp_r, dcp_k, dcp_mask;
  float *out_f32;
  // NVFP4 pools (byte addresses of the micro scales); rows_total then counts
  // the pools' 64-byte rows
  const uint8_t *k_pool;
  const uint8_t *v_pool;
};

struct PrefillParams {
  const pkv_work_item *items;
  const __nv_bfloat16 *q;
  const int32_t *block_tables;
  int32_t bt_stride;
  const float *k_scale;   // E4M3 pools: [num_blocks][hkv] block scales
  const float *v_scale;
  __nv_bfloat16 *out;
  float *lse;
  int32_t *err;
  int32_t hq, hkv, group, bs;
  int32_t rows_total;
  int64_t num_blocks;
  float scale_log2;
  int32_t validate;
  // items split over key ranges (part >= 0): partial slots shared with the
  // decode items (a prefill partial spans kPfPartSlots slots), merged by
  // launch_prefill_merge
  float *part_o;
  float *part_lse;
  // K/V staged as bf16 (stage_kv.cu; kernel formats kFmtStaged and
  // kFmtStagedV): block j of request i is staging block stage_base[i] + j of
  // stage_blocks, stage_rows rows in the staging pools; kFmtStaged: k_scale
  // holds the K scale of each staging (block, KV head); NULL: blocks come
  // from block_tables
  const int32_t *stage_base;
  int64_t stage_blocks;
  int32_t stage_rows;
};

// Kernel formats of the tensor-core prefill over staged K/V (beyond the
// pkv_kv_dtype values).  kFmtStaged (NVFP4 pools): K and V staged as bf16
// tiles, K exact code values with a block scale per 16-key group, V already
// scaled.  kFmtStagedV (E4M3 pools): K read from the pool as for E4M3 (FP8
// QK, block scale per 16-key group), V staged as bf16, already scaled.
constexpr int kFmtStaged = 3;
constexpr int kFmtStagedV = 4;

// Staging for the tensor-core prefill (stage_kv.cu): NVFP4 K and V, or
// E4M3 V alone, as bf16.  reqs[3 r .. 3 r + 2] = (request index, first staging
// block, context length) for the staged requests, ascending by first block.
struct StageParams {
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_tables;
  int32_t bt_stride;
  const int32_t *reqs;
  int32_t n_reqs;
  __nv_bfloat16 *k_stage;   // [staging blocks][hkv][bs][128]; NVFP4 only
  __nv_bfloat16 *v_stage;
  float *k_stage_scale;     // [staging blocks][hkv]; NVFP4 only
  int32_t hkv, bs;
  int64_t num_blocks;       // blocks of the quantised pools
  int32_t *err;
};

struct AppendParams {
  const __nv_bfloat16 *k_new;
  const __nv_bfloat16 *v_new;
  const int64_t *slots;
  void *k_cache;
  void *v_cache;
  const float *k_scale;
  const float *v_scale;
  int32_t *err;
  int64_t num_tokens;
  int32_t hkv, bs;
  int64_t num_blocks;
  int32_t validate;
};

// Rotary embedding fused with the KV append: q rotated in place, K rotated
// then written, V written.  cos_sin: [max_pos][128] fp32, cos in columns
// 0..63 and sin in 64..127 for the 64 rotation pairs.
struct RopeAppendParams {
  AppendParams a;
  __nv_bfloat16 *q;          // [num_tokens][hq][128], rotated in place
  const int64_t *positions;  // [num_tokens]
  const float *cos_sin;
  int64_t max_pos;
  int32_t hq;
};

struct CheckParams {
  const int32_t *qsl;
  const int32_t *seq_lens;
  const int32_t *block_tables;
  const int32_t *qsl_expect;       // host mirrors uploaded with the plan
  const int32_t *seq_lens_expect;
  int32_t bt_stride;
  int32_t num_seqs;
  int32_t bs;
  int64_t num_blocks;
  int32_t *err;
  // E4M3 and NVFP4 pools: block scales of every block in use are checked
  // against kQuantScaleMax (NULL: not checked)
  const float *k_scale;
  const float *v_scale;
  int32_t hkv;
};

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_append(const AppendParams &p, int kv_dtype, cudaStream_t s);
cudaError_t launch_rope_append(const RopeAppendParams &p, int kv_dtype, bool neox, cudaStream_t s);
cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap,
                          const DecodeParams &p, int num_items, int kv_dtype,
                          cudaStream_t s);
cudaError_t launch_prefill_tc(const CUtensorMap &qmap, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, const PrefillParams &p,
                              int num_items, int kv_dtype, cudaStream_t s);
// Merge the key ranges of split items: the first num_groups items of
// p.items are the first ranges of the split (request, KV head) pairs (decode)
// or row tiles (prefill); rows and log-sum-exps go to the outputs.  max_split
// is the largest number of ranges of a decode pair (above 32, each row's
// ranges are spread over a CTA's warps).
cudaError_t launch_decode_merge(const DecodeParams &p, int num_groups, int max_split,
                                cudaStream_t s);
cudaError_t launch_prefill_merge(const PrefillParams &p, int num_groups, cudaStream_t s);
cudaError_t launch_check(const CheckParams &p, cudaStream_t s);
cudaError_t launch_stage_kv(const StageParams &p, int num_stage_blocks, int kv_dtype,
                            cudaStream_t s);
cudaError_t launch_wait_selftest(int32_t *err, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_lse_merge(const float *parts_o, const float *parts_lse, int num_parts,
                             int64_t num_rows, __nv_bfloat16 *out, float *lse,
                             cudaStream_t s);
cudaError_t launch_mixed(const CUtensorMap &qmap, const CUtensorMap &kmap_pf,
                         const CUtensorMap &vmap_pf, const CUtensorMap &kmap_dec,
                         const CUtensorMap &vmap_dec, const PrefillParams &pp,
                         const DecodeParams &dp, int n_prefill, int n_decode,
                         cudaStream_t s);

// Prefill runs on the tcgen05 kernel: a work item is two Q tiles of
// pf_tile_rows(G) = G * floor(128 / G) rows (whole tokens of G query heads;
// 128 for powers of two, the rest of the 128 TMEM lanes idle otherwise).
// It needs G <= 128 (any pool format).
constexpr int kPfQTile = 128;
constexpr int pf_tile_rows(int G) { return G * (kPfQTile / G); }
// A prefill item split over key ranges keeps one partial per range: 2 Q
// tiles of 128 rows, i.e. kPfPartSlots decode partial slots; a range holds
// at least kPfMinSplitTiles 128-key tiles.
constexpr int kPfPartSlots = 2 * kPfQTile / kDecCols;
constexpr int kPfMinSplitTiles = 2;
constexpr int kPfMaxSplits = 32;
inline bool prefill_uses_tc(const pkv_config &c) {
  const int G = c.num_q_heads / c.num_kv_heads;
  return G > 0 && G <= kPfQTile;
}
cudaError_t configure_kernels();

}  // namespace pkv
