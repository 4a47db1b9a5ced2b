// libpkv host side: the C ABI of include/pkv.h.  Argument validation, the
// work planner (split-KV decode items and prefill tiles), workspace, TMA
// descriptors for the paged pools, kernel launches and timing.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pkv_internal.h"

namespace pkv {
cudaError_t configure_decode();
cudaError_t configure_prefill_tc();
cudaError_t configure_mixed();
}  // namespace pkv

using namespace pkv;

namespace {

constexpr int kTimingSlots = 4096;
constexpr int kMaxPartials = 16384;        // split-KV partial slots
constexpr int64_t kMaxPoolRows = (int64_t(1) << 31) - 4096;

thread_local std::string g_create_error;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

std::string fmt(const char *f, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, f);
  vsnprintf(buf, sizeof buf, f, ap);
  va_end(ap);
  return buf;
}

// Planner: split-KV decode items and prefill tiles, longest first.
struct Plan {
  std::vector<pkv_work_item> dec, pre;
  int partials = 0;
  int dec_groups = 0;   // split decode pairs: their first ranges lead `dec`
  int dec_max_split = 1;   // most ranges of one decode pair
  int pre_groups = 0;   // split prefill items: their first ranges lead `pre`
  // scratch of make_plan; a handle keeps its Plan from step to step, so
  // these (and dec, pre) stop allocating once they have grown
  std::vector<pkv_work_item> tmp;
  std::vector<int64_t> unit_cost, unit_id, group_cost;
  std::vector<uint64_t> keys;
  std::vector<std::pair<int64_t, int32_t>> groups, tiles;
};

// Moves the items for which lead(item) holds to the front of v, both parts
// in their order (a stable partition through the scratch vector tmp);
// returns how many lead.
template <class F>
int lead_first(std::vector<pkv_work_item> &v, std::vector<pkv_work_item> &tmp, F lead) {
  tmp.clear();
  for (const auto &w : v)
    if (lead(w)) tmp.push_back(w);
  const int n = static_cast<int>(tmp.size());
  if (n == 0) return 0;
  for (const auto &w : v)
    if (!lead(w)) tmp.push_back(w);
  v.swap(tmp);
  return n;
}

struct TimingRing {
  cudaEvent_t start[kTimingSlots];
  cudaEvent_t stop[kTimingSlots];
  int count = 0;
};

}  // namespace

struct pkv_handle {
  pkv_config cfg{};
  Plan plan;   // the last step's plan (its vectors keep their capacity)
  int device = 0;
  int num_sms = 0;
  std::string last_error;
  // workspace
  uint8_t *d_work = nullptr;      // work list + host-mirror copies
  size_t work_bytes = 0;
  int max_items = 0;
  float *d_part_o = nullptr;
  float *d_part_lse = nullptr;
  int32_t *d_err = nullptr;
  // E4M3 / NVFP4 pools: V (and NVFP4 K) staged as bf16 for the tensor-core
  // prefill (stage_kv.cu), stage_blocks blocks of [hkv][bs][128] each,
  // NVFP4 K's block scales, and the pools' tensor maps
  __nv_bfloat16 *d_stage_k = nullptr, *d_stage_v = nullptr;
  float *d_stage_ks = nullptr;   // [stage_blocks][hkv]
  int64_t stage_blocks = 0;
  CUtensorMap stage_map_k{}, stage_map_v{};
  uint8_t *h_stage[2] = {nullptr, nullptr};   // pinned staging (double buffer)
  cudaEvent_t staged[2] = {nullptr, nullptr};
  int stage_cur = 0;
  // timing
  bool timing = false;
  TimingRing rings[PKV_KERNEL_KINDS];
  // cached pool descriptors
  const void *map_k_ptr = nullptr, *map_v_ptr = nullptr;
  CUtensorMap dec_k{}, dec_v{}, pf_k{}, pf_v{};
  // CUDA-graph capture: a step prepared by pkv_graph_prepare (work list and
  // mirrors in their own device buffer, lengths kept to check the capture)
  uint8_t *d_graph_work = nullptr;
  bool graph_ready = false;
  std::vector<int32_t> graph_qsl, graph_lens;
  bool capturing = false;   // set while a call enqueues onto a capturing stream
};

namespace {

pkv_status fail(pkv_handle *h, pkv_status s, const std::string &msg) {
  if (h) h->last_error = msg;
  return s;
}

pkv_status cuda_fail(pkv_handle *h, cudaError_t e, const char *what) {
  return fail(h, PKV_ERR_CUDA, fmt("%s: %s", what, cudaGetErrorString(e)));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

std::string check_config(const pkv_config *c, pkv_status *st) {
  *st = PKV_ERR_INVALID_ARG;
  if (c == nullptr) return "config is NULL";
  if (c->num_kv_heads <= 0 || c->num_q_heads <= 0 ||
      c->num_q_heads % c->num_kv_heads != 0)
    return fmt("num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
               c->num_q_heads, c->num_kv_heads);
  if (!(c->softmax_scale > 0.f) || c->softmax_scale > 1e30f)
    return "softmax_scale must be finite and > 0";
  if (c->num_blocks <= 0) return "num_blocks must be > 0";
  if (c->max_num_seqs <= 0 || c->max_num_tokens <= 0)
    return "max_num_seqs and max_num_tokens must be > 0";
  if (c->kv_dtype != PKV_KV_BF16 && c->kv_dtype != PKV_KV_FP8_E4M3 &&
      c->kv_dtype != PKV_KV_NVFP4)
    return fmt("unknown kv_dtype %d", c->kv_dtype);
  if (c->flags & ~static_cast<uint32_t>(PKV_FLAG_VALIDATE | PKV_FLAG_TIMING | PKV_FLAG_SEPARATE))
    return fmt("unknown flag bits 0x%x", c->flags);
  if (c->stage_tokens < 0) return "stage_tokens must be >= 0";
  *st = PKV_ERR_UNSUPPORTED;
  if (c->head_dim != kHeadDim) return fmt("head_dim %d is not supported (only 128)", c->head_dim);
  const int bs = c->block_size;
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128 && bs != 256)
    return fmt("block_size %d is not supported (16, 32, 64, 128 or 256)", bs);
  // NVFP4 pools are addressed in 64-byte rows: 9 per 8 tokens
  const int64_t pool_rows = c->num_blocks * c->num_kv_heads * bs *
                            (c->kv_dtype == PKV_KV_NVFP4 ? 9 : 8) / 8;
  if (pool_rows > kMaxPoolRows)
    return "pool too large: num_blocks * num_kv_heads * block_size must be < 2^31 - 4096 "
           "(NVFP4: 8/9 of that)";
  *st = PKV_OK;
  return "";
}


// Keys an item list walks for a sequence of L keys: all of them, or, for
// context-parallel shard r of n with tokens dealt out in runs of k (run j
// to shard j % n), the shard's own keys; with dcp[3] set (runs shorter than
// a decode stage) every key, the others masked in the kernel.
int64_t shard_keys(int64_t L, const int32_t *dcp) {
  if (dcp == nullptr || dcp[0] <= 1 || dcp[3]) return L;
  const int64_t n = dcp[0], r = dcp[1], k = dcp[2];
  const int64_t runs = L / k, rem = L % k;
  return (runs / n) * k + (runs % n > r ? k : 0) + (runs % n == r ? rem : 0);
}

std::string make_plan(const pkv_config &c, const int32_t *qsl, const int32_t *lens,
                      int32_t B, int32_t T, int num_sms, int max_partials, Plan *plan,
                      pkv_status *st, const int32_t *dcp = nullptr) {
  *st = PKV_ERR_INVALID_ARG;
  if (B < 0 || T < 0) return "num_seqs and num_tokens must be >= 0";
  if (B > 0 && (qsl == nullptr || lens == nullptr))
    return "query_start_loc_host and seq_lens_host are required";
  plan->dec.clear();
  plan->pre.clear();
  plan->partials = plan->dec_groups = plan->pre_groups = 0;
  plan->dec_max_split = 1;
  if (B == 0) {
    if (T != 0) return "num_tokens must be 0 when num_seqs is 0";
    *st = PKV_OK;
    return "";
  }
  if (qsl[0] != 0) return "query_start_loc_host[0] must be 0";
  if (qsl[B] != T)
    return fmt("query_start_loc_host[num_seqs] = %d but num_tokens = %d", qsl[B], T);
  const int G = c.num_q_heads / c.num_kv_heads;
  const int H = c.num_kv_heads;
  int64_t dec_keys = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t q = int64_t(qsl[i + 1]) - qsl[i];
    if (q < 0) return fmt("query_start_loc_host decreases at %d", i);
    if (lens[i] < q) return fmt("seq_lens_host[%d] = %d is less than its %lld new tokens", i, lens[i], (long long)q);
    if (q > 0 && q * G <= kDecCols) dec_keys += shard_keys(lens[i], dcp) * H;
    if (dcp != nullptr && q * G > kDecCols) {
      *st = PKV_ERR_UNSUPPORTED;
      return fmt("request %d has %lld query rows per KV head; shard partials cover decode "
                 "rows (q * G <= %d) only", i, (long long)(q * G), kDecCols);
    }
  }
  // decode split size: ~4 whole waves of the resident decode CTAs (2 per SM
  // for bf16 pools, 3 for E4M3 and NVFP4), at least 1024 keys
  const int64_t resident = c.kv_dtype == PKV_KV_BF16       ? 2
                           : c.kv_dtype == PKV_KV_FP8_E4M3 ? 3
                                                           : kDecCtasNvfp4;
  const int64_t target = 4 * resident * std::max(num_sms, 1);
  int64_t chunk = std::max<int64_t>(1024, (dec_keys / target + kSplitAlign - 1) / kSplitAlign * kSplitAlign);
  for (;;) {
    int64_t parts = 0;
    for (int i = 0; i < B; ++i) {
      const int64_t q = int64_t(qsl[i + 1]) - qsl[i];
      if (q > 0 && q * G <= kDecCols) {
        const int64_t ns = (shard_keys(lens[i], dcp) + chunk - 1) / chunk;
        if (ns > 1) parts += ns * H;
      }
    }
    if (parts <= max_partials) break;
    chunk *= 2;
  }
  int part = 0;
  for (int i = 0; i < B; ++i) {
    const int q = qsl[i + 1] - qsl[i];
    if (q == 0) continue;
    const int L = lens[i];
    const int hist = L - q;
    if (q * G <= kDecCols) {
      // a shard may own no key of a short request: it still writes (0, -inf)
      const int64_t Ls = shard_keys(L, dcp);
      const int ns = std::max(1, static_cast<int>((Ls + chunk - 1) / chunk));
      for (int h = 0; h < H; ++h) {
        const int base = ns > 1 ? part : -1;
        for (int s = 0; s < ns; ++s) {
          pkv_work_item w{};
          w.kind = 0;
          w.seq = i;
          w.kv_head = h;
          w.tok0 = qsl[i];
          w.row0 = 0;
          w.n_rows = q * G;
          w.hist = hist;
          w.k_begin = static_cast<int32_t>(s * chunk);
          w.k_end = static_cast<int32_t>(std::min<int64_t>(Ls, (s + 1) * chunk));
          w.part = ns > 1 ? part++ : -1;
          w.pair = base;
          w.n_split = ns;
          plan->dec.push_back(w);
        }
      }
    } else if (!prefill_uses_tc(c)) {
      // E4M3 pools and groups above 128: the decode kernel takes the prefill
      // rows in chunks of kDecCols, each over its own causal key range.  The
      // chunks of one (request, KV head) are adjacent in the list, so CTAs
      // running together read the same keys and mostly hit L2.
      const int rows = q * G;
      for (int h = 0; h < H; ++h) {
        for (int r0 = 0; r0 < rows; r0 += kDecCols) {
          pkv_work_item w{};
          w.kind = 0;
          w.seq = i;
          w.kv_head = h;
          w.tok0 = qsl[i];
          w.row0 = r0;
          w.n_rows = std::min(kDecCols, rows - r0);
          w.hist = hist;
          w.k_begin = 0;
          w.k_end = hist + (r0 + w.n_rows - 1) / G + 1;
          w.part = -1;
          w.pair = -1;
          w.n_split = 1;
          plan->dec.push_back(w);
        }
      }
    } else {
      const int rows = q * G;
      const int tile = 2 * pf_tile_rows(std::min(G, kPfQTile));
      for (int h = 0; h < H; ++h) {
        for (int r0 = 0; r0 < rows; r0 += tile) {
          pkv_work_item w{};
          w.kind = 1;
          w.seq = i;
          w.kv_head = h;
          w.tok0 = qsl[i];
          w.row0 = r0;
          w.n_rows = std::min(tile, rows - r0);
          w.hist = hist;
          w.k_begin = 0;
          w.k_end = hist + (r0 + w.n_rows - 1) / G + 1;
          w.part = -1;
          w.pair = -1;
          w.n_split = 1;
          plan->pre.push_back(w);
        }
      }
    }
  }
  // Few prefill tiles leave most SMs idle while each walks its whole key
  // range (an incremental prefill of a few new tokens over a long history):
  // split the key ranges into runs of whole 128-key tiles so that the step
  // has about one tile per SM; each range writes a partial (O / l and the
  // log-sum-exp), merged by a second small kernel.  Boundaries lie at
  // multiples of 128 keys and of the block size, at or below the item's
  // first query position, so every query row sees at least one key in
  // every range.  A prefill partial slot is kPfPartSlots decode slots (256
  // rows) of the same partial buffers.
  if (dcp == nullptr && !plan->pre.empty() &&
      int64_t(plan->pre.size()) * 2 <= std::max(num_sms, 1)) {
    int64_t total_tiles = 0;
    for (const auto &w : plan->pre) total_tiles += (w.k_end + 127) / 128;
    std::vector<pkv_work_item> &split = plan->tmp;
    split.clear();
    for (const auto &w : plan->pre) {
      const int nt = (w.k_end + 127) / 128;
      const int unit = std::max(1, c.block_size / 128);    // boundary granularity, tiles
      // last allowed boundary, in tiles
      const int max_bound = (w.hist + w.row0 / G) / (128 * unit) * unit;
      const int want = static_cast<int>(
          std::min<int64_t>(nt, std::max<int64_t>(1, (int64_t(num_sms) * nt + total_tiles / 2) /
                                                         std::max<int64_t>(total_tiles, 1))));
      int ns = std::min({want, nt / kPfMinSplitTiles, max_bound + 1, kPfMaxSplits});
      if (ns > 1 && part + int64_t(ns) * kPfPartSlots > max_partials) ns = 1;
      if (ns <= 1) {
        split.push_back(w);
        continue;
      }
      const int cs = ((nt + ns - 1) / ns + unit - 1) / unit * unit;   // tiles per range
      int bounds = 0;                       // interior boundaries s * cs <= max_bound
      while (bounds + 1 < ns && (bounds + 1) * cs <= max_bound) ++bounds;
      ns = bounds + 1;
      if (ns <= 1) {
        split.push_back(w);
        continue;
      }
      const int base = part;
      for (int s = 0; s < ns; ++s) {
        pkv_work_item v = w;
        v.k_begin = s * cs * 128;
        v.k_end = s + 1 < ns ? (s + 1) * cs * 128 : w.k_end;
        v.part = part;
        v.pair = base;
        v.n_split = ns;
        part += kPfPartSlots;
        split.push_back(v);
      }
    }
    plan->pre.swap(split);
  }
  plan->partials = part;
  // Decode items longest first.  Prefill row chunks (row0 > 0 or more than
  // one chunk per request) stay together per (request, KV head), the group
  // placed by its longest chunk, so the CTAs of a group run side by side.
  auto dec_cost = [](const pkv_work_item &w) { return int64_t(w.k_end) - w.k_begin; };
  {
    const size_t n = plan->dec.size();
    std::vector<int64_t> &unit_cost = plan->unit_cost, &unit_id = plan->unit_id;
    std::vector<int64_t> &group_max = plan->group_cost;
    unit_cost.resize(n);
    unit_id.resize(n);
    group_max.assign(size_t(B) * H, -1);
    auto chunked = [&](const pkv_work_item &w) {
      return int64_t(qsl[w.seq + 1] - qsl[w.seq]) * G > kDecCols;
    };
    for (const auto &w : plan->dec)
      if (chunked(w)) {
        int64_t &m = group_max[size_t(w.seq) * H + w.kv_head];
        m = std::max(m, dec_cost(w));
      }
    for (size_t k = 0; k < n; ++k) {
      const pkv_work_item &w = plan->dec[k];
      const bool ch = chunked(w);
      unit_cost[k] = ch ? group_max[size_t(w.seq) * H + w.kv_head] : dec_cost(w);
      unit_id[k] = ch ? int64_t(w.seq) * H + w.kv_head : int64_t(B) * H + int64_t(k);
    }
    std::vector<pkv_work_item> &sorted = plan->tmp;
    sorted.resize(n);
    bool any_chunked = false;
    for (size_t k = 0; k < n && !any_chunked; ++k) any_chunked = unit_id[k] < int64_t(B) * H;
    if (!any_chunked) {
      // every item its own unit: cost descending, then item order.  All
      // ranges but a request's last have the full split length, the largest
      // cost: those lead in item order, and only the others are sorted (one
      // 64-bit key each; costs and indices below 2^31)
      int64_t top = 0;
      for (size_t k = 0; k < n; ++k) top = std::max(top, unit_cost[k]);
      std::vector<uint64_t> &keys = plan->keys;
      keys.clear();
      size_t m = 0;
      for (size_t k = 0; k < n; ++k) {
        if (unit_cost[k] == top)
          sorted[m++] = plan->dec[k];
        else
          keys.push_back((uint64_t(0x7FFFFFFF - unit_cost[k]) << 32) | uint64_t(k));
      }
      std::sort(keys.begin(), keys.end());
      for (const uint64_t key : keys) sorted[m++] = plan->dec[key & 0xFFFFFFFFu];
    } else {
      // unit cost descending, unit id ascending, own cost descending, then
      // the original index: the order a stable sort on the first three gives
      struct Key {
        int64_t cost, unit;
        int32_t own, idx;
        bool operator<(const Key &o) const {
          if (cost != o.cost) return cost > o.cost;
          if (unit != o.unit) return unit < o.unit;
          if (own != o.own) return own > o.own;
          return idx < o.idx;
        }
      };
      std::vector<Key> keys(n);
      for (size_t k = 0; k < n; ++k)
        keys[k] = Key{unit_cost[k], unit_id[k], static_cast<int32_t>(dec_cost(plan->dec[k])),
                      static_cast<int32_t>(k)};
      std::sort(keys.begin(), keys.end());
      for (size_t k = 0; k < n; ++k) sorted[k] = plan->dec[keys[k].idx];
    }
    plan->dec.swap(sorted);
    // the first range of each split pair leads the list (the merge kernel
    // takes its groups from there); these are full-length ranges, so the
    // longest-first order barely moves
    plan->dec_groups = lead_first(plan->dec, plan->tmp, [](const pkv_work_item &w) {
      return w.part >= 0 && w.part == w.pair;
    });
    plan->dec_max_split = 1;
    for (const auto &w : plan->dec) plan->dec_max_split = std::max(plan->dec_max_split, int(w.n_split));
  }
  // Prefill tiles of one (request, KV head) read the same K/V stream: keep
  // them adjacent so the CTAs running together share it through L2, and
  // order the groups longest first.
  auto pre_cost = [](const pkv_work_item &w) {
    return (int64_t(w.k_end) - w.k_begin) * w.n_rows;
  };
  std::vector<int64_t> &group_cost = plan->group_cost;
  group_cost.assign(size_t(B) * H, 0);
  for (const auto &w : plan->pre) group_cost[size_t(w.seq) * H + w.kv_head] += pre_cost(w);
  {
    // The tiles of one (request, KV head) are adjacent in plan->pre (built
    // per request and KV head; a split keeps its ranges in place): order the
    // groups by cost descending, then (request, KV head), and the tiles of a
    // group by cost descending, then their original order.
    const size_t n = plan->pre.size();
    std::vector<std::pair<int64_t, int32_t>> &groups = plan->groups;   // (cost, first tile)
    groups.clear();
    for (size_t k = 0; k < n; ++k) {
      const pkv_work_item &w = plan->pre[k];
      if (k == 0 || w.seq != plan->pre[k - 1].seq || w.kv_head != plan->pre[k - 1].kv_head)
        groups.emplace_back(group_cost[size_t(w.seq) * H + w.kv_head], static_cast<int32_t>(k));
    }
    // cost descending, first tile ascending (the groups' original order)
    std::sort(groups.begin(), groups.end(),
              [](const std::pair<int64_t, int32_t> &a, const std::pair<int64_t, int32_t> &b) {
                return a.first != b.first ? a.first > b.first : a.second < b.second;
              });
    std::vector<pkv_work_item> &sorted = plan->tmp;
    sorted.clear();
    std::vector<std::pair<int64_t, int32_t>> &tiles = plan->tiles;   // (-cost, index)
    for (const auto &gr : groups) {
      size_t e = size_t(gr.second) + 1;
      const pkv_work_item &w0 = plan->pre[size_t(gr.second)];
      while (e < n && plan->pre[e].seq == w0.seq && plan->pre[e].kv_head == w0.kv_head) ++e;
      tiles.clear();
      for (size_t k = size_t(gr.second); k < e; ++k)
        tiles.emplace_back(-pre_cost(plan->pre[k]), static_cast<int32_t>(k));
      std::sort(tiles.begin(), tiles.end());
      for (const auto &tl : tiles) sorted.push_back(plan->pre[size_t(tl.second)]);
    }
    plan->pre.swap(sorted);
  }
  // the first range of each split item leads the list: the merge kernel
  // takes its groups from there
  plan->pre_groups = lead_first(plan->pre, plan->tmp, [](const pkv_work_item &w) {
    return w.part >= 0 && w.part == w.pair;
  });
  *st = PKV_OK;
  return "";
}

// NVFP4 pool as rows of 64 bytes (code rows and micro-scale rows alike);
// boxes of one group's code rows, 64-byte swizzled.
bool encode_nvfp4_map(CUtensorMap *m, const void *base, int64_t rows, int box_rows,
                      bool swizzle = true) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_pool_map(CUtensorMap *m, const void *base, bool fp8, int64_t rows,
                     int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * (fp8 ? 1 : 2))};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(fp8 ? 128 : 64),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q viewed as [T][Hq][128] bf16 with boxes of {64 columns, G heads, 128/G
// tokens}: one box is a 64-column half of a 128-row prefill tile with rows
// r = t * G + g, 128-byte swizzled.
bool encode_q_map(CUtensorMap *m, const void *q, int hq, int group, int64_t tokens) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(hq), cuuint64_t(tokens)};
  const cuuint64_t strides[2] = {cuuint64_t(kHeadDim * 2), cuuint64_t(hq) * kHeadDim * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(kPfQTile / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K/V staging of a step's tensor-core prefill requests over E4M3 / NVFP4
// pools (stage_kv.cu): base[i] = first staging block of request i (-1: not
// staged) and reqs = (request, first block, context length) per staged
// request.  Returns the staging blocks used, or 0 when the step does not
// stage (bf16 pools, no such request, or more blocks than the handle has).
int64_t plan_staging(const pkv_config &c, int64_t capacity, const int32_t *qsl,
                     const int32_t *lens, int B, std::vector<int32_t> *base,
                     std::vector<int32_t> *reqs) {
  base->assign(size_t(std::max(B, 0)), -1);
  reqs->clear();
  if (c.kv_dtype == PKV_KV_BF16 || capacity <= 0 || !prefill_uses_tc(c)) return 0;
  const int G = c.num_q_heads / c.num_kv_heads;
  int64_t next = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t q = int64_t(qsl[i + 1]) - qsl[i];
    if (q * G <= kDecCols) continue;
    (*base)[i] = static_cast<int32_t>(std::min<int64_t>(next, INT32_MAX));
    reqs->insert(reqs->end(), {i, (*base)[i], lens[i]});
    next += (int64_t(lens[i]) + c.block_size - 1) / c.block_size;
  }
  if (next == 0 || next > capacity) {
    base->assign(size_t(B), -1);
    reqs->clear();
    return 0;
  }
  return next;
}

// Offsets in the work buffer: the work items, the host mirrors (validate
// mode), then the staging bases (per request) and staged requests (3 ints
// each).
size_t mirror_offset(int max_items);
size_t stage_base_offset(int max_items, int max_seqs) {
  return (mirror_offset(max_items) + sizeof(int32_t) * (2 * size_t(max_seqs) + 1) + 15) & ~size_t(15);
}
size_t stage_reqs_offset(int max_items, int max_seqs) {
  return stage_base_offset(max_items, max_seqs) + sizeof(int32_t) * size_t(max_seqs);
}

// 16-token pools viewed as [2 halves][rows][64 columns] (the halves 128 B
// apart, rows 256 B apart) with boxes of {64, 16, 2}: one box carries a whole
// (block, KV head) tile of 4 KB as [half][16 rows][64], 128-byte swizzled.
size_t items_bytes(int max_items) { return sizeof(pkv_work_item) * size_t(max_items); }
size_t mirror_offset(int max_items) { return items_bytes(max_items); }

// Lays out a plan's work items (decode items, then prefill tiles) at `dst`,
// the host mirrors at dst + mirror_off in validate mode, and the K/V staging
// tables (when the step stages) at their offsets; returns the bytes of the
// work items.
size_t stage_plan(const Plan &plan, const int32_t *qsl_host, const int32_t *lens_host,
                  int num_seqs, bool validate, size_t mirror_off, uint8_t *dst,
                  const std::vector<int32_t> &sbase, const std::vector<int32_t> &sreqs,
                  size_t base_off, size_t reqs_off) {
  std::memcpy(dst, plan.dec.data(), items_bytes(plan.dec.size()));
  std::memcpy(dst + items_bytes(plan.dec.size()), plan.pre.data(), items_bytes(plan.pre.size()));
  if (validate) {
    std::memcpy(dst + mirror_off, qsl_host, sizeof(int32_t) * (num_seqs + 1));
    std::memcpy(dst + mirror_off + sizeof(int32_t) * (num_seqs + 1), lens_host,
                sizeof(int32_t) * num_seqs);
  }
  if (!sreqs.empty()) {
    std::memcpy(dst + base_off, sbase.data(), sizeof(int32_t) * sbase.size());
    std::memcpy(dst + reqs_off, sreqs.data(), sizeof(int32_t) * sreqs.size());
  }
  return items_bytes(plan.dec.size() + plan.pre.size());
}

void timing_begin(pkv_handle *h, int kind, cudaStream_t s) {
  if (!h->timing || h->capturing) return;
  TimingRing &r = h->rings[kind];
  cudaEventRecord(r.start[r.count % kTimingSlots], s);
}
void timing_end(pkv_handle *h, int kind, cudaStream_t s) {
  if (!h->timing || h->capturing) return;
  TimingRing &r = h->rings[kind];
  cudaEventRecord(r.stop[r.count % kTimingSlots], s);
  ++r.count;
}

// The merges of split key ranges (decode pairs, then prefill row tiles),
// after the attention kernels of the step, timed as one PKV_KERNEL_MERGE.
pkv_status launch_merges(pkv_handle *h, const DecodeParams &dp, const PrefillParams &pp,
                         const Plan &plan, cudaStream_t s) {
  if (plan.dec_groups == 0 && plan.pre_groups == 0) return PKV_OK;
  timing_begin(h, PKV_KERNEL_MERGE, s);
  cudaError_t e = launch_decode_merge(dp, plan.dec_groups, plan.dec_max_split, s);
  if (e == cudaSuccess) e = launch_prefill_merge(pp, plan.pre_groups, s);
  timing_end(h, PKV_KERNEL_MERGE, s);
  return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "merge launch");
}

}  // namespace

extern "C" {

const char *pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_OUT_OF_MEMORY: return "out of device memory";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
    case PKV_ERR_TIMEOUT: return "device-side wait timed out";
    case PKV_ERR_WORKSPACE: return "workspace too small for this step";
  }
  return "unknown status";
}

const char *pkv_last_error(const pkv_handle *h) {
  return h ? h->last_error.c_str() : g_create_error.c_str();
}

pkv_status pkv_create(const pkv_config *config, int device, pkv_handle **out) {
  g_create_error.clear();
  if (out == nullptr) {
    g_create_error = "out is NULL";
    return PKV_ERR_INVALID_ARG;
  }
  *out = nullptr;
  pkv_status st;
  std::string msg = check_config(config, &st);
  if (st != PKV_OK) {
    g_create_error = msg;
    return st;
  }
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess || device < 0 || device >= ndev) {
    g_create_error = fmt("no CUDA device %d (%s)", device,
                         e != cudaSuccess ? cudaGetErrorString(e) : "out of range");
    return PKV_ERR_CUDA;
  }
  if ((e = cudaSetDevice(device)) != cudaSuccess) {
    g_create_error = fmt("cudaSetDevice: %s", cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  if (encode_fn() == nullptr) {
    g_create_error = "cuTensorMapEncodeTiled is not available from the driver";
    return PKV_ERR_CUDA;
  }
  if ((e = configure_decode()) != cudaSuccess ||
      (e = configure_prefill_tc()) != cudaSuccess || (e = configure_mixed()) != cudaSuccess) {
    g_create_error = fmt("configuring kernels: %s", cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  pkv_handle *h = new pkv_handle();
  h->cfg = *config;
  h->device = device;
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device);
  const int64_t G = config->num_q_heads / config->num_kv_heads;
  // prefill rows: 256-row tiles on the tensor-core kernel, else chunks of
  // kDecCols rows on the decode kernel
  const int64_t pre_rows = prefill_uses_tc(*config)
                               ? 2 * pf_tile_rows(static_cast<int>(std::min<int64_t>(G, kPfQTile)))
                               : kDecCols;
  const int64_t pre_items =
      (int64_t(config->max_num_tokens) * G / pre_rows + config->max_num_seqs) * config->num_kv_heads;
  const int64_t max_items = kMaxPartials + int64_t(config->max_num_seqs) * config->num_kv_heads + pre_items;
  if (max_items > INT32_MAX / 2) {
    g_create_error = "max_num_tokens * query group too large for the work list";
    delete h;
    return PKV_ERR_INVALID_ARG;
  }
  h->max_items = static_cast<int>(max_items);
  h->work_bytes = stage_reqs_offset(h->max_items, config->max_num_seqs) +
                  sizeof(int32_t) * 3 * size_t(config->max_num_seqs);
  if (config->kv_dtype != PKV_KV_BF16 && config->stage_tokens > 0 && prefill_uses_tc(*config)) {
    h->stage_blocks = (config->stage_tokens + config->block_size - 1) / config->block_size;
    if (h->stage_blocks * config->num_kv_heads * config->block_size > kMaxPoolRows) {
      g_create_error = "stage_tokens too large: the staging pools would exceed 2^31 - 4096 rows";
      delete h;
      return PKV_ERR_INVALID_ARG;
    }
  }
  bool ok = cudaMalloc(&h->d_work, h->work_bytes) == cudaSuccess &&
            cudaMalloc(&h->d_part_o, sizeof(float) * size_t(kMaxPartials) * kDecCols * kHeadDim) == cudaSuccess &&
            cudaMalloc(&h->d_part_lse, sizeof(float) * size_t(kMaxPartials) * kDecCols) == cudaSuccess &&
            cudaMalloc(&h->d_err, sizeof(int32_t)) == cudaSuccess &&
            cudaMallocHost(&h->h_stage[0], h->work_bytes) == cudaSuccess &&
            cudaMallocHost(&h->h_stage[1], h->work_bytes) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->staged[0], cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->staged[1], cudaEventDisableTiming) == cudaSuccess;
  if (ok) {
    ok = cudaMemset(h->d_err, 0, sizeof(int32_t)) == cudaSuccess;
  }
  if (ok && h->stage_blocks > 0) {
    // E4M3 pools stage V alone (the prefill reads E4M3 K with FP8 MMAs)
    const bool with_k = config->kv_dtype == PKV_KV_NVFP4;
    const int64_t rows = h->stage_blocks * config->num_kv_heads * config->block_size;
    const size_t bytes = size_t(rows) * kHeadDim * sizeof(__nv_bfloat16);
    ok = cudaMalloc(&h->d_stage_v, bytes) == cudaSuccess &&
         encode_pool_map(&h->stage_map_v, h->d_stage_v, false, rows,
                         std::min(config->block_size, 128));
    if (ok && with_k)
      ok = cudaMalloc(&h->d_stage_k, bytes) == cudaSuccess &&
           cudaMalloc(&h->d_stage_ks, sizeof(float) * size_t(h->stage_blocks) *
                                          config->num_kv_heads) == cudaSuccess &&
           encode_pool_map(&h->stage_map_k, h->d_stage_k, false, rows,
                           std::min(config->block_size, 128));
  }
  if (ok && (config->flags & PKV_FLAG_TIMING)) {
    h->timing = true;
    for (auto &r : h->rings)
      for (int i = 0; i < kTimingSlots && ok; ++i)
        ok = cudaEventCreate(&r.start[i]) == cudaSuccess &&
             cudaEventCreate(&r.stop[i]) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    pkv_destroy(h);
    g_create_error = "could not allocate the workspace";
    return PKV_ERR_OUT_OF_MEMORY;
  }
  *out = h;
  return PKV_OK;
}

pkv_status pkv_destroy(pkv_handle *h) {
  if (h == nullptr) return PKV_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->d_work);
  cudaFree(h->d_graph_work);
  cudaFree(h->d_part_o);
  cudaFree(h->d_part_lse);
  cudaFree(h->d_err);
  cudaFree(h->d_stage_k);
  cudaFree(h->d_stage_v);
  cudaFree(h->d_stage_ks);
  for (int i = 0; i < 2; ++i) {
    if (h->h_stage[i]) cudaFreeHost(h->h_stage[i]);
    if (h->staged[i]) cudaEventDestroy(h->staged[i]);
  }
  if (h->timing)
    for (auto &r : h->rings)
      for (int i = 0; i < kTimingSlots; ++i) {
        if (r.start[i]) cudaEventDestroy(r.start[i]);
        if (r.stop[i]) cudaEventDestroy(r.stop[i]);
      }
  delete h;
  return PKV_OK;
}

pkv_status pkv_write_slots(pkv_handle *h, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, int32_t num_tokens,
                           void *k_cache, void *v_cache, const float *k_scale,
                           const float *v_scale, void *stream) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  if (num_tokens < 0) return fail(h, PKV_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (num_tokens > h->cfg.max_num_tokens)
    return fail(h, PKV_ERR_INVALID_ARG,
                fmt("num_tokens %d exceeds max_num_tokens %d", num_tokens, h->cfg.max_num_tokens));
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
    return fail(h, PKV_ERR_INVALID_ARG, "NULL buffer");
  const bool quantised = h->cfg.kv_dtype != PKV_KV_BF16;
  if (quantised && (!k_scale || !v_scale))
    return fail(h, PKV_ERR_INVALID_ARG, "FP8 and NVFP4 pools need k_scale and v_scale");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(h, PKV_ERR_INVALID_ARG, "K/V buffers must be 16-byte aligned");
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  AppendParams p{};
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.slots = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = h->d_err;
  p.num_tokens = num_tokens;
  p.hkv = h->cfg.num_kv_heads;
  p.bs = h->cfg.block_size;
  p.num_blocks = h->cfg.num_blocks;
  p.validate = (h->cfg.flags & PKV_FLAG_VALIDATE) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return cuda_fail(h, e, "capture query");
  h->capturing = cap != cudaStreamCaptureStatusNone;
  timing_begin(h, PKV_KERNEL_APPEND, s);
  e = launch_append(p, h->cfg.kv_dtype, s);
  timing_end(h, PKV_KERNEL_APPEND, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "KV append launch");
  return PKV_OK;
}

}  // extern "C"

namespace {

// One attention step: the whole batch (dcp == NULL, bf16 out), or one
// context-parallel shard's partial (dcp = {n, r, k}: decode rows only, the
// shard's own keys, fp32 out_f32 and lse).
pkv_status attention_step(pkv_handle *h, const void *q, const void *k_cache,
                          const void *v_cache, const float *k_scale, const float *v_scale,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          const int32_t *block_tables, int32_t block_table_stride,
                          const int32_t *qsl_host, const int32_t *lens_host,
                          int32_t num_seqs, int32_t num_tokens, void *out, float *lse,
                          void *stream, const int32_t *dcp, float *out_f32) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  const pkv_config &c = h->cfg;
  if (num_seqs > c.max_num_seqs)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("num_seqs %d exceeds max_num_seqs %d", num_seqs, c.max_num_seqs));
  if (num_tokens > c.max_num_tokens)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("num_tokens %d exceeds max_num_tokens %d", num_tokens, c.max_num_tokens));
  Plan &plan = h->plan;
  pkv_status st;
  std::string msg = make_plan(c, qsl_host, lens_host, num_seqs, num_tokens, h->num_sms,
                              kMaxPartials, &plan, &st, dcp);
  if (st != PKV_OK) return fail(h, st, msg);
  if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !query_start_loc || !seq_lens || !block_tables ||
      !(out || out_f32))
    return fail(h, PKV_ERR_INVALID_ARG, "NULL buffer");
  const bool fp8 = c.kv_dtype == PKV_KV_FP8_E4M3;
  const bool nvfp4 = c.kv_dtype == PKV_KV_NVFP4;
  if ((fp8 || nvfp4) && (!k_scale || !v_scale))
    return fail(h, PKV_ERR_INVALID_ARG, "FP8 and NVFP4 pools need k_scale and v_scale");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(out_f32))
    return fail(h, PKV_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");
  const int bs = c.block_size;
  for (int i = 0; i < num_seqs; ++i) {
    const int64_t nb = (int64_t(lens_host[i]) + bs - 1) / bs;
    if (nb > block_table_stride)
      return fail(h, PKV_ERR_INVALID_ARG,
                  fmt("request %d needs %lld block-table entries but the stride is %d", i,
                      (long long)nb, block_table_stride));
  }
  const int n_items = static_cast<int>(plan.dec.size() + plan.pre.size());
  if (n_items > h->max_items)
    return fail(h, PKV_ERR_WORKSPACE, fmt("step needs %d work items, workspace holds %d", n_items, h->max_items));

  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return cuda_fail(h, e, "capture query");
  h->capturing = cap != cudaStreamCaptureStatusNone;
  if (h->capturing && dcp != nullptr)
    return fail(h, PKV_ERR_UNSUPPORTED, "shard partials are not captured in CUDA graphs");
  if (h->capturing &&
      !(h->graph_ready && int(h->graph_lens.size()) == num_seqs &&
        std::equal(h->graph_lens.begin(), h->graph_lens.end(), lens_host) &&
        std::equal(h->graph_qsl.begin(), h->graph_qsl.end(), qsl_host)))
    return fail(h, PKV_ERR_INVALID_ARG,
                "a captured step needs pkv_graph_prepare with the same query_start_loc and "
                "seq_lens first");

  // pool descriptors (re-encoded when the pools move)
  if (k_cache != h->map_k_ptr || v_cache != h->map_v_ptr) {
    const int64_t rows = c.num_blocks * c.num_kv_heads * bs;
    const int dec_box = std::min(bs, fp8 ? kDecKeysFp8 : kDecKeysBf16);
    const int pf_box = std::min(bs, 128);
    const int nv_box = std::min(std::min(bs, kNvfp4Group), kDecKeysNvfp4);
    bool ok = nvfp4 ? encode_nvfp4_map(&h->dec_k, k_cache, rows / 8 * 9, nv_box) &&
                          encode_nvfp4_map(&h->dec_v, v_cache, rows / 8 * 9, nv_box)
                    : encode_pool_map(&h->dec_k, k_cache, fp8, rows, dec_box) &&
                          encode_pool_map(&h->dec_v, v_cache, fp8, rows, dec_box);
    // prefill: NVFP4 boxes are whole row groups (codes then micro scales,
    // 9/8 rows of 64 bytes per token), unswizzled
    if (ok && nvfp4)
      ok = encode_nvfp4_map(&h->pf_k, k_cache, rows / 8 * 9, std::min(bs, kNvfp4Group) / 8 * 9,
                            false) &&
           encode_nvfp4_map(&h->pf_v, v_cache, rows / 8 * 9, std::min(bs, kNvfp4Group) / 8 * 9,
                            false);
    if (ok && !nvfp4)
      ok = encode_pool_map(&h->pf_k, k_cache, fp8, rows, pf_box) &&
           encode_pool_map(&h->pf_v, v_cache, fp8, rows, pf_box);
    if (!ok) {
      h->map_k_ptr = h->map_v_ptr = nullptr;
      return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled rejected the pool layout");
    }
    h->map_k_ptr = k_cache;
    h->map_v_ptr = v_cache;
  }

  // E4M3 / NVFP4 pools: stage the tensor-core prefill requests' K and V as
  // bf16 when they fit the handle's staging pools
  std::vector<int32_t> sbase, sreqs;
  const int64_t n_stage =
      dcp == nullptr
          ? plan_staging(c, h->stage_blocks, qsl_host, lens_host, num_seqs, &sbase, &sreqs)
          : 0;
  const size_t base_off = stage_base_offset(h->max_items, c.max_num_seqs);
  const size_t reqs_off = stage_reqs_offset(h->max_items, c.max_num_seqs);

  // the work list (+ host mirrors for validate mode, + staging tables) in
  // device memory
  const bool validate = (c.flags & PKV_FLAG_VALIDATE) != 0;
  const size_t mirror_off = items_bytes(h->max_items);
  uint8_t *work = h->d_work;
  if (h->capturing) {
    work = h->d_graph_work;   // uploaded by pkv_graph_prepare: nothing to copy
  } else {
    const int cur = h->stage_cur;
    h->stage_cur ^= 1;
    e = cudaEventSynchronize(h->staged[cur]);   // this buffer's previous copy is done
    if (e != cudaSuccess) return cuda_fail(h, e, "staging event");
    uint8_t *hs = h->h_stage[cur];
    const size_t nbytes = stage_plan(plan, qsl_host, lens_host, num_seqs, validate, mirror_off,
                                     hs, sbase, sreqs, base_off, reqs_off);
    e = cudaMemcpyAsync(h->d_work, hs, nbytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && validate)
      e = cudaMemcpyAsync(h->d_work + mirror_off, hs + mirror_off,
                          sizeof(int32_t) * (2 * num_seqs + 1), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && n_stage > 0)
      e = cudaMemcpyAsync(h->d_work + base_off, hs + base_off,
                          reqs_off - base_off + sizeof(int32_t) * sreqs.size(),
                          cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaEventRecord(h->staged[cur], s);
    if (e != cudaSuccess) return cuda_fail(h, e, "work-list upload");
  }
  const pkv_work_item *d_items = reinterpret_cast<const pkv_work_item *>(work);

  if (validate) {
    CheckParams cp{};
    cp.qsl = query_start_loc;
    cp.seq_lens = seq_lens;
    cp.block_tables = block_tables;
    cp.qsl_expect = reinterpret_cast<const int32_t *>(work + mirror_off);
    cp.seq_lens_expect = cp.qsl_expect + num_seqs + 1;
    cp.bt_stride = block_table_stride;
    cp.num_seqs = num_seqs;
    cp.bs = bs;
    cp.num_blocks = c.num_blocks;
    cp.err = h->d_err;
    if (fp8 || nvfp4) {
      cp.k_scale = k_scale;
      cp.v_scale = v_scale;
      cp.hkv = c.num_kv_heads;
    }
    if ((e = launch_check(cp, s)) != cudaSuccess) return cuda_fail(h, e, "check launch");
  }

  const float scale_log2 = c.softmax_scale * 1.4426950408889634f;
  const int G = c.num_q_heads / c.num_kv_heads;
  const int32_t rows_total = static_cast<int32_t>(c.num_blocks * c.num_kv_heads * bs);
  const int32_t nvfp4_rows = static_cast<int32_t>(c.num_blocks * c.num_kv_heads * bs / 8 * 9);
  DecodeParams dp{};
  dp.items = d_items;
  dp.q = static_cast<const __nv_bfloat16 *>(q);
  dp.block_tables = block_tables;
  dp.bt_stride = block_table_stride;
  dp.k_scale = k_scale;
  dp.v_scale = v_scale;
  dp.out = static_cast<__nv_bfloat16 *>(out);
  dp.lse = lse;
  dp.part_o = h->d_part_o;
  dp.part_lse = h->d_part_lse;
  dp.err = h->d_err;
  dp.hq = c.num_q_heads;
  dp.hkv = c.num_kv_heads;
  dp.group = G;
  dp.bs = bs;
  dp.rows_total = nvfp4 ? nvfp4_rows : rows_total;
  dp.k_pool = static_cast<const uint8_t *>(k_cache);
  dp.v_pool = static_cast<const uint8_t *>(v_cache);
  dp.num_blocks = c.num_blocks;
  dp.scale_log2 = scale_log2;
  dp.validate = validate;
  if (dcp != nullptr) {
    dp.dcp_n = dcp[0];
    dp.dcp_r = dcp[1];
    dp.dcp_k = dcp[2];
    dp.dcp_mask = dcp[0] > 1 ? dcp[3] : 0;
  }
  dp.out_f32 = out_f32;
  PrefillParams pp{};
  pp.items = d_items + plan.dec.size();
  pp.q = static_cast<const __nv_bfloat16 *>(q);
  pp.block_tables = block_tables;
  pp.bt_stride = block_table_stride;
  pp.k_scale = k_scale;
  pp.v_scale = v_scale;
  pp.out = static_cast<__nv_bfloat16 *>(out);
  pp.lse = lse;
  pp.err = h->d_err;
  pp.hq = c.num_q_heads;
  pp.hkv = c.num_kv_heads;
  pp.group = G;
  pp.bs = bs;
  pp.rows_total = nvfp4 ? nvfp4_rows : rows_total;
  pp.num_blocks = c.num_blocks;
  pp.scale_log2 = scale_log2;
  pp.validate = validate;
  pp.part_o = h->d_part_o;
  pp.part_lse = h->d_part_lse;
  const bool tc = prefill_uses_tc(c);
  CUtensorMap qmap;
  if (!plan.pre.empty() && tc && !encode_q_map(&qmap, q, c.num_q_heads, G, num_tokens))
    return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled rejected the query layout");
  const int n_dec = static_cast<int>(plan.dec.size());
  const int n_pre = static_cast<int>(plan.pre.size());
  if (n_dec > 0 && n_pre > 0 && tc && c.kv_dtype == PKV_KV_BF16 &&
      !(c.flags & PKV_FLAG_SEPARATE)) {
    // a mixed step: one launch for both kinds of work
    timing_begin(h, PKV_KERNEL_MIXED, s);
    e = launch_mixed(qmap, h->pf_k, h->pf_v, h->dec_k, h->dec_v, pp, dp, n_pre, n_dec, s);
    timing_end(h, PKV_KERNEL_MIXED, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "mixed-step launch");
    return launch_merges(h, dp, pp, plan, s);
  }
  if (n_dec > 0) {
    timing_begin(h, PKV_KERNEL_DECODE, s);
    e = launch_decode(h->dec_k, h->dec_v, dp, n_dec, c.kv_dtype, s);
    timing_end(h, PKV_KERNEL_DECODE, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "decode launch");
  }
  if (n_pre > 0 && n_stage > 0) {
    // NVFP4 K and V, or E4M3 V, converted once to bf16, then the prefill
    StageParams sp{};
    sp.k_pool = static_cast<const uint8_t *>(k_cache);
    sp.v_pool = static_cast<const uint8_t *>(v_cache);
    sp.k_scale = k_scale;
    sp.v_scale = v_scale;
    sp.block_tables = block_tables;
    sp.bt_stride = block_table_stride;
    sp.reqs = reinterpret_cast<const int32_t *>(work + reqs_off);
    sp.n_reqs = static_cast<int32_t>(sreqs.size() / 3);
    sp.k_stage = h->d_stage_k;
    sp.v_stage = h->d_stage_v;
    sp.k_stage_scale = h->d_stage_ks;
    sp.hkv = c.num_kv_heads;
    sp.bs = bs;
    sp.num_blocks = c.num_blocks;
    sp.err = h->d_err;
    timing_begin(h, PKV_KERNEL_STAGE, s);
    e = launch_stage_kv(sp, static_cast<int>(n_stage), c.kv_dtype, s);
    timing_end(h, PKV_KERNEL_STAGE, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "K/V staging launch");
    PrefillParams ps = pp;
    ps.stage_base = reinterpret_cast<const int32_t *>(work + base_off);
    ps.stage_blocks = n_stage;
    ps.stage_rows = static_cast<int32_t>(n_stage * c.num_kv_heads * bs);
    const bool with_k = c.kv_dtype == PKV_KV_NVFP4;
    if (with_k) {   // K from the staging pool too, with its staged block scales
      ps.k_scale = h->d_stage_ks;
      ps.v_scale = nullptr;
      ps.num_blocks = n_stage;
      ps.rows_total = ps.stage_rows;
    }
    timing_begin(h, PKV_KERNEL_PREFILL, s);
    e = launch_prefill_tc(qmap, with_k ? h->stage_map_k : h->pf_k, h->stage_map_v, ps, n_pre,
                          with_k ? kFmtStaged : kFmtStagedV, s);
    timing_end(h, PKV_KERNEL_PREFILL, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "prefill launch");
  } else if (n_pre > 0) {
    timing_begin(h, PKV_KERNEL_PREFILL, s);
    e = launch_prefill_tc(qmap, h->pf_k, h->pf_v, pp, n_pre, c.kv_dtype, s);
    timing_end(h, PKV_KERNEL_PREFILL, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "prefill launch");
  }
  return launch_merges(h, dp, pp, plan, s);
}

}  // namespace

extern "C" {

pkv_status pkv_attention_varlen(pkv_handle *h, const void *q, const void *k_cache,
                                const void *v_cache, const float *k_scale,
                                const float *v_scale, const int32_t *query_start_loc,
                                const int32_t *seq_lens, const int32_t *block_tables,
                                int32_t block_table_stride,
                                const int32_t *qsl_host, const int32_t *lens_host,
                                int32_t num_seqs, int32_t num_tokens, void *out,
                                float *lse, void *stream) {
  return attention_step(h, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens,
                        block_tables, block_table_stride, qsl_host, lens_host, num_seqs,
                        num_tokens, out, lse, stream, nullptr, nullptr);
}

pkv_status pkv_attention_partial(pkv_handle *h, const void *q, const void *k_cache,
                                 const void *v_cache, const float *k_scale,
                                 const float *v_scale, const int32_t *query_start_loc,
                                 const int32_t *seq_lens, const int32_t *block_tables,
                                 int32_t block_table_stride, const int32_t *qsl_host,
                                 const int32_t *lens_host, int32_t num_seqs,
                                 int32_t num_tokens, int32_t shard, int32_t num_shards,
                                 int32_t interleave, float *out, float *lse, void *stream) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  const int stage = h->cfg.kv_dtype == PKV_KV_FP8_E4M3 ? kDecKeysFp8
                    : h->cfg.kv_dtype == PKV_KV_NVFP4  ? kDecKeysNvfp4
                                                       : kDecKeysBf16;
  if (num_shards < 1 || shard < 0 || shard >= num_shards)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("shard %d of %d", shard, num_shards));
  if (interleave < 1)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("interleave %d: must be at least 1", interleave));
  if (out == nullptr || lse == nullptr)
    return fail(h, PKV_ERR_INVALID_ARG, "a partial needs out and lse");
  // runs that fill whole decode stages are read compactly; shorter ones
  // (the pages' interleave of 1) by walking every key and masking the rest
  const int32_t dcp[4] = {num_shards, shard, interleave, interleave % stage != 0 ? 1 : 0};
  return attention_step(h, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens,
                        block_tables, block_table_stride, qsl_host, lens_host, num_seqs,
                        num_tokens, nullptr, lse, stream, dcp, out);
}

pkv_status pkv_lse_merge(pkv_handle *h, const float *parts_o, const float *parts_lse,
                         int32_t num_parts, int64_t num_rows, void *out, float *lse,
                         void *stream) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  if (num_parts < 1 || num_rows < 0)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("num_parts %d, num_rows %lld", num_parts, (long long)num_rows));
  if (num_rows == 0) return PKV_OK;
  if (!parts_o || !parts_lse || !out)
    return fail(h, PKV_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned16(parts_o) || !aligned16(out))
    return fail(h, PKV_ERR_INVALID_ARG, "parts_o and out must be 16-byte aligned");
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  e = launch_lse_merge(parts_o, parts_lse, num_parts, num_rows,
                       static_cast<__nv_bfloat16 *>(out), lse, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "merge launch");
  return PKV_OK;
}

pkv_status pkv_rope_write_slots(pkv_handle *h, void *q, const void *k_new,
                                const void *v_new, const int64_t *positions,
                                const float *cos_sin_cache, int64_t max_pos, int32_t neox,
                                const int64_t *slot_mapping, int32_t num_tokens,
                                void *k_cache, void *v_cache, const float *k_scale,
                                const float *v_scale, void *stream) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  if (num_tokens < 0 || num_tokens > h->cfg.max_num_tokens)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("num_tokens %d outside [0, max_num_tokens]", num_tokens));
  if (num_tokens == 0) return PKV_OK;
  if (!q || !k_new || !v_new || !positions || !cos_sin_cache || !slot_mapping || !k_cache ||
      !v_cache)
    return fail(h, PKV_ERR_INVALID_ARG, "NULL buffer");
  if (max_pos < 1) return fail(h, PKV_ERR_INVALID_ARG, "max_pos must be >= 1");
  const bool quantised = h->cfg.kv_dtype != PKV_KV_BF16;
  if (quantised && (!k_scale || !v_scale))
    return fail(h, PKV_ERR_INVALID_ARG, "FP8 and NVFP4 pools need k_scale and v_scale");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(cos_sin_cache))
    return fail(h, PKV_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  RopeAppendParams rp{};
  rp.a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  rp.a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  rp.a.slots = slot_mapping;
  rp.a.k_cache = k_cache;
  rp.a.v_cache = v_cache;
  rp.a.k_scale = k_scale;
  rp.a.v_scale = v_scale;
  rp.a.err = h->d_err;
  rp.a.num_tokens = num_tokens;
  rp.a.hkv = h->cfg.num_kv_heads;
  rp.a.bs = h->cfg.block_size;
  rp.a.num_blocks = h->cfg.num_blocks;
  rp.a.validate = (h->cfg.flags & PKV_FLAG_VALIDATE) != 0;
  rp.q = static_cast<__nv_bfloat16 *>(q);
  rp.positions = positions;
  rp.cos_sin = cos_sin_cache;
  rp.max_pos = max_pos;
  rp.hq = h->cfg.num_q_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return cuda_fail(h, e, "capture query");
  h->capturing = cap != cudaStreamCaptureStatusNone;
  timing_begin(h, PKV_KERNEL_APPEND, s);
  e = launch_rope_append(rp, h->cfg.kv_dtype, neox != 0, s);
  timing_end(h, PKV_KERNEL_APPEND, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "rope + KV append launch");
  return PKV_OK;
}

pkv_status pkv_graph_prepare(pkv_handle *h, const int32_t *qsl_host,
                             const int32_t *lens_host, int32_t num_seqs,
                             int32_t num_tokens) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  const pkv_config &c = h->cfg;
  if (num_seqs > c.max_num_seqs || num_tokens > c.max_num_tokens)
    return fail(h, PKV_ERR_INVALID_ARG, "step larger than the handle serves");
  Plan &plan = h->plan;
  pkv_status st;
  std::string msg = make_plan(c, qsl_host, lens_host, num_seqs, num_tokens, h->num_sms,
                              kMaxPartials, &plan, &st);
  if (st != PKV_OK) return fail(h, st, msg);
  const int n_items = static_cast<int>(plan.dec.size() + plan.pre.size());
  if (n_items > h->max_items)
    return fail(h, PKV_ERR_WORKSPACE, fmt("step needs %d work items, workspace holds %d", n_items, h->max_items));
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  h->graph_ready = false;
  if (h->d_graph_work == nullptr && (e = cudaMalloc(&h->d_graph_work, h->work_bytes)) != cudaSuccess)
    return fail(h, PKV_ERR_OUT_OF_MEMORY, fmt("graph work list: %s", cudaGetErrorString(e)));
  std::vector<uint8_t> host(h->work_bytes, 0);
  const size_t mirror_off = items_bytes(h->max_items);
  std::vector<int32_t> sbase, sreqs;
  plan_staging(c, h->stage_blocks, qsl_host, lens_host, num_seqs, &sbase, &sreqs);
  stage_plan(plan, qsl_host, lens_host, num_seqs, true, mirror_off, host.data(), sbase, sreqs,
             stage_base_offset(h->max_items, c.max_num_seqs),
             stage_reqs_offset(h->max_items, c.max_num_seqs));
  // synchronous on purpose: the buffer must hold this plan before any replay
  if ((e = cudaMemcpy(h->d_graph_work, host.data(), h->work_bytes, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(h, e, "graph work-list upload");
  h->graph_qsl.assign(qsl_host, qsl_host + num_seqs + 1);
  h->graph_lens.assign(lens_host, lens_host + num_seqs);
  h->graph_ready = true;
  return PKV_OK;
}

pkv_status pkv_wait_selftest(pkv_handle *h, uint64_t limit_ns, void *stream) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  h->last_error.clear();
  if (limit_ns < 1 || limit_ns > kWaitLimitNs)
    return fail(h, PKV_ERR_INVALID_ARG,
                fmt("limit_ns %llu outside [1, %llu]", (unsigned long long)limit_ns,
                    (unsigned long long)kWaitLimitNs));
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  e = launch_wait_selftest(h->d_err, limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "wait self-test launch");
  return PKV_OK;
}

pkv_status pkv_check_device_errors(pkv_handle *h) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  cudaError_t e = cudaSetDevice(h->device);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "device");
  int32_t word = 0;
  e = cudaMemcpy(&word, h->d_err, sizeof word, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int32_t));
  if (e != cudaSuccess) return cuda_fail(h, e, "reading the error word");
  if (word & kErrTimeout)
    return fail(h, PKV_ERR_TIMEOUT, "a device-side wait gave up (error word 0x" + fmt("%x", word) + ")");
  if (word != 0) {
    std::string what;
    if (word & kErrBadBlock) what += " block-table entry outside the pool;";
    if (word & kErrBadSlot) what += " slot outside the pool;";
    if (word & kErrMismatch) what += " device metadata differs from the host mirrors;";
    if (word & kErrBadPosition) what += " rotary position outside the cos/sin cache;";
    if (word & kErrBadScale) what += " E4M3/NVFP4 block scale above 16 (or NaN);";
    return fail(h, PKV_ERR_DEVICE_CHECK, "device check:" + what);
  }
  return PKV_OK;
}

pkv_status pkv_plan(const pkv_config *config, const int32_t *qsl_host,
                    const int32_t *lens_host, int32_t num_seqs, int32_t num_tokens,
                    int32_t num_sms, pkv_work_item *items, int32_t max_items,
                    int32_t *num_items, int32_t *num_partials) {
  pkv_status st;
  std::string msg = check_config(config, &st);
  if (st != PKV_OK) {
    g_create_error = msg;
    return st;
  }
  static thread_local Plan plan;   // scratch reused by this thread's calls
  msg = make_plan(*config, qsl_host, lens_host, num_seqs, num_tokens, num_sms,
                  kMaxPartials, &plan, &st);
  if (st != PKV_OK) {
    g_create_error = msg;
    return st;
  }
  const int n = static_cast<int>(plan.dec.size() + plan.pre.size());
  if (num_items) *num_items = n;
  if (num_partials) *num_partials = plan.partials;
  if (items) {
    int k = 0;
    for (const auto &w : plan.dec)
      if (k < max_items) items[k++] = w;
    for (const auto &w : plan.pre)
      if (k < max_items) items[k++] = w;
  }
  return PKV_OK;
}

pkv_status pkv_timing_reset(pkv_handle *h) {
  if (h == nullptr) return PKV_OK;
  for (auto &r : h->rings) r.count = 0;
  return PKV_OK;
}

pkv_status pkv_timing_read(pkv_handle *h, int32_t kind, int32_t *launches,
                           double *total_ms) {
  if (launches) *launches = 0;
  if (total_ms) *total_ms = 0.0;
  if (h == nullptr) return PKV_OK;
  if (kind < 0 || kind >= PKV_KERNEL_KINDS)
    return fail(h, PKV_ERR_INVALID_ARG, fmt("unknown kernel kind %d", kind));
  if (!h->timing) return PKV_OK;
  TimingRing &r = h->rings[kind];
  const int n = std::min(r.count, kTimingSlots);
  double sum = 0.0;
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(r.stop[i]);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start[i], r.stop[i]);
    if (e != cudaSuccess) return cuda_fail(h, e, "timing events");
    sum += ms;
  }
  if (launches) *launches = n;
  if (total_ms) *total_ms = sum;
  return PKV_OK;
}

}  // extern "C"
