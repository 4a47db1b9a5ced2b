// pkv_decode_static: split-KV decode whose scratch lives in a fixed device
// array compiled into the library, for callers that cannot allocate GPU
// memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// pool or arena that owns every byte of the device (a serving engine that
// pre-reserves HBM for its KV cache), code that must not allocate after
// start-up for latency reasons, or host code that is not allowed to create a
// handle (pkv_create allocates its workspace).  This entry point takes only
// the caller's inputs and outputs; the work list, the split partials and
// the error word come from g_scratch below, which every GPU that loads the
// library holds until the process exits.
#include <algorithm>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
cudaError_t configure_decode();
}  // namespace pkv

namespace {

using namespace pkv;

// Limits of the static scratch.
constexpr int kStaticItems = 2048;      // decode work items per call
constexpr int kStaticPartials = 1024;   // split partial slots per call
constexpr int kMaxDevices = 64;

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kItemsOff = 0;
constexpr size_t kPartOOff = align256(kItemsOff + sizeof(pkv_work_item) * kStaticItems);
constexpr size_t kPartLseOff =
    align256(kPartOOff + sizeof(float) * size_t(kStaticPartials) * kDecCols * kHeadDim);
constexpr size_t kErrOff = align256(kPartLseOff + sizeof(float) * size_t(kStaticPartials) * kDecCols);
constexpr size_t kScratchBytes = align256(kErrOff + sizeof(int32_t));  // ~4.3 MB

// The scratch.  In host code this name is only a stand-in: its device address
// comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  The first use on a
// device loads the module there (lazy loading gives its device variables
// memory only then), sets the kernels' shared-memory limits and clears the
// error word, synchronously.
cudaError_t scratch_address(int device, uint8_t **out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[device] == nullptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    e = configure_decode();
    if (e != cudaSuccess) return e;
    e = cudaMemset(static_cast<uint8_t *>(p) + kErrOff, 0, sizeof(int32_t));
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = p;
  }
  *out = static_cast<uint8_t *>(g_scratch_ptr[device]);
  return cudaSuccess;
}

// Current device, checked against the per-device table.
cudaError_t current_device(int *dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e == cudaSuccess && (*dev < 0 || *dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
  return e;
}

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

bool encode_map(CUtensorMap *m, const void *base, bool fp8, int64_t rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(kHeadDim * (fp8 ? 1 : 2))};
  const cuuint32_t box[2] = {cuuint32_t(fp8 ? 128 : 64), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NVFP4 pool as rows of 64 bytes; boxes of code rows, 64-byte swizzled (the
// layout the NVFP4 decode reads).
bool encode_nvfp4_map(CUtensorMap *m, const void *base, int64_t rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {64, cuuint64_t(rows)};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host staging for the work list: a fixed array, no heap.  Serialised by
// g_plan_mutex; the upload copies it before cudaMemcpyAsync returns
// (pageable source).
std::mutex g_plan_mutex;
pkv_work_item g_items[kStaticItems];

}  // namespace

extern "C" pkv_status pkv_decode_static(
    const pkv_config *c, const void *q, const void *k_cache, const void *v_cache,
    const float *k_scale, const float *v_scale, const int32_t *block_tables,
    int32_t block_table_stride, const int32_t *qsl, const int32_t *lens,
    int32_t num_seqs, int32_t num_tokens, void *out, float *lse, void *stream) {
  if (c == nullptr || num_seqs < 0 || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
  const int bs = c->block_size;
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128 && bs != 256) return PKV_ERR_UNSUPPORTED;
  if (c->num_kv_heads <= 0 || c->num_q_heads <= 0 || c->num_q_heads % c->num_kv_heads ||
      c->num_blocks <= 0 || !(c->softmax_scale > 0.f))
    return PKV_ERR_INVALID_ARG;
  const bool nvfp4 = c->kv_dtype == PKV_KV_NVFP4;
  if (c->num_blocks * c->num_kv_heads * bs * (nvfp4 ? 9 : 8) / 8 >= (int64_t(1) << 31) - 4096)
    return PKV_ERR_UNSUPPORTED;
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (num_seqs == 0) {
    // nothing to run: the call only sets the device up (a warm-up)
    if (num_tokens != 0) return PKV_ERR_INVALID_ARG;
    uint8_t *unused = nullptr;
    return scratch_address(dev, &unused) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  if (!q || !k_cache || !v_cache || !block_tables || !qsl || !lens || !out)
    return PKV_ERR_INVALID_ARG;
  const bool fp8 = c->kv_dtype == PKV_KV_FP8_E4M3;
  if (c->kv_dtype != PKV_KV_BF16 && !fp8 && !nvfp4) return PKV_ERR_INVALID_ARG;
  if ((fp8 || nvfp4) && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  const int G = c->num_q_heads / c->num_kv_heads;
  const int H = c->num_kv_heads;
  if (qsl[0] != 0 || qsl[num_seqs] != num_tokens) return PKV_ERR_INVALID_ARG;
  int64_t keys = 0;
  int max_len = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int qi = qsl[i + 1] - qsl[i];
    if (qi < 0 || lens[i] < qi) return PKV_ERR_INVALID_ARG;
    if (qi * G > kDecCols) return PKV_ERR_UNSUPPORTED;   // decode rows only
    if ((int64_t(lens[i]) + bs - 1) / bs > block_table_stride) return PKV_ERR_INVALID_ARG;
    if (qi > 0) keys += int64_t(lens[i]) * H;
    max_len = std::max(max_len, int(lens[i]));
  }

  // split size: fill the machine, then grow until the static scratch holds it
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t chunk = std::max<int64_t>(1024, (keys / (8 * std::max(sms, 1)) + kSplitAlign - 1) /
                                              kSplitAlign * kSplitAlign);
  int64_t n_items = 0, n_parts = 0;
  for (;;) {
    n_items = n_parts = 0;
    for (int i = 0; i < num_seqs; ++i) {
      if (qsl[i + 1] == qsl[i]) continue;
      const int64_t ns = (lens[i] + chunk - 1) / chunk;
      n_items += ns * H;
      if (ns > 1) n_parts += ns * H;
    }
    if ((n_items <= kStaticItems && n_parts <= kStaticPartials) || chunk >= max_len) break;
    chunk *= 2;
  }
  if (n_items > kStaticItems || n_parts > kStaticPartials) return PKV_ERR_WORKSPACE;

  uint8_t *scratch = nullptr;
  if (scratch_address(dev, &scratch) != cudaSuccess) return PKV_ERR_CUDA;
  const int64_t rows = c->num_blocks * c->num_kv_heads * bs;
  CUtensorMap kmap, vmap;
  if (nvfp4) {
    const int box = std::min(std::min(bs, kNvfp4Group), kDecKeysNvfp4);
    if (!encode_nvfp4_map(&kmap, k_cache, rows / 8 * 9, box) ||
        !encode_nvfp4_map(&vmap, v_cache, rows / 8 * 9, box))
      return PKV_ERR_CUDA;
  } else {
    const int box = std::min(bs, fp8 ? kDecKeysFp8 : kDecKeysBf16);
    if (!encode_map(&kmap, k_cache, fp8, rows, box) || !encode_map(&vmap, v_cache, fp8, rows, box))
      return PKV_ERR_CUDA;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_plan_mutex);
  int n = 0, part = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int qi = qsl[i + 1] - qsl[i];
    if (qi == 0) continue;
    const int L = lens[i];
    const int ns = static_cast<int>((L + chunk - 1) / chunk);
    for (int h = 0; h < H; ++h) {
      const int base = ns > 1 ? part : -1;
      for (int sp = 0; sp < ns; ++sp) {
        pkv_work_item &w = g_items[n++];
        w = pkv_work_item{};
        w.kind = 0;
        w.seq = i;
        w.kv_head = h;
        w.tok0 = qsl[i];
        w.row0 = 0;
        w.n_rows = qi * G;
        w.hist = L - qi;
        w.k_begin = static_cast<int32_t>(sp * chunk);
        w.k_end = static_cast<int32_t>(std::min<int64_t>(L, (sp + 1) * chunk));
        w.part = ns > 1 ? part++ : -1;
        w.pair = base;
        w.n_split = ns;
      }
    }
  }
  std::sort(g_items, g_items + n, [](const pkv_work_item &a, const pkv_work_item &b) {
    const int la = a.k_end - a.k_begin, lb = b.k_end - b.k_begin;
    if (la != lb) return la > lb;
    if (a.seq != b.seq) return a.seq < b.seq;
    if (a.kv_head != b.kv_head) return a.kv_head < b.kv_head;
    return a.k_begin < b.k_begin;
  });
  // the first range of each split pair leads the list: the merge kernel
  // takes its groups from there
  const int groups = static_cast<int>(
      std::stable_partition(g_items, g_items + n,
                            [](const pkv_work_item &w) { return w.part >= 0 && w.part == w.pair; }) -
      g_items);
  if (n == 0) return PKV_OK;
  int max_split = 1;
  for (int k = 0; k < n; ++k) max_split = std::max(max_split, int(g_items[k].n_split));
  // the error word keeps what earlier calls recorded until
  // pkv_decode_static_errors reads it; the rest is overwritten
  if (cudaMemcpyAsync(scratch + kItemsOff, g_items, sizeof(pkv_work_item) * n,
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return PKV_ERR_CUDA;

  DecodeParams p{};
  p.items = reinterpret_cast<const pkv_work_item *>(scratch + kItemsOff);
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.block_tables = block_tables;
  p.bt_stride = block_table_stride;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.lse = lse;
  p.part_o = reinterpret_cast<float *>(scratch + kPartOOff);
  p.part_lse = reinterpret_cast<float *>(scratch + kPartLseOff);
  p.err = reinterpret_cast<int32_t *>(scratch + kErrOff);
  p.hq = c->num_q_heads;
  p.hkv = H;
  p.group = G;
  p.bs = bs;
  p.rows_total = static_cast<int32_t>(nvfp4 ? rows / 8 * 9 : rows);
  p.k_pool = static_cast<const uint8_t *>(k_cache);
  p.v_pool = static_cast<const uint8_t *>(v_cache);
  p.num_blocks = c->num_blocks;
  p.scale_log2 = c->softmax_scale * 1.4426950408889634f;
  p.validate = 0;
  return launch_decode(kmap, vmap, p, n, c->kv_dtype, s) == cudaSuccess &&
                 launch_decode_merge(p, groups, max_split, s) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

extern "C" pkv_status pkv_decode_static_errors(void *stream) {
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  uint8_t *scratch = nullptr;
  if (scratch_address(dev, &scratch) != cudaSuccess) return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  if (cudaMemcpyAsync(&word, scratch + kErrOff, sizeof word, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemsetAsync(scratch + kErrOff, 0, sizeof(int32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (word & kErrTimeout) return PKV_ERR_TIMEOUT;
  return word != 0 ? PKV_ERR_DEVICE_CHECK : PKV_OK;
}
