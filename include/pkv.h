/*
 * pkv.h -- C ABI of libpkv: causal attention over a paged, prefix-cached KV
 * cache on GB300 (sm_103a).
 *
 * The operations and where they are described:
 *
 *  - pkv_write_slots: the KV append ("KV 写入") that stores this step's new
 *    K/V rows at the physical slots the scheduler assigned them.  Page "vLLM
 *    Agentic 推理｜面向 Agent 负载的推理优化", section 5.2 (每层两个 Kernel,
 *    the KV write inside K1).
 *  - pkv_attention_varlen: one step of attention for a mixed batch of
 *    incremental-prefill chunks (l_incr new tokens attending to l_hist cached
 *    tokens plus themselves) and decodes (l_incr = 1).  Page "AMPD：PD 分离遇上
 *    多轮推理，incremental prefill 到底该在哪跑", sections 1 and 3; GQA head
 *    sharing, page "vLLM Agentic 推理", section 4.3.1; split attention with a
 *    log-sum-exp combine of partial results, same page, sections 4.3.3 (step
 *    4) and 5.2 (Split Attention + Combine).
 *  - Block tables: request i owns cdiv(seq_len, block_size) blocks, listed in
 *    row i of block_tables; blocks may be shared by several requests with a
 *    common prefix.  Page "vLLM/V1 推理调度器", section 源码片段
 *    (KVCacheManager.allocate_slots and the per-request block-id record).
 *
 * Conventions shared by every call
 *  - head_dim is 128.  Query heads h = 0..Hq-1 read KV head h / G, where
 *    G = Hq / Hkv.
 *  - A KV pool is [num_blocks][Hkv][block_size][128] elements: bf16, or E4M3
 *    codes (OCP FP8, "FN" variant) with one fp32 scale per (block, KV head)
 *    in a [num_blocks][Hkv] array; an element's value is e4m3(code) * scale.
 *    E4M3 block scales must be at most 16 (values up to 7168; the kernels
 *    round values times scales to f16); validate mode checks this for every
 *    block in use and reports PKV_ERR_DEVICE_CHECK.
 *    NVFP4 pools (the compressed KV format of page "vLLM 优化
 *    DeepSeek-V4.1-Flash：智能体吞吐提升 5 倍", section Kernels) are
 *    [num_blocks][Hkv][block_size * 72] bytes: per (block, KV head), rows in
 *    groups of min(block_size, 64); a group is its rows' 64 code bytes each
 *    (OCP FP4 E2M1, element 2j in the low nibble of byte j) followed by their
 *    8 micro-scale bytes each (E4M3, one per 16 elements); with the fp32
 *    (block, KV head) scale an element's value is e2m1(code) * e4m3(micro
 *    scale) * scale.  NVFP4 block scales must be at most 16 as well
 *    (checked the same way).
 *    Logical position p of request i lives in block block_tables[i][p / bs]
 *    at row p % bs; its slot is block * bs + p % bs.
 *  - Query token t (0-based) of request i, which has q_i new tokens and
 *    seq_len L_i context tokens including them, sits at position
 *    L_i - q_i + t and sees keys 0 .. L_i - q_i + t.
 *  - Device pointers are CUDA device addresses on the handle's device; host
 *    pointers are ordinary host memory.  The caller owns every buffer and the
 *    stream; the library owns only the handle and its workspace.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Buffers must stay valid until that stream's work
 *    completes.  Neither hot call allocates memory.  pkv_attention_varlen
 *    plans on the host and uploads the plan from one of two pinned staging
 *    buffers; before refilling a buffer it waits for that buffer's upload
 *    from two calls earlier, and for nothing else on the device.
 *  - Argument errors are detected on the host before anything is enqueued and
 *    return PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED with a message in
 *    pkv_last_error().  Launch failures return PKV_ERR_CUDA.  In validate
 *    mode (PKV_FLAG_VALIDATE) the kernels also check block ids and slots on
 *    the device, skip anything out of range and record it; the record is read
 *    by pkv_check_device_errors().  No kernel ever traps.
 *  - One handle is used from one host thread at a time.
 */
#ifndef PKV_H
#define PKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_handle pkv_handle;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* a pointer, size or metadata value is wrong */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim != 128, ...) */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    PKV_ERR_OUT_OF_MEMORY = 4, /* pkv_create could not allocate its workspace */
    PKV_ERR_DEVICE_CHECK = 5,  /* validate mode found a bad block id or slot */
    PKV_ERR_TIMEOUT = 6,       /* a device-side wait gave up (never expected) */
    PKV_ERR_WORKSPACE = 7      /* the step needs more workspace than created */
} pkv_status;

typedef enum {
    PKV_KV_BF16 = 0,
    PKV_KV_FP8_E4M3 = 1,
    PKV_KV_NVFP4 = 2
} pkv_kv_dtype;

enum {
    PKV_FLAG_VALIDATE = 1u,    /* device-side checks of block ids and slots */
    PKV_FLAG_TIMING = 2u,      /* record CUDA events around every kernel */
    PKV_FLAG_SEPARATE = 4u     /* run a mixed step as separate decode and
                                  prefill launches (per-kind timing) */
};

/* Fixed shape of a KV cache and the largest step a handle serves. */
typedef struct {
    int32_t num_q_heads;       /* Hq, a multiple of num_kv_heads */
    int32_t num_kv_heads;      /* Hkv */
    int32_t head_dim;          /* must be 128 */
    int32_t block_size;        /* tokens per block: 16, 32, 64, 128 or 256 */
    int32_t kv_dtype;          /* pkv_kv_dtype */
    float softmax_scale;       /* scores are softmax_scale * q . k */
    int64_t num_blocks;        /* blocks in each pool */
    int32_t max_num_seqs;      /* largest batch (requests) per step */
    int32_t max_num_tokens;    /* largest number of query tokens per step */
    uint32_t flags;            /* PKV_FLAG_* */
    int64_t stage_tokens;      /* E4M3 / NVFP4 pools: capacity, in tokens
                                  (rounded up to whole blocks), of the
                                  staging pools for the tensor-core prefill
                                  (V for E4M3, K and V for NVFP4; see
                                  pkv_attention_varlen); 0 = none */
} pkv_config;

/*
 * Create a handle on CUDA device `device` and allocate its workspace (work
 * list, split partials, error word: a few tens of MB,
 * sized from max_num_seqs and max_num_tokens; with E4M3 / NVFP4 pools and
 * stage_tokens > 0 also the staging pools, stage_tokens * Hkv * 256
 * bytes for E4M3 (V) and stage_tokens * Hkv * 516 for NVFP4 (K, V and K's
 * block scales), rounded up to whole blocks).  *out receives the handle, or
 * NULL on failure.  Errors: PKV_ERR_INVALID_ARG (NULL pointers, bad config),
 * PKV_ERR_UNSUPPORTED (head_dim or block_size not handled), PKV_ERR_CUDA (no
 * such device), PKV_ERR_OUT_OF_MEMORY.
 */
pkv_status pkv_create(const pkv_config *config, int device, pkv_handle **out);

/*
 * KV append.  For each token t < num_tokens with slot_mapping[t] >= 0, store
 * row t of k_new and v_new (each [num_tokens][Hkv][128] bf16, device) at that
 * slot of k_cache / v_cache for every KV head.  bf16 pools receive the bits
 * unchanged.  FP8 pools receive E4M3(x / scale[block][head]): the quotient is
 * one correctly rounded fp32 division, then rounded to nearest even and
 * saturated to +-448; k_scale / v_scale ([num_blocks][Hkv] fp32, device) are
 * read, never written, and must be finite and > 0 for the blocks written.
 * NVFP4 pools receive, per 16 elements, the micro scale E4M3(amax / (6 *
 * scale)) (amax the largest |x| of the 16; fp32 product and quotient) and,
 * unless it is zero (then all codes are 0), the codes E2M1(x / (scale *
 * micro scale)) (fp32 product and quotient; nearest, ties to even,
 * saturating at +-6).
 * slot_mapping is int64 on the device; negative entries are padding.
 * Entries must be distinct.  A slot past the pool is an argument error the
 * host cannot see: in validate mode it is skipped and reported, otherwise it
 * is undefined behaviour.
 */
pkv_status pkv_write_slots(pkv_handle *h, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, int32_t num_tokens,
                           void *k_cache, void *v_cache, const float *k_scale,
                           const float *v_scale, void *stream);

/*
 * Rotary position embedding fused with the KV append: the pages' first
 * per-layer kernel applies RoPE and writes the KV in one launch (page "vLLM
 * Agentic 推理｜面向 Agent 负载的推理优化", section 5.2, K1).  For each token t:
 * q[t] (all Hq heads) is rotated in place, k_new[t] is rotated and stored at
 * slot_mapping[t] like pkv_write_slots (k_new itself is not modified), and
 * v_new[t] is stored unrotated.  Rotation of the 64 pairs of a 128-element
 * head row by the angles of position p = positions[t]:
 *   y_a = x_a cos_i - x_b sin_i,  y_b = x_b cos_i + x_a sin_i,
 * with (a, b) = (i, i + 64) when neox != 0 (rotate-half layout) or
 * (2i, 2i + 1) otherwise, cos_i = cos_sin_cache[p][i] and sin_i =
 * cos_sin_cache[p][64 + i].  Computed in fp32, rounded to bf16 (an E4M3
 * pool then quantises that bf16 value as pkv_write_slots does).
 *  q              [num_tokens][Hq][128] bf16, device, read and written;
 *  positions      [num_tokens] int64, device, each in [0, max_pos);
 *  cos_sin_cache  [max_pos][128] fp32, device, 16-byte aligned.
 * Other arguments as pkv_write_slots.  A position outside [0, max_pos) skips
 * that token (q and KV untouched) and is recorded for
 * pkv_check_device_errors (PKV_ERR_DEVICE_CHECK).
 */
pkv_status pkv_rope_write_slots(pkv_handle *h, void *q, const void *k_new,
                                const void *v_new, const int64_t *positions,
                                const float *cos_sin_cache, int64_t max_pos,
                                int32_t neox, const int64_t *slot_mapping,
                                int32_t num_tokens, void *k_cache, void *v_cache,
                                const float *k_scale, const float *v_scale,
                                void *stream);

/*
 * Attention for one step.
 *  q                [num_tokens][Hq][128] bf16, device; the tokens of request
 *                   i are rows query_start_loc[i] .. query_start_loc[i+1]-1.
 *  k_cache/v_cache  pools as above (FP8: with k_scale / v_scale, else NULL).
 *  query_start_loc  [num_seqs + 1] int32, device, and its host mirror
 *                   query_start_loc_host (identical contents): 0 = first,
 *                   non-decreasing, last = num_tokens.
 *  seq_lens         [num_seqs] int32, device, and host mirror seq_lens_host:
 *                   L_i >= q_i >= 0, including this step's new tokens.
 *  block_tables     [num_seqs][block_table_stride] int32, device; entries
 *                   0 .. cdiv(L_i, block_size) - 1 of row i must be block ids
 *                   < num_blocks; later entries are never read.
 *  out              [num_tokens][Hq][128] bf16, device (written).
 *  lse              NULL, or [num_tokens][Hq] fp32, device: natural-log
 *                   log-sum-exp of each row's scaled scores (written).
 * The work is planned on the host from the host mirrors (so they must match
 * the device copies; validate mode checks that), uploaded asynchronously and
 * executed by the kernels.  The new tokens' K/V must already be in the pools
 * (call pkv_write_slots first on the same stream).  A step that needs more
 * workspace than the handle was created for returns PKV_ERR_WORKSPACE.
 * Requests with more than 8 query rows per KV head (q_i * G > 8) run on the
 * tensor-core prefill kernel when G <= 128 (every pool format); with
 * G > 128 the decode kernel takes their rows 8 at a time (same results within
 * tolerance, at memory-bound speed).  Over E4M3 / NVFP4 pools, when the
 * contexts of the step's tensor-core prefill requests (each rounded up to
 * whole blocks) fit the handle's staging pools (stage_tokens), a staging
 * kernel (PKV_KERNEL_STAGE) first converts every block they read to bf16
 * (NVFP4 K: its exact code values, the block scale kept apart for the
 * scores; V: value times block scale, rounded once), and the prefill kernel
 * reads those with bf16 MMAs (E4M3 K stays in the pool and feeds FP8 MMAs);
 * otherwise the prefill kernel converts the codes itself.  When a step holds fewer tensor-core
 * prefill items than half the multiprocessors, their key ranges are split
 * into runs of whole 128-key tiles (boundaries at multiples of the block
 * size too, at or below each item's first query position); each range
 * writes an fp32 partial and a second kernel merges them with log-sum-exp
 * weights, as it merges the key ranges of split decode items
 * (PKV_KERNEL_MERGE).
 */
pkv_status pkv_attention_varlen(pkv_handle *h, const void *q,
                                const void *k_cache, const void *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *query_start_loc,
                                const int32_t *seq_lens,
                                const int32_t *block_tables,
                                int32_t block_table_stride,
                                const int32_t *query_start_loc_host,
                                const int32_t *seq_lens_host, int32_t num_seqs,
                                int32_t num_tokens, void *out, float *lse,
                                void *stream);

/*
 * Decode context parallelism, emulated on one GPU.  DCP deals a request's KV
 * tokens out to N ranks in runs of `interleave` tokens (run j to rank j % N);
 * each rank attends with all query heads to its own share, producing a
 * partial output and its log-sum-exp, and the partials are exchanged and
 * merged with log-sum-exp weights (page "vLLM Agentic 推理｜面向 Agent 负载的
 * 推理优化", sections 4.3.1 and 4.3.3).  Here every shard reads its share
 * from the one shared pool.
 *
 * pkv_attention_partial: shard `shard` (0 <= shard < num_shards) of one step,
 * decode rows only (q_i * G <= 8; a request with more rows returns
 * PKV_ERR_UNSUPPORTED).  Arguments as for pkv_attention_varlen, except:
 *  interleave  tokens per run, >= 1 (the pages' default is 1).  A multiple
 *              of the decode stage (16 keys for bf16 pools, 32 for E4M3, 64
 *              for NVFP4) lets the shard read only its own keys; any other
 *              value makes the shard walk the request's whole context and
 *              mask the keys it does not own (same result, the pool read
 *              once per shard: on real ranks each rank's pool holds only
 *              its own tokens and the plain decode reads them);
 *  out         [num_tokens][Hq][128] fp32, device: the shard's softmax-
 *              normalised partial output (0 where the shard owns no visible
 *              key);
 *  lse         [num_tokens][Hq] fp32, device: its natural-log log-sum-exp
 *              (-inf where the shard owns no visible key).  Required.
 * Not capturable in a CUDA graph (PKV_ERR_UNSUPPORTED while capturing).
 */
pkv_status pkv_attention_partial(pkv_handle *h, const void *q,
                                 const void *k_cache, const void *v_cache,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *query_start_loc,
                                 const int32_t *seq_lens,
                                 const int32_t *block_tables,
                                 int32_t block_table_stride,
                                 const int32_t *query_start_loc_host,
                                 const int32_t *seq_lens_host, int32_t num_seqs,
                                 int32_t num_tokens, int32_t shard,
                                 int32_t num_shards, int32_t interleave,
                                 float *out, float *lse, void *stream);

/*
 * The merge step: for each of num_rows rows, lse = ln sum_s exp(lse_s) and
 * out = sum_s exp(lse_s - lse) * o_s over the num_parts partials (parts with
 * lse_s = -inf contribute nothing; a row with no part gets 0 and -inf).
 *  parts_o    [num_parts][num_rows][128] fp32, device, 16-byte aligned;
 *  parts_lse  [num_parts][num_rows] fp32, device (natural log);
 *  out        [num_rows][128] bf16, device (written);
 *  lse        NULL or [num_rows] fp32, device (written).
 * With the rows of pkv_attention_partial (num_rows = num_tokens * Hq) this
 * is the exchange-then-merge of DCP; the partials may come from any source.
 */
pkv_status pkv_lse_merge(pkv_handle *h, const float *parts_o,
                         const float *parts_lse, int32_t num_parts,
                         int64_t num_rows, void *out, float *lse, void *stream);

/*
 * Prepare a step for CUDA-graph capture.  Small steps are dominated by
 * launch overhead unless captured in a CUDA graph (page "vLLM 优化
 * DeepSeek-V4.1-Flash：智能体吞吐提升 5 倍", section "裁剪层的 CUDA graphs");
 * the calls of this library can be captured the same way.  This call plans the
 * step from the host mirrors (same meaning as in pkv_attention_varlen) and
 * copies the work list into a device buffer kept for captured steps; it is
 * synchronous and may allocate that buffer (once per handle), so call it
 * before cudaStreamBeginCapture.  While `stream` is capturing,
 * pkv_attention_varlen enqueues kernels only, reading this prepared work
 * list: its host mirrors must equal the prepared ones (else
 * PKV_ERR_INVALID_ARG and nothing is enqueued), and the graph replays that
 * plan as long as the handle lives and no later pkv_graph_prepare replaces
 * it.  pkv_write_slots needs no preparation.  Timing (PKV_FLAG_TIMING)
 * records nothing for captured calls.
 */
pkv_status pkv_graph_prepare(pkv_handle *h, const int32_t *query_start_loc_host,
                             const int32_t *seq_lens_host, int32_t num_seqs,
                             int32_t num_tokens);

/*
 * Wait for the handle's device (cudaDeviceSynchronize) and read the device
 * error word, clearing it.  Returns PKV_OK, PKV_ERR_DEVICE_CHECK (validate
 * mode found a bad block id, slot or host-mirror mismatch),
 * PKV_ERR_TIMEOUT, or PKV_ERR_CUDA if the device reported an error.
 */
pkv_status pkv_check_device_errors(pkv_handle *h);

/*
 * Self-test of failure detection.  Every wait inside the kernels (on a copy
 * or an MMA completing) gives up after 1 s, records PKV_ERR_TIMEOUT in the
 * handle's error word and lets the kernel wind down, so a lost completion
 * is reported instead of hanging the GPU.  This call exercises that path
 * without breaking anything: it launches one CTA on `stream` that waits,
 * through the same bounded-wait code, on a barrier nothing arrives at and no
 * copy or MMA completes, with a limit of limit_ns nanoseconds
 * (1 .. 1000000000).  The wait runs out and the timeout is recorded, so the
 * next pkv_check_device_errors returns PKV_ERR_TIMEOUT (and clears the
 * word); the handle stays usable.  Errors: PKV_ERR_INVALID_ARG (limit_ns out
 * of range), PKV_ERR_CUDA.
 */
pkv_status pkv_wait_selftest(pkv_handle *h, uint64_t limit_ns, void *stream);

/* Static description of a status code; never NULL. */
const char *pkv_status_string(pkv_status status);

/* Message of the last failed call on this handle ("" if none); never NULL.
 * With h == NULL, the message of the last failed pkv_create. */
const char *pkv_last_error(const pkv_handle *h);

/* Free the workspace and the handle (waits for the device first).  NULL is
 * accepted and ignored. */
pkv_status pkv_destroy(pkv_handle *h);

/* ---- planning and diagnostics -------------------------------------------- */

/* One unit of kernel work: a (request, KV head) pair restricted to a query
 * row range and a key range.  Rows r = t * G + g enumerate (query token t,
 * head g of the group). */
typedef struct {
    int32_t kind;        /* 0 = decode kernel (decode rows, or a chunk of
                            8 prefill rows when G > 128),
                            1 = tensor-core prefill tile */
    int32_t seq;         /* request index */
    int32_t kv_head;
    int32_t tok0;        /* index of the request's first query token in q */
    int32_t row0;        /* first row of this item */
    int32_t n_rows;      /* rows in this item */
    int32_t hist;        /* l_hist = L - q of the request */
    int32_t k_begin;     /* first key position */
    int32_t k_end;       /* one past the last key position */
    int32_t part;        /* partial-result slot, or -1: writes the output.
                            A split prefill item's partial takes 32
                            consecutive slots (256 rows of 8) */
    int32_t pair;        /* slot of the first range of the split, or -1 */
    int32_t n_split;     /* key ranges of this (request, KV head, rows) */
} pkv_work_item;

/*
 * Plan a step on the host without a GPU: the work items the kernels of
 * pkv_attention_varlen would run for these lengths on a device with
 * `num_sms` multiprocessors.  Items of each kind are in launch order
 * (longest first; the prefill items of one (request, KV head) adjacent,
 * after the first ranges of split items, which lead the decode and the
 * prefill items).  *num_items receives the count; if it exceeds
 * max_items only the first max_items are stored.  *num_partials receives the
 * split partial slots used.  Errors: PKV_ERR_INVALID_ARG for inconsistent
 * metadata (same checks as pkv_attention_varlen).
 */
pkv_status pkv_plan(const pkv_config *config, const int32_t *query_start_loc_host,
                    const int32_t *seq_lens_host, int32_t num_seqs,
                    int32_t num_tokens, int32_t num_sms,
                    pkv_work_item *items, int32_t max_items,
                    int32_t *num_items, int32_t *num_partials);

/* Kernel kinds reported by pkv_timing_read.  A step holding both decodes
 * and prefill chunks (bf16 pools, query groups of at most 128) runs as
 * one PKV_KERNEL_MIXED launch; otherwise decode and prefill launch apart.
 * PKV_KERNEL_MERGE: the merge of split key ranges (decode pairs and prefill
 * row tiles), one window after the attention launches of a step that split
 * any ranges.  PKV_KERNEL_STAGE: the staging of E4M3 V or NVFP4 K and V
 * before the tensor-core prefill. */
enum {
    PKV_KERNEL_APPEND = 0,
    PKV_KERNEL_DECODE = 1,
    PKV_KERNEL_PREFILL = 2,
    PKV_KERNEL_MIXED = 3,
    PKV_KERNEL_MERGE = 4,
    PKV_KERNEL_STAGE = 5,
    PKV_KERNEL_KINDS = 6
};

/*
 * With PKV_FLAG_TIMING, every kernel launch of the handle is bracketed by CUDA
 * events on its stream (the first 4096 launches per kind since the last
 * reset are kept).
 * pkv_timing_read waits for those events and returns, per kind, the number
 * of launches recorded and their summed device time in milliseconds;
 * pkv_timing_reset forgets them.  Both take a NULL-safe handle; reading
 * without the flag returns counts of 0.
 */
pkv_status pkv_timing_reset(pkv_handle *h);
pkv_status pkv_timing_read(pkv_handle *h, int32_t kind, int32_t *launches,
                           double *total_ms);

/* ---- decode without allocation ----------------------------------------------
 *
 * The pages describe nothing like this entry point; it exists for callers
 * that cannot allocate GPU memory: an engine whose memory pool already owns
 * all of HBM (the KV cache reservation), code that must not allocate after
 * start-up, or code that cannot hold a handle (pkv_create allocates its
 * workspace).
 *
 * pkv_decode_static runs the split-KV decode of pkv_attention_varlen for a
 * batch in which every request has q_i * G <= 8 query rows, on the CURRENT
 * CUDA device, without a handle.  The caller passes the inputs and outputs
 * exactly as for pkv_attention_varlen (same layouts and meaning, minus the
 * device copies of query_start_loc and seq_lens, which are not read) and a
 * config describing the pools (max_num_seqs, max_num_tokens and flags are
 * ignored).  Nothing is allocated: the work list, split partials and the
 * error word live in one fixed array of about 4.3 MB compiled into the library,
 * which every GPU that loads the library keeps until the process exits.
 * Limits: at most 2048 work items and 1024 split partials per call (the split
 * size grows to fit; a batch with more than 2048 (request, KV head) pairs is
 * rejected with PKV_ERR_WORKSPACE).
 *  - Set-up: the first call on a device looks up the array's device address
 *    (which loads the library's device code there and, with CUDA's lazy
 *    module loading, is when the array gets its memory), sets the kernels'
 *    shared-memory limits and clears the error word, synchronously.  A call
 *    with num_seqs = 0 and num_tokens = 0 does only that: make it at
 *    start-up, before the caller reserves the rest of device memory and
 *    before any stream capture.
 *  - Every call shares the array and leaves its contents behind; each call
 *    overwrites the work list and partials it uses.  A call runs the decode
 *    kernel and, when it split any key range, the merge kernel.  Calls whose
 *    GPU work overlaps (on different streams, or from different threads)
 *    race on it: serialise them.
 *  - The kernels record a block-table entry outside the pool (its keys read
 *    as zeros) and a device-side wait that gave up in an error word inside
 *    the array; it accumulates over calls until pkv_decode_static_errors
 *    reads and clears it.
 *  - Returns PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED (prefill rows,
 *    head_dim or block_size not handled), PKV_ERR_WORKSPACE or PKV_ERR_CUDA.
 *    It does not update pkv_last_error().
 */
pkv_status pkv_decode_static(const pkv_config *config, const void *q,
                             const void *k_cache, const void *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int32_t *block_tables,
                             int32_t block_table_stride,
                             const int32_t *query_start_loc_host,
                             const int32_t *seq_lens_host, int32_t num_seqs,
                             int32_t num_tokens, void *out, float *lse,
                             void *stream);

/*
 * Read and clear the error word of pkv_decode_static on the current device,
 * after the work already enqueued on `stream` (a cudaStream_t; NULL = legacy
 * default stream) has finished: waits for that stream, copies the word into
 * host memory of the library and clears it, allocating nothing.  Returns
 * PKV_OK, PKV_ERR_DEVICE_CHECK (a block-table entry in use was outside the
 * pool), PKV_ERR_TIMEOUT (a device-side wait gave up) or PKV_ERR_CUDA.
 * Like every pkv_decode_static call, it must not overlap another one's GPU
 * work.  The pages describe nothing like it (see pkv_decode_static).
 */
pkv_status pkv_decode_static_errors(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
