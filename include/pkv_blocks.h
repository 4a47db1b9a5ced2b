/*
 * pkv_blocks.h -- host-side KV block pool with prefix caching, the producer
 * of the block tables and slot mappings that pkv.h's kernels consume.
 *
 * What it implements, and where the pages describe it:
 *  - KV is stored in blocks of block_size tokens; a request holding n
 *    tokens (plus lookahead) needs cdiv(n, block_size) blocks
 *    (page "vLLM/V1 推理调度器", section 源码片段, KVCacheManager.allocate_slots).
 *  - Prefix caching: every full block is identified by a hash of its
 *    tokens chained with the hash of the block before it, so a block hit
 *    means the whole prefix up to it matches; hit blocks are reused instead
 *    of recomputed (page "vLLM Agentic 推理｜面向 Agent 负载的推理优化", section
 *    4.1).
 *  - Reference counts: a block shared by several requests is freed only
 *    when the last of them releases it; a cached block whose count drops to
 *    0 stays cached as an eviction candidate until its memory is needed.
 *    The capacity check does not count hit blocks that are themselves
 *    eviction candidates as free (same section 源码片段 of "vLLM/V1 推理调度器").
 *
 * All calls are host-only, synchronous and single-threaded per pool.
 * Statuses are pkv_status values from pkv.h (PKV_OK = 0,
 * PKV_ERR_INVALID_ARG = 1); a pool that cannot hold a request is not an
 * error: the call reports *ok = 0 and changes nothing.
 */
#ifndef PKV_BLOCKS_H
#define PKV_BLOCKS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_blocks pkv_blocks;   /* opaque, owned by the library */

/* A pool of num_blocks blocks (ids 0 .. num_blocks-1) of block_size tokens;
 * every block starts free.  *out receives the pool.  Errors: num_blocks < 1,
 * block_size < 1, out == NULL -> 1 (PKV_ERR_INVALID_ARG). */
int pkv_blocks_create(int64_t num_blocks, int32_t block_size, pkv_blocks **out);

/* Frees the pool (NULL is accepted). */
int pkv_blocks_destroy(pkv_blocks *b);

/* Longest cached prefix of a token sequence, without taking references:
 * *hit_tokens = block_size * (number of leading full blocks of tokens[0 ..
 * num_tokens) whose chained hash and tokens match a cached block), at most
 * num_tokens - 1 rounded down to whole blocks (the last known token is
 * always computed, so a request that is all hits still produces output). */
int pkv_blocks_lookup(pkv_blocks *b, const int32_t *tokens, int64_t num_tokens,
                      int64_t *hit_tokens);

/* Schedules num_new_tokens more tokens of request `req` (any caller-chosen
 * id).  tokens[0 .. num_tokens) are the request's known tokens.  For a
 * request the pool does not hold yet, its cached prefix (as
 * pkv_blocks_lookup) is reused first.  Then the request holds
 * cdiv(num_computed + num_new_tokens + num_lookahead, block_size) blocks,
 * new ones taken from the free blocks, least recently released first
 * (a cached one loses its cache entry).  On success *ok = 1, the request's
 * block table is written to table[0 .. *n_blocks) (table_cap entries
 * available) and *num_computed is the number of its tokens already in the
 * cache (hit prefix or earlier steps).  If the free blocks, not counting
 * hit blocks that are eviction candidates themselves, cannot cover the new
 * blocks: *ok = 0 and nothing changes. */
int pkv_blocks_allocate(pkv_blocks *b, int64_t req, const int32_t *tokens,
                        int64_t num_tokens, int64_t num_new_tokens,
                        int32_t num_lookahead, int32_t *table, int64_t table_cap,
                        int64_t *n_blocks, int64_t *num_computed, int32_t *ok);

/* Records that the first num_computed tokens of `req` are now in the KV
 * cache (their K/V were written); its full blocks among them enter the
 * prefix cache (a block whose content is already cached elsewhere stays
 * private).  num_computed may not exceed the request's allocated tokens or
 * num_tokens. */
int pkv_blocks_commit(pkv_blocks *b, int64_t req, const int32_t *tokens,
                      int64_t num_tokens, int64_t num_computed);

/* Releases the request's references (last block first, so a request's tail
 * blocks are evicted before its head) and forgets the request. */
int pkv_blocks_free(pkv_blocks *b, int64_t req);

/* Slots of positions pos0 .. pos0 + n - 1 of `req`:
 * slots[i] = table[p / block_size] * block_size + p % block_size. */
int pkv_blocks_slots(pkv_blocks *b, int64_t req, int64_t pos0, int64_t n,
                     int64_t *slots);

/* *free_blocks: blocks with no reference (eviction candidates included);
 * *cached_blocks: blocks with a cache entry; *evictable: cached blocks with
 * no reference.  Any pointer may be NULL. */
int pkv_blocks_stats(pkv_blocks *b, int64_t *free_blocks, int64_t *cached_blocks,
                     int64_t *evictable);

/* Reference count of one block (-1 if the id is out of range). */
int32_t pkv_blocks_ref_count(pkv_blocks *b, int32_t block);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCKS_H */
