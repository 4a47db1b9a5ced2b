// Host-side KV block pool with prefix caching (see include/pkv_blocks.h).
//
// Free blocks (reference count 0, cached or not) sit in one intrusive
// doubly linked queue: released blocks go to the back, new allocations take
// from the front, so the least recently released block is reused first.
// Cached blocks are found through a hash map from their chained hash; the
// block also keeps its tokens, and a hit requires the tokens to match, so a
// hash collision can never hand out the wrong KV.
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "../../include/pkv_blocks.h"

namespace {

constexpr int kOk = 0, kBadArg = 1;

// Chained block hash: FNV-1a over the parent hash and the block's tokens,
// finished with the splitmix64 avalanche.
uint64_t block_hash(uint64_t parent, const int32_t *tok, int32_t n) {
  uint64_t h = 0xcbf29ce484222325ull;
  auto mix = [&](uint64_t x) {
    for (int i = 0; i < 8; ++i) {
      h ^= (x >> (8 * i)) & 0xffu;
      h *= 0x100000001b3ull;
    }
  };
  mix(parent);
  for (int32_t i = 0; i < n; ++i) mix(static_cast<uint32_t>(tok[i]));
  h ^= h >> 30;
  h *= 0xbf58476d1ce4e5b9ull;
  h ^= h >> 27;
  h *= 0x94d049bb133111ebull;
  h ^= h >> 31;
  return h;
}

struct Block {
  int32_t ref = 0;
  bool cached = false;
  uint64_t hash = 0;
  std::vector<int32_t> tokens;    // content of a cached block
  int32_t prev = -1, next = -1;   // free queue links
  bool queued = false;
};

struct Request {
  std::vector<int32_t> table;
  int64_t num_computed = 0;
  int64_t num_committed_blocks = 0;   // leading blocks already offered to the cache
  uint64_t last_hash = 0;             // chained hash of block num_committed_blocks - 1
};

}  // namespace

struct pkv_blocks {
  int32_t bs = 0;
  std::vector<Block> blocks;
  int32_t head = -1, tail = -1;
  int64_t n_free = 0;
  int64_t n_cached = 0;
  std::unordered_map<uint64_t, int32_t> cache;
  std::unordered_map<int64_t, Request> reqs;

  void push_back(int32_t id) {
    Block &b = blocks[id];
    b.prev = tail;
    b.next = -1;
    if (tail >= 0) blocks[tail].next = id; else head = id;
    tail = id;
    b.queued = true;
    ++n_free;
  }
  void unlink(int32_t id) {
    Block &b = blocks[id];
    if (b.prev >= 0) blocks[b.prev].next = b.next; else head = b.next;
    if (b.next >= 0) blocks[b.next].prev = b.prev; else tail = b.prev;
    b.prev = b.next = -1;
    b.queued = false;
    --n_free;
  }
  void uncache(int32_t id) {
    Block &b = blocks[id];
    if (!b.cached) return;
    cache.erase(b.hash);
    b.cached = false;
    b.tokens.clear();
    --n_cached;
  }
  // Leading full blocks of tokens that are cached, capped so that at least
  // one token is left to compute.
  std::vector<int32_t> hits(const int32_t *tok, int64_t n) const {
    std::vector<int32_t> out;
    const int64_t max_blocks = n > 0 ? (n - 1) / bs : 0;
    uint64_t h = 0;
    for (int64_t i = 0; i < max_blocks; ++i) {
      h = block_hash(h, tok + i * bs, bs);
      auto it = cache.find(h);
      if (it == cache.end()) break;
      const Block &b = blocks[it->second];
      if (std::memcmp(b.tokens.data(), tok + i * bs, sizeof(int32_t) * bs) != 0) break;
      out.push_back(it->second);
    }
    return out;
  }
};

extern "C" {

int pkv_blocks_create(int64_t num_blocks, int32_t block_size, pkv_blocks **out) {
  if (out == nullptr || num_blocks < 1 || block_size < 1 || num_blocks > INT32_MAX) return kBadArg;
  pkv_blocks *b = new pkv_blocks();
  b->bs = block_size;
  b->blocks.resize(static_cast<size_t>(num_blocks));
  for (int64_t i = 0; i < num_blocks; ++i) b->push_back(static_cast<int32_t>(i));
  *out = b;
  return kOk;
}

int pkv_blocks_destroy(pkv_blocks *b) {
  delete b;
  return kOk;
}

int pkv_blocks_lookup(pkv_blocks *b, const int32_t *tokens, int64_t num_tokens,
                      int64_t *hit_tokens) {
  if (b == nullptr || hit_tokens == nullptr || num_tokens < 0 || (num_tokens > 0 && !tokens))
    return kBadArg;
  *hit_tokens = static_cast<int64_t>(b->hits(tokens, num_tokens).size()) * b->bs;
  return kOk;
}

int pkv_blocks_allocate(pkv_blocks *b, int64_t req, const int32_t *tokens,
                        int64_t num_tokens, int64_t num_new_tokens,
                        int32_t num_lookahead, int32_t *table, int64_t table_cap,
                        int64_t *n_blocks, int64_t *num_computed, int32_t *ok) {
  if (b == nullptr || ok == nullptr || n_blocks == nullptr || num_computed == nullptr ||
      num_tokens < 0 || num_new_tokens < 0 || num_lookahead < 0 ||
      (num_tokens > 0 && tokens == nullptr))
    return kBadArg;
  *ok = 0;
  auto found = b->reqs.find(req);
  const bool fresh = found == b->reqs.end();
  std::vector<int32_t> hit;
  int64_t computed = 0, held = 0;
  if (fresh) {
    hit = b->hits(tokens, num_tokens);
    computed = static_cast<int64_t>(hit.size()) * b->bs;
  } else {
    computed = found->second.num_computed;
    held = static_cast<int64_t>(found->second.table.size());
  }
  if (computed + num_new_tokens > num_tokens) return kBadArg;   // tokens must be known
  const int64_t need = computed + num_new_tokens + num_lookahead;
  const int64_t required = (need + b->bs - 1) / b->bs;
  const int64_t n_new = required - held - static_cast<int64_t>(hit.size());
  int64_t hit_evictable = 0;
  for (int32_t id : hit) hit_evictable += b->blocks[id].ref == 0 ? 1 : 0;
  if (n_new > b->n_free - hit_evictable) return kOk;   // does not fit: *ok = 0
  const int64_t total = held + static_cast<int64_t>(hit.size()) + (n_new > 0 ? n_new : 0);
  if (table != nullptr && table_cap < total) return kBadArg;
  Request &r = b->reqs[req];   // creates a fresh request
  for (int32_t id : hit) {
    Block &blk = b->blocks[id];
    if (blk.ref == 0) b->unlink(id);
    ++blk.ref;
    r.table.push_back(id);
  }
  if (fresh) {
    r.num_computed = computed;
    r.num_committed_blocks = static_cast<int64_t>(hit.size());
    uint64_t h = 0;
    for (size_t i = 0; i < hit.size(); ++i) h = block_hash(h, tokens + i * b->bs, b->bs);
    r.last_hash = h;
  }
  for (int64_t i = 0; i < n_new; ++i) {
    const int32_t id = b->head;
    b->unlink(id);
    b->uncache(id);
    b->blocks[id].ref = 1;
    r.table.push_back(id);
  }
  *n_blocks = static_cast<int64_t>(r.table.size());
  *num_computed = r.num_computed;
  if (table != nullptr) std::memcpy(table, r.table.data(), sizeof(int32_t) * r.table.size());
  *ok = 1;
  return kOk;
}

int pkv_blocks_commit(pkv_blocks *b, int64_t req, const int32_t *tokens, int64_t num_tokens,
                      int64_t num_computed) {
  if (b == nullptr || num_computed < 0 || num_computed > num_tokens ||
      (num_tokens > 0 && tokens == nullptr))
    return kBadArg;
  auto found = b->reqs.find(req);
  if (found == b->reqs.end()) return kBadArg;
  Request &r = found->second;
  if (num_computed > static_cast<int64_t>(r.table.size()) * b->bs) return kBadArg;
  if (num_computed > r.num_computed) r.num_computed = num_computed;
  const int64_t full = r.num_computed / b->bs;
  for (int64_t i = r.num_committed_blocks; i < full; ++i) {
    const int32_t *tk = tokens + i * b->bs;
    r.last_hash = block_hash(r.last_hash, tk, b->bs);
    const int32_t id = r.table[static_cast<size_t>(i)];
    Block &blk = b->blocks[id];
    if (!blk.cached && b->cache.find(r.last_hash) == b->cache.end()) {
      blk.cached = true;
      blk.hash = r.last_hash;
      blk.tokens.assign(tk, tk + b->bs);
      b->cache.emplace(r.last_hash, id);
      ++b->n_cached;
    }
  }
  if (full > r.num_committed_blocks) r.num_committed_blocks = full;
  return kOk;
}

int pkv_blocks_free(pkv_blocks *b, int64_t req) {
  if (b == nullptr) return kBadArg;
  auto found = b->reqs.find(req);
  if (found == b->reqs.end()) return kBadArg;
  const std::vector<int32_t> &t = found->second.table;
  for (auto it = t.rbegin(); it != t.rend(); ++it) {
    Block &blk = b->blocks[*it];
    if (--blk.ref == 0) b->push_back(*it);
  }
  b->reqs.erase(found);
  return kOk;
}

int pkv_blocks_slots(pkv_blocks *b, int64_t req, int64_t pos0, int64_t n, int64_t *slots) {
  if (b == nullptr || pos0 < 0 || n < 0 || (n > 0 && slots == nullptr)) return kBadArg;
  auto found = b->reqs.find(req);
  if (found == b->reqs.end()) return kBadArg;
  const std::vector<int32_t> &t = found->second.table;
  if ((pos0 + n + b->bs - 1) / b->bs > static_cast<int64_t>(t.size()) && n > 0) return kBadArg;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t p = pos0 + i;
    slots[i] = static_cast<int64_t>(t[static_cast<size_t>(p / b->bs)]) * b->bs + p % b->bs;
  }
  return kOk;
}

int pkv_blocks_stats(pkv_blocks *b, int64_t *free_blocks, int64_t *cached_blocks,
                     int64_t *evictable) {
  if (b == nullptr) return kBadArg;
  if (free_blocks) *free_blocks = b->n_free;
  if (cached_blocks) *cached_blocks = b->n_cached;
  if (evictable) {
    int64_t e = 0;
    for (int32_t id = b->head; id >= 0; id = b->blocks[id].next) e += b->blocks[id].cached ? 1 : 0;
    *evictable = e;
  }
  return kOk;
}

int32_t pkv_blocks_ref_count(pkv_blocks *b, int32_t block) {
  if (b == nullptr || block < 0 || block >= static_cast<int32_t>(b->blocks.size())) return -1;
  return b->blocks[block].ref;
}

}  // extern "C"
