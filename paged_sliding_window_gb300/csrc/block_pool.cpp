// block_pool.cpp -- host-side page allocator with prefix caching.
//
// The abstractions of "Gemma 4 model architecture analysis" (vLLM-Kunlun),
// section 6.2: a physical page is a KVCacheBlock {block_id, ref_cnt,
// block_hash}; the BlockPool keeps the pages nobody references in a free
// queue in least-recently-used order (a doubly linked list); a block table
// row lists a sequence's pages. Section 6.6, prefix caching: a full page is
// known by the hash of its tokens chained with its predecessor's hash, and a
// request whose prefix matches cached pages shares those physical pages
// (get_cached_block: a hit touches the page and raises its reference count,
// a miss allocates a new one).
//
// Design: an array of blocks indexed by id, the free queue threaded through
// the blocks themselves (prev/next ids, O(1) removal from the middle when a
// freed page is hit again), and a hash map from chained hash to block id.
// Freed pages keep their hash until the queue hands them out again, which is
// what lets a later request hit them. All operations take the pool's mutex.
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/psw.h"

struct psw_block_pool {
  struct Block {
    int32_t ref_cnt = 0;
    bool hashed = false;
    uint64_t hash = 0;
    int32_t prev = -1, next = -1;  // free-queue links, -1: none
    bool in_queue = false;
  };
  std::vector<Block> blocks;
  int32_t head = -1, tail = -1;  // free queue: head = least recently freed
  int64_t n_free = 0;
  bool prefix_cache = true;
  std::unordered_map<uint64_t, int32_t> cached;
  std::mutex mu;

  void push_tail(int32_t id) {
    Block& b = blocks[id];
    b.prev = tail;
    b.next = -1;
    if (tail >= 0) blocks[tail].next = id; else head = id;
    tail = id;
    b.in_queue = true;
    ++n_free;
  }
  void unlink(int32_t id) {
    Block& b = blocks[id];
    if (b.prev >= 0) blocks[b.prev].next = b.next; else head = b.next;
    if (b.next >= 0) blocks[b.next].prev = b.prev; else tail = b.prev;
    b.prev = b.next = -1;
    b.in_queue = false;
    --n_free;
  }
  void drop_hash(int32_t id) {
    Block& b = blocks[id];
    if (!b.hashed) return;
    auto it = cached.find(b.hash);
    if (it != cached.end() && it->second == id) cached.erase(it);
    b.hashed = false;
  }
  bool valid(int32_t id) const { return id >= 0 && static_cast<size_t>(id) < blocks.size(); }
};

namespace {

// FNV-1a, 64 bits (offset basis 14695981039346656037, prime 1099511628211),
// over little-endian bytes.
uint64_t fnv1a(uint64_t h, const void* data, size_t n) {
  const unsigned char* p = static_cast<const unsigned char*>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

void le_bytes(uint64_t v, unsigned char* out, int n) {
  for (int i = 0; i < n; ++i) out[i] = static_cast<unsigned char>(v >> (8 * i));
}

}  // namespace

extern "C" {

uint64_t psw_block_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
  uint64_t h = 14695981039346656037ull;
  unsigned char b[8];
  le_bytes(parent, b, 8);
  h = fnv1a(h, b, 8);
  for (int32_t i = 0; i < n; ++i) {
    le_bytes(static_cast<uint32_t>(tokens[i]), b, 4);
    h = fnv1a(h, b, 4);
  }
  return h;
}

int psw_block_pool_create(int64_t num_blocks, int32_t enable_prefix_cache,
                          psw_block_pool_t** out) {
  if (out == nullptr) return PSW_ENULL;
  *out = nullptr;
  if (num_blocks <= 0 || num_blocks > INT32_MAX) return PSW_ECAPACITY;
  psw_block_pool* p = new (std::nothrow) psw_block_pool();
  if (p == nullptr) return PSW_ENOBLOCKS;
  try {
    p->blocks.resize(static_cast<size_t>(num_blocks));
  } catch (...) {
    delete p;
    return PSW_ENOBLOCKS;
  }
  p->prefix_cache = enable_prefix_cache != 0;
  for (int32_t i = 0; i < static_cast<int32_t>(num_blocks); ++i) p->push_tail(i);
  *out = p;
  return PSW_OK;
}

void psw_block_pool_destroy(psw_block_pool_t* pool) { delete pool; }

int64_t psw_block_pool_num_free(psw_block_pool_t* pool) {
  if (pool == nullptr) return PSW_ENULL;
  std::lock_guard<std::mutex> lock(pool->mu);
  return pool->n_free;
}

int psw_block_pool_allocate(psw_block_pool_t* pool, int32_t n, int32_t* ids_out) {
  if (pool == nullptr || (n > 0 && ids_out == nullptr)) return PSW_ENULL;
  if (n < 0) return PSW_EINVAL_NSEQS;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (n > pool->n_free) return PSW_ENOBLOCKS;  // all or nothing
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = pool->head;
    pool->unlink(id);
    pool->drop_hash(id);  // the page is reused: its old contents are gone
    pool->blocks[id].ref_cnt = 1;
    ids_out[i] = id;
  }
  return PSW_OK;
}

int psw_block_pool_free(psw_block_pool_t* pool, const int32_t* ids, int32_t n) {
  if (pool == nullptr || (n > 0 && ids == nullptr)) return PSW_ENULL;
  if (n < 0) return PSW_EINVAL_NSEQS;
  std::lock_guard<std::mutex> lock(pool->mu);
  // check first (an id may appear several times): nothing changes on an error
  std::unordered_map<int32_t, int32_t> uses;
  for (int32_t i = 0; i < n; ++i) {
    if (!pool->valid(ids[i])) return PSW_EBLOCK;
    if (++uses[ids[i]] > pool->blocks[ids[i]].ref_cnt) return PSW_EBLOCK;
  }
  for (int32_t i = 0; i < n; ++i) {
    psw_block_pool::Block& b = pool->blocks[ids[i]];
    if (--b.ref_cnt == 0) pool->push_tail(ids[i]);
  }
  return PSW_OK;
}

int psw_block_pool_get_cached(psw_block_pool_t* pool, uint64_t hash, int32_t* id_out) {
  if (pool == nullptr || id_out == nullptr) return PSW_ENULL;
  std::lock_guard<std::mutex> lock(pool->mu);
  *id_out = -1;
  if (!pool->prefix_cache) return PSW_OK;
  auto it = pool->cached.find(hash);
  if (it == pool->cached.end()) return PSW_OK;
  const int32_t id = it->second;
  psw_block_pool::Block& b = pool->blocks[id];
  if (b.in_queue) pool->unlink(id);  // touch: no longer free
  ++b.ref_cnt;
  *id_out = id;
  return PSW_OK;
}

int psw_block_pool_cache(psw_block_pool_t* pool, int32_t id, uint64_t hash) {
  if (pool == nullptr) return PSW_ENULL;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (!pool->valid(id) || pool->blocks[id].ref_cnt <= 0) return PSW_EBLOCK;
  if (!pool->prefix_cache) return PSW_OK;
  if (pool->cached.count(hash)) return PSW_OK;  // first page with this content stays
  pool->drop_hash(id);
  psw_block_pool::Block& b = pool->blocks[id];
  b.hashed = true;
  b.hash = hash;
  pool->cached.emplace(hash, id);
  return PSW_OK;
}

int psw_block_pool_ref_count(psw_block_pool_t* pool, int32_t id, int32_t* out) {
  if (pool == nullptr || out == nullptr) return PSW_ENULL;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (!pool->valid(id)) return PSW_EBLOCK;
  *out = pool->blocks[id].ref_cnt;
  return PSW_OK;
}

int psw_block_pool_admit(psw_block_pool_t* pool, const int32_t* tokens, int32_t n_tokens,
                         int32_t* table_row, int32_t max_blocks, int32_t* n_cached_tokens) {
  if (pool == nullptr || table_row == nullptr || n_cached_tokens == nullptr ||
      (n_tokens > 0 && tokens == nullptr))
    return PSW_ENULL;
  if (n_tokens < 0) return PSW_EINVAL_NSEQS;
  constexpr int32_t bs = 16;
  const int32_t need = (n_tokens + bs - 1) / bs;
  if (need > max_blocks) return PSW_ECAPACITY;
  // Full pages of the prompt, except the page holding its last token: that
  // token's query must run, so its page is always computed.
  const int32_t full = n_tokens > 0 ? (n_tokens - 1) / bs : 0;
  int32_t hits = 0;
  uint64_t parent = 0;
  for (int32_t i = 0; i < full; ++i) {
    const uint64_t h = psw_block_hash(parent, tokens + static_cast<int64_t>(i) * bs, bs);
    int32_t id = -1;
    const int rc = psw_block_pool_get_cached(pool, h, &id);
    if (rc != PSW_OK) return rc;
    if (id < 0) break;
    table_row[hits++] = id;
    parent = h;
  }
  const int rc = psw_block_pool_allocate(pool, need - hits, table_row + hits);
  if (rc != PSW_OK) {  // undo the hits: nothing is held on an error
    psw_block_pool_free(pool, table_row, hits);
    return rc;
  }
  for (int32_t i = need; i < max_blocks; ++i) table_row[i] = -1;
  *n_cached_tokens = hits * bs;
  return PSW_OK;
}

int psw_block_pool_commit(psw_block_pool_t* pool, const int32_t* tokens, int32_t n_tokens,
                          const int32_t* table_row) {
  if (pool == nullptr || table_row == nullptr || (n_tokens > 0 && tokens == nullptr))
    return PSW_ENULL;
  if (n_tokens < 0) return PSW_EINVAL_NSEQS;
  constexpr int32_t bs = 16;
  uint64_t parent = 0;
  for (int32_t i = 0; i < n_tokens / bs; ++i) {
    const uint64_t h = psw_block_hash(parent, tokens + static_cast<int64_t>(i) * bs, bs);
    const int rc = psw_block_pool_cache(pool, table_row[i], h);
    if (rc != PSW_OK) return rc;
    parent = h;
  }
  return PSW_OK;
}

}  // extern "C"
