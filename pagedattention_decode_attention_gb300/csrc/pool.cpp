// Host block pool: free list, refcounts, lazy allocation, fork, copy-on-write,
// prefix sharing, pinning and swapping to a host tier.  It produces block
// tables, slots and copy pairs for the device kernels and never touches
// device memory.
//
// Sources: "vLLM: treating the KV cache as virtual memory", section
// 碎片从哪里来 (fixed blocks, free list, refcounts, fork copies the table,
// copy-on-write, prefix blocks kept outside the free list); "第 6 章 缓存管理",
// section 块表长什么样 (refcount 1 -> 2 on sharing, -1 when a request ends,
// free at 0); OS-lab appendix sections 3.3 (allocate a physical page only when
// generation reaches it) and 4.4 (copy a shared partly-filled block on write;
// the last holder writes in place); "vLLM: treating the KV cache as virtual
// memory", section 调度：词一级的进入与退出 (a preempted sequence's KV goes to
// host memory block by block and comes back later; section 碎片从哪里来: the
// prefix cache keeps hot prefixes outside the free list) and "第 6 章 缓存管理",
// section 缓存放不下的时候 (spill cold cache to CPU memory; evict in
// least-recently-used order and recompute on the next use).
#include <algorithm>
#include <cstdint>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"
#include "status.h"

namespace {

struct Seq {
  std::vector<int32_t> table;  // device blocks, or host blocks while swapped
  int64_t ctx = 0;
  bool swapped = false;
  bool tokens_known = false;     // prefix cache: the token ids are tracked
  std::vector<int32_t> tokens;
  std::vector<uint64_t> hashes;  // key hash of each full block
};

// 64-bit FNV-1a over the parent hash (8 bytes, little-endian) and the token
// ids (int32, little-endian): the prefix-cache key of a full block.
uint64_t block_key_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = 0xCBF29CE484222325ull;
  auto mix = [&](uint8_t byte) {
    h ^= byte;
    h *= 0x100000001B3ull;
  };
  for (int i = 0; i < 8; ++i) mix(static_cast<uint8_t>(parent >> (8 * i)));
  for (int t = 0; t < n; ++t) {
    const uint32_t v = static_cast<uint32_t>(tokens[t]);
    for (int i = 0; i < 4; ++i) mix(static_cast<uint8_t>(v >> (8 * i)));
  }
  return h;
}

}  // namespace

struct pa_pool {
  int num_blocks = 0;
  int block_size = 16;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> refcount;
  std::vector<uint8_t> pinned;
  std::vector<uint8_t> on_free;     // mirrors membership of free_stack
  std::unordered_map<int, Seq> seqs;
  int next_id = 0;
  int64_t cow_copies = 0;
  int num_host_blocks = 0;
  std::vector<int32_t> host_free;   // top = back()
  // prefix cache
  bool prefix_cache = false;
  std::unordered_map<uint64_t, int32_t> cache;  // key hash -> block
  std::vector<uint8_t> keyed;
  std::vector<uint64_t> key_hash;
  std::vector<int32_t> key_parent;
  std::vector<int32_t> key_tokens;              // block_size ids per block
  // evictable keyed blocks, least recently used at the head
  std::vector<int32_t> lru_prev, lru_next;
  std::vector<uint8_t> in_lru;
  int32_t lru_head = -1, lru_tail = -1;
  int64_t lru_size = 0, hit_tokens = 0, evictions = 0;

  int64_t available() const { return static_cast<int64_t>(free_stack.size()) + lru_size; }
  void lru_push(int32_t b) {
    lru_prev[b] = lru_tail;
    lru_next[b] = -1;
    if (lru_tail >= 0) lru_next[lru_tail] = b;
    else lru_head = b;
    lru_tail = b;
    in_lru[b] = 1;
    ++lru_size;
  }
  void lru_remove(int32_t b) {
    if (lru_prev[b] >= 0) lru_next[lru_prev[b]] = lru_next[b];
    else lru_head = lru_next[b];
    if (lru_next[b] >= 0) lru_prev[lru_next[b]] = lru_prev[b];
    else lru_tail = lru_prev[b];
    in_lru[b] = 0;
    --lru_size;
  }
  // caller checks available() > 0 first
  int32_t alloc() {
    int32_t b;
    if (!free_stack.empty()) {
      b = free_stack.back();
      free_stack.pop_back();
      on_free[b] = 0;
    } else {
      b = lru_head;  // least recently used cached block: drop its key
      lru_remove(b);
      cache.erase(key_hash[b]);
      keyed[b] = 0;
      ++evictions;
    }
    refcount[b] = 1;
    return b;
  }
  void to_idle(int32_t b) {
    if (keyed[b]) {
      lru_push(b);
    } else {
      free_stack.push_back(b);
      on_free[b] = 1;
    }
  }
  void release(int32_t b) {
    if (--refcount[b] == 0 && !pinned[b]) to_idle(b);
  }
  Seq* find(int id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
};

namespace {
// A live sequence whose blocks are on the device, or null with the error set.
Seq* resident(pa_pool* pool, int id, const char* who, int* rc) {
  Seq* s = pool->find(id);
  if (!s) {
    *rc = pa::fail(PA_ERR_NOT_FOUND, "%s: unknown sequence", who);
    return nullptr;
  }
  if (s->swapped) {
    *rc = pa::fail(PA_ERR_INVALID_ARG, "%s: sequence is swapped out", who);
    return nullptr;
  }
  *rc = PA_OK;
  return s;
}
}  // namespace

extern "C" {

PA_API int pa_pool_create(int num_blocks, int block_size, const int32_t* initial_order,
                          pa_pool** pool) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: pool is NULL");
  *pool = nullptr;
  if (num_blocks <= 0 || block_size <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: num_blocks and block_size must be > 0");
  auto* p = new pa_pool();
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->refcount.assign(num_blocks, 0);
  p->pinned.assign(num_blocks, 0);
  p->on_free.assign(num_blocks, 0);
  p->keyed.assign(num_blocks, 0);
  p->key_hash.assign(num_blocks, 0);
  p->key_parent.assign(num_blocks, -1);
  p->key_tokens.assign(size_t(num_blocks) * block_size, 0);
  p->lru_prev.assign(num_blocks, -1);
  p->lru_next.assign(num_blocks, -1);
  p->in_lru.assign(num_blocks, 0);
  p->free_stack.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) {
    int32_t b = initial_order ? initial_order[i] : i;
    if (b < 0 || b >= num_blocks || p->on_free[b]) {
      delete p;
      return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: initial_order is not a permutation");
    }
    p->on_free[b] = 1;
    p->free_stack[num_blocks - 1 - i] = b;  // initial_order[0] ends on top
  }
  *pool = p;
  return PA_OK;
}

PA_API int pa_pool_destroy(pa_pool* pool) {
  delete pool;
  return PA_OK;
}

PA_API int pa_pool_new_seq(pa_pool* pool, int* seq_id) {
  if (!pool || !seq_id) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_new_seq: NULL argument");
  *seq_id = pool->next_id;
  pool->seqs.emplace(pool->next_id, Seq());
  pool->next_id++;
  return PA_OK;
}

PA_API int pa_pool_append_slot(pa_pool* pool, int seq, int64_t* slot, int64_t* cow_src,
                               int64_t* cow_dst) {
  if (!pool || !slot || !cow_src || !cow_dst)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_append_slot: NULL argument");
  int rc = PA_OK;
  Seq* s = resident(pool, seq, "pa_pool_append_slot", &rc);
  if (!s) return rc;
  const int64_t logical = s->ctx / pool->block_size;
  const int64_t offset = s->ctx % pool->block_size;
  int64_t src = -1, dst = -1;
  int32_t block;
  if (offset == 0) {
    if (pool->available() == 0) return pa::fail(PA_ERR_NO_BLOCKS, "pa_pool_append_slot: pool exhausted");
    block = pool->alloc();
    s->table.push_back(block);
  } else {
    block = s->table[logical];
    if (pool->refcount[block] > 1) {
      if (pool->available() == 0)
        return pa::fail(PA_ERR_NO_BLOCKS, "pa_pool_append_slot: pool exhausted (copy-on-write)");
      int32_t fresh = pool->alloc();
      pool->refcount[block] -= 1;  // stays >= 1: another holder remains
      s->table[logical] = fresh;
      src = block;
      dst = fresh;
      pool->cow_copies++;
      block = fresh;
    }
  }
  s->ctx += 1;
  s->tokens_known = false;  // the content of the new slot is unknown
  *slot = static_cast<int64_t>(block) * pool->block_size + offset;
  *cow_src = src;
  *cow_dst = dst;
  return PA_OK;
}

PA_API int pa_pool_enable_prefix_cache(pa_pool* pool, int on) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_enable_prefix_cache: NULL pool");
  if (!pool->seqs.empty() || pool->next_id != 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_enable_prefix_cache: enable before the first sequence");
  pool->prefix_cache = on != 0;
  return PA_OK;
}

PA_API int pa_pool_new_seq_with_prompt(pa_pool* pool, const int32_t* tokens, int n, int* seq_id,
                                       int* hit_tokens) {
  if (!pool || !seq_id || !hit_tokens || n < 0 || (n > 0 && !tokens))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_new_seq_with_prompt: bad argument");
  Seq s;
  s.tokens_known = true;
  const int bs = pool->block_size;
  if (pool->prefix_cache && n > 0) {
    const int limit = (n - 1) / bs;  // leave at least one token to compute
    uint64_t parent_hash = 0;
    int32_t parent_block = -1;
    for (int i = 0; i < limit; ++i) {
      const int32_t* chunk = tokens + size_t(i) * bs;
      const uint64_t h = block_key_hash(parent_hash, chunk, bs);
      auto it = pool->cache.find(h);
      if (it == pool->cache.end()) break;
      const int32_t b = it->second;
      if (pool->key_parent[b] != parent_block ||
          !std::equal(chunk, chunk + bs, pool->key_tokens.begin() + size_t(b) * bs))
        break;
      if (pool->refcount[b] == 0 && pool->in_lru[b]) pool->lru_remove(b);
      pool->refcount[b] += 1;
      s.table.push_back(b);
      s.hashes.push_back(h);
      s.tokens.insert(s.tokens.end(), chunk, chunk + bs);
      s.ctx += bs;
      parent_hash = h;
      parent_block = b;
    }
  }
  pool->hit_tokens += s.ctx;
  *hit_tokens = static_cast<int>(s.ctx);
  *seq_id = pool->next_id;
  pool->seqs.emplace(pool->next_id, std::move(s));
  pool->next_id++;
  return PA_OK;
}

PA_API int pa_pool_append_token(pa_pool* pool, int seq, int32_t token, int64_t* slot,
                                int64_t* cow_src, int64_t* cow_dst) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_append_token: NULL pool");
  int rc = PA_OK;
  Seq* s = resident(pool, seq, "pa_pool_append_token", &rc);
  if (!s) return rc;
  const bool known = s->tokens_known;
  rc = pa_pool_append_slot(pool, seq, slot, cow_src, cow_dst);
  if (rc != PA_OK || !known) return rc;
  s->tokens_known = true;
  s->tokens.push_back(token);
  const int bs = pool->block_size;
  if (pool->prefix_cache && s->ctx % bs == 0) {
    const int64_t i = s->ctx / bs - 1;
    const uint64_t parent_hash = i > 0 ? s->hashes[i - 1] : 0;
    const int32_t parent_block = i > 0 ? s->table[i - 1] : -1;
    const int32_t* chunk = s->tokens.data() + size_t(i) * bs;
    const uint64_t h = block_key_hash(parent_hash, chunk, bs);
    s->hashes.push_back(h);
    const int32_t b = s->table[i];
    if (!pool->cache.count(h) && !pool->keyed[b]) {
      pool->cache.emplace(h, b);
      pool->keyed[b] = 1;
      pool->key_hash[b] = h;
      pool->key_parent[b] = parent_block;
      std::copy(chunk, chunk + bs, pool->key_tokens.begin() + size_t(b) * bs);
    }
  }
  return PA_OK;
}

PA_API int pa_pool_append_tokens(pa_pool* pool, const int32_t* seqs, const int32_t* tokens,
                                 int n, int64_t* slots, int64_t* pairs, int pair_cap,
                                 int* num_pairs, int* done) {
  if (!pool || (n > 0 && (!seqs || !tokens || !slots)) || !num_pairs || !done || n < 0 ||
      pair_cap < 0 || (pair_cap > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_append_tokens: bad argument");
  *num_pairs = 0;
  *done = 0;
  for (int i = 0; i < n; ++i) {
    int64_t src, dst;
    // as in pa_pool_append_slots: room for a copy pair before the slot is taken
    Seq* s = pool->find(seqs[i]);
    if (s && !s->swapped && s->ctx % pool->block_size != 0 &&
        pool->refcount[s->table[s->ctx / pool->block_size]] > 1 && *num_pairs >= pair_cap)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_append_tokens: pair buffer full");
    int rc = pa_pool_append_token(pool, seqs[i], tokens[i], &slots[i], &src, &dst);
    if (rc != PA_OK) return rc;
    if (src >= 0) {
      pairs[2 * *num_pairs] = src;
      pairs[2 * *num_pairs + 1] = dst;
      (*num_pairs)++;
    }
    (*done)++;
  }
  return PA_OK;
}

PA_API int pa_pool_append_slots(pa_pool* pool, const int32_t* seqs, int n, int64_t* slots,
                                int64_t* pairs, int pair_cap, int* num_pairs, int* done) {
  if (!pool || (n > 0 && (!seqs || !slots)) || !num_pairs || !done || n < 0 ||
      pair_cap < 0 || (pair_cap > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_append_slots: bad argument");
  *num_pairs = 0;
  *done = 0;
  for (int i = 0; i < n; ++i) {
    int64_t src, dst;
    // A copy pair needs room before the slot is taken, so a full pair buffer
    // never leaves a copy unreported.
    Seq* s = pool->find(seqs[i]);
    if (s && !s->swapped && s->ctx % pool->block_size != 0 &&
        pool->refcount[s->table[s->ctx / pool->block_size]] > 1 && *num_pairs >= pair_cap)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_append_slots: pair buffer full");
    int rc = pa_pool_append_slot(pool, seqs[i], &slots[i], &src, &dst);
    if (rc != PA_OK) return rc;
    if (src >= 0) {
      pairs[2 * *num_pairs] = src;
      pairs[2 * *num_pairs + 1] = dst;
      (*num_pairs)++;
    }
    (*done)++;
  }
  return PA_OK;
}

PA_API int pa_pool_fork(pa_pool* pool, int parent, int* child) {
  if (!pool || !child) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_fork: NULL argument");
  int rc = PA_OK;
  Seq* p = resident(pool, parent, "pa_pool_fork", &rc);
  if (!p) return rc;
  Seq c;
  c.table = p->table;
  c.ctx = p->ctx;
  c.tokens_known = p->tokens_known;
  c.tokens = p->tokens;
  c.hashes = p->hashes;
  for (int32_t b : c.table) pool->refcount[b] += 1;
  *child = pool->next_id;
  pool->seqs.emplace(pool->next_id, std::move(c));
  pool->next_id++;
  return PA_OK;
}

PA_API int pa_pool_share_prefix(pa_pool* pool, int src_seq, int dst_seq, int num_tokens) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_share_prefix: NULL pool");
  int rc = PA_OK;
  Seq* src = resident(pool, src_seq, "pa_pool_share_prefix", &rc);
  if (!src) return rc;
  Seq* dst = resident(pool, dst_seq, "pa_pool_share_prefix", &rc);
  if (!dst) return rc;
  if (dst->ctx != 0 || !dst->table.empty())
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_share_prefix: destination must be empty");
  if (num_tokens <= 0 || num_tokens > src->ctx)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_share_prefix: num_tokens out of range");
  const int64_t count = (num_tokens + pool->block_size - 1) / pool->block_size;
  dst->table.assign(src->table.begin(), src->table.begin() + count);
  dst->ctx = num_tokens;
  dst->tokens_known = src->tokens_known;
  const size_t nt = src->tokens_known ? std::min(src->tokens.size(), size_t(num_tokens)) : 0;
  dst->tokens.assign(src->tokens.begin(), src->tokens.begin() + nt);
  const size_t nh = std::min(src->hashes.size(), size_t(num_tokens / pool->block_size));
  dst->hashes.assign(src->hashes.begin(), src->hashes.begin() + nh);
  for (int32_t b : dst->table) pool->refcount[b] += 1;
  return PA_OK;
}

PA_API int pa_pool_pin(pa_pool* pool, int seq, int num_tokens) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_pin: NULL pool");
  int rc = PA_OK;
  Seq* s = resident(pool, seq, "pa_pool_pin", &rc);
  if (!s) return rc;
  if (num_tokens < 0 || num_tokens > s->ctx)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_pin: num_tokens out of range");
  const int64_t count = (num_tokens + pool->block_size - 1) / pool->block_size;
  for (int64_t i = 0; i < count; ++i) pool->pinned[s->table[i]] = 1;
  return PA_OK;
}

PA_API int pa_pool_unpin(pa_pool* pool, int block) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_unpin: NULL pool");
  if (block < 0 || block >= pool->num_blocks || !pool->pinned[block])
    return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_unpin: block is not pinned");
  pool->pinned[block] = 0;
  if (pool->refcount[block] == 0) pool->to_idle(block);
  return PA_OK;
}

PA_API int pa_pool_free_seq(pa_pool* pool, int seq) {
  if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_free_seq: NULL pool");
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_free_seq: unknown sequence");
  const auto& table = it->second.table;
  for (auto b = table.rbegin(); b != table.rend(); ++b) {
    if (it->second.swapped)
      pool->host_free.push_back(*b);
    else
      pool->release(*b);
  }
  pool->seqs.erase(it);
  return PA_OK;
}

PA_API int pa_pool_set_host_blocks(pa_pool* pool, int num_host_blocks,
                                   const int32_t* initial_order) {
  if (!pool || num_host_blocks < 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_set_host_blocks: bad argument");
  for (const auto& kv : pool->seqs)
    if (kv.second.swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_set_host_blocks: sequences are swapped out");
  std::vector<uint8_t> seen(num_host_blocks, 0);
  std::vector<int32_t> stack(num_host_blocks);
  for (int i = 0; i < num_host_blocks; ++i) {
    const int32_t b = initial_order ? initial_order[i] : i;
    if (b < 0 || b >= num_host_blocks || seen[b])
      return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_set_host_blocks: initial_order is not a permutation");
    seen[b] = 1;
    stack[num_host_blocks - 1 - i] = b;  // initial_order[0] ends on top
  }
  pool->num_host_blocks = num_host_blocks;
  pool->host_free.swap(stack);
  return PA_OK;
}

PA_API int pa_pool_swap_out(pa_pool* pool, int seq, int64_t* pairs, int cap, int* n) {
  if (!pool || !n || cap < 0 || (cap > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_swap_out: bad argument");
  int rc = PA_OK;
  Seq* s = resident(pool, seq, "pa_pool_swap_out", &rc);
  if (!s) return rc;
  const int len = static_cast<int>(s->table.size());
  for (int32_t b : s->table)
    if (pool->refcount[b] != 1 || pool->pinned[b])
      return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_swap_out: a shared or pinned block cannot leave");
  if (len > cap) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_swap_out: pair buffer too small");
  if (len > static_cast<int>(pool->host_free.size()))
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_pool_swap_out: host tier exhausted");
  std::vector<int32_t> host(len);
  for (int i = 0; i < len; ++i) {
    host[i] = pool->host_free.back();
    pool->host_free.pop_back();
    pairs[2 * i] = s->table[i];
    pairs[2 * i + 1] = host[i];
  }
  for (int i = len - 1; i >= 0; --i) pool->release(s->table[i]);
  s->table.swap(host);
  s->swapped = true;
  *n = len;
  return PA_OK;
}

PA_API int pa_pool_swap_in(pa_pool* pool, int seq, int64_t* pairs, int cap, int* n) {
  if (!pool || !n || cap < 0 || (cap > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_swap_in: bad argument");
  Seq* s = pool->find(seq);
  if (!s) return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_swap_in: unknown sequence");
  if (!s->swapped) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_swap_in: sequence is not swapped out");
  const int len = static_cast<int>(s->table.size());
  if (len > cap) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_swap_in: pair buffer too small");
  if (len > pool->available())
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_pool_swap_in: pool exhausted");
  std::vector<int32_t> dev(len);
  for (int i = 0; i < len; ++i) {
    dev[i] = pool->alloc();
    pairs[2 * i] = s->table[i];
    pairs[2 * i + 1] = dev[i];
  }
  for (int i = len - 1; i >= 0; --i) pool->host_free.push_back(s->table[i]);
  s->table.swap(dev);
  s->swapped = false;
  *n = len;
  return PA_OK;
}

PA_API int pa_pool_is_swapped(pa_pool* pool, int seq, int* swapped) {
  if (!pool || !swapped) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_is_swapped: NULL argument");
  Seq* s = pool->find(seq);
  if (!s) return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_is_swapped: unknown sequence");
  *swapped = s->swapped ? 1 : 0;
  return PA_OK;
}

PA_API int pa_pool_block_table(pa_pool* pool, int seq, int32_t* out, int cap, int* n,
                               int* ctx_len) {
  if (!pool || !n || !ctx_len || cap < 0 || (cap > 0 && !out))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_block_table: bad argument");
  Seq* s = pool->find(seq);
  if (!s) return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_block_table: unknown sequence");
  const int len = static_cast<int>(s->table.size());
  std::copy(s->table.begin(), s->table.begin() + std::min(len, cap), out);
  *n = len;
  *ctx_len = static_cast<int>(s->ctx);
  return PA_OK;
}

PA_API int pa_pool_refcount(pa_pool* pool, int block, int* rc) {
  if (!pool || !rc) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_refcount: NULL argument");
  if (block < 0 || block >= pool->num_blocks)
    return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_refcount: block out of range");
  *rc = pool->refcount[block];
  return PA_OK;
}

PA_API int pa_pool_stats(pa_pool* pool, pa_pool_stats_t* st) {
  if (!pool || !st) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_stats: NULL argument");
  st->num_blocks = pool->num_blocks;
  st->free_blocks = static_cast<int64_t>(pool->free_stack.size());
  st->used_blocks = st->pinned_blocks = st->shared_blocks = 0;
  for (int b = 0; b < pool->num_blocks; ++b) {
    st->used_blocks += pool->refcount[b] > 0;
    st->shared_blocks += pool->refcount[b] > 1;
    st->pinned_blocks += pool->pinned[b] != 0;
  }
  st->cow_copies = pool->cow_copies;
  st->live_seqs = static_cast<int64_t>(pool->seqs.size());
  st->tokens = st->internal_frag_slots = 0;
  st->cached_blocks = static_cast<int64_t>(pool->cache.size());
  st->evictable_blocks = pool->lru_size;
  st->prefix_hit_tokens = pool->hit_tokens;
  st->evictions = pool->evictions;
  st->host_blocks = pool->num_host_blocks;
  st->host_free_blocks = static_cast<int64_t>(pool->host_free.size());
  st->swapped_seqs = 0;
  for (const auto& kv : pool->seqs) {
    st->swapped_seqs += kv.second.swapped;
    st->tokens += kv.second.ctx;
    st->internal_frag_slots +=
        static_cast<int64_t>(kv.second.table.size()) * pool->block_size - kv.second.ctx;
  }
  return PA_OK;
}

}  // extern "C"
