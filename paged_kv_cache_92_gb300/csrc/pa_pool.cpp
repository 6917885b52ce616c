// Host-side block pool: free list, per-sequence block tables, refcounts,
// copy-on-write planning.
//
// What it models: "How Paged Attention and Continuous Batching Actually
// Work", §Paged attention: virtual memory for the KV cache (fixed 16-token
// blocks carved into a pool held in a free list; allocation pops, freeing
// pushes, both O(1); a sequence holds ceil(t/16) blocks; sharing by
// reference count). "Paged Attention as a Memory Manager", §Prefix Caching
// and Copy-on-Write (allocate a fresh block, copy, decrement the old block's
// refcount, update the table). PagedAttention architecture walk-through,
// §The architecture: every piece explained (table entry i backs tokens
// [16i, 16i+15]; every 16th token grabs a fresh block; blocks are immutable
// while shared).
//
// Prefix cache: "How Paged Attention and Continuous Batching Actually
// Work", FAQ (prefix caching is a consequence of paging: blocks are
// content-hashed, a prompt that hashes to resident blocks points at them);
// PagedAttention architecture walk-through, §The architecture (each full
// block's token ids hashed chained with its prefix hash; a match maps the
// existing block with a bumped refcount) and §End-to-end flow (the shared
// preamble stays warm for the next request).
//
// Policy choices the pages leave open, stated in pagedkv.h: the free list is
// a stack seeded from a caller-given order; a fresh block is taken when the
// length is a multiple of the block size before the append; a failing call
// leaves the pool unchanged; cached blocks freed to refcount 0 stay cached
// and are handed out only after every never-cached free block, least
// recently freed first.
#include <cstdint>
#include <cstring>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_internal.h"

struct pa_pool {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // back() is handed out next
  std::vector<int32_t> ref;
  struct Seq {
    bool live = false;
    int32_t len = 0;
    std::vector<int32_t> table;
  };
  std::vector<Seq> seqs;
  int32_t live_seqs = 0;

  // prefix cache: per-block chain key, the key of the block before it, its
  // token ids; key -> block; cached blocks with refcount 0, least recently
  // freed first
  std::vector<uint8_t> cached;
  std::vector<uint64_t> key, parent_key;
  std::vector<std::vector<int32_t>> key_tokens;
  std::unordered_map<uint64_t, int32_t> by_key;
  std::list<int32_t> evictable;
  std::vector<std::list<int32_t>::iterator> ev_pos;
  int64_t lookups = 0, hits = 0;

  bool valid_block(int32_t b) const { return b >= 0 && b < num_blocks; }
  bool valid_seq(int32_t s) const {
    return s >= 0 && s < static_cast<int32_t>(seqs.size()) && seqs[s].live;
  }
  // blocks that can be handed out
  size_t available() const { return free_stack.size() + evictable.size(); }
  void uncache(int32_t b) {
    auto it = by_key.find(key[b]);
    if (it != by_key.end() && it->second == b) by_key.erase(it);
    cached[b] = 0;
    key_tokens[b].clear();
  }
  int32_t pop() {
    int32_t b;
    if (!free_stack.empty()) {
      b = free_stack.back();
      free_stack.pop_back();
    } else {  // evict the least recently freed cached block
      b = evictable.front();
      evictable.pop_front();
      uncache(b);
    }
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) {
      if (cached[b]) {
        evictable.push_back(b);
        ev_pos[b] = std::prev(evictable.end());
      } else {
        free_stack.push_back(b);
      }
    }
  }
};

namespace {

pa_status fail(pa_status s, const char* msg) { return pa::set_error(s, msg); }

// Appends one token to seq s. The caller has checked that enough free blocks
// exist, so this cannot fail.
void append_one(pa_pool* p, pa_pool::Seq& q, int64_t* slot, int32_t* src, int32_t* dst,
                bool* cow) {
  const int32_t bs = p->block_size;
  const int32_t pos = q.len;
  const int32_t j = pos / bs;
  *cow = false;
  if (pos % bs == 0) {
    q.table.push_back(p->pop());
  } else {
    const int32_t old = q.table[j];
    if (p->ref[old] > 1 || p->cached[old]) {  // shared, or cached (immutable)
      const int32_t fresh = p->pop();
      p->release(old);
      q.table[j] = fresh;
      *cow = true;
      *src = old;
      *dst = fresh;
    }
  }
  q.len = pos + 1;
  *slot = static_cast<int64_t>(q.table[j]) * bs + pos % bs;
}

// Whether appending n tokens to q finds enough blocks, following the order
// in which append_one takes and releases them.
bool append_fits(const pa_pool* p, const pa_pool::Seq& q, int32_t n) {
  if (n <= 0) return true;
  const int32_t bs = p->block_size;
  int64_t avail = static_cast<int64_t>(p->available());
  // the partially filled last block, if shared or cached, is first copied
  // into a fresh block; a cached block only this sequence held then becomes
  // free (evictable) again
  if (q.len % bs != 0) {
    const int32_t b = q.table[q.len / bs];
    if (p->ref[b] > 1 || p->cached[b]) {
      if (avail < 1) return false;
      if (p->ref[b] > 1) avail -= 1;
    }
  }
  // fresh blocks for every boundary crossed: positions len..len+n-1 that are multiples of bs
  const int64_t first = q.len, last = static_cast<int64_t>(q.len) + n - 1;
  return avail >= last / bs - (first + bs - 1) / bs + 1;
}

// Chain key of a full block: its predecessor's key and its token ids
// (splitmix64-style mixing; collisions are caught by the stored ids).
uint64_t mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}
uint64_t chain_key(uint64_t parent, const int32_t* tokens, int32_t n) {
  uint64_t k = mix64(parent ^ 0xC2B2AE3D27D4EB4Full);
  for (int32_t i = 0; i < n; ++i) k = mix64(k ^ static_cast<uint32_t>(tokens[i]));
  return k;
}

}  // namespace

extern "C" {

pa_status pa_pool_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                         pa_pool** out) {
  if (!out) return fail(PA_ERR_INVALID_ARG, "pa_pool_create: out is NULL");
  *out = nullptr;
  if (num_blocks < 1 || block_size < 1)
    return fail(PA_ERR_INVALID_ARG, "pa_pool_create: num_blocks and block_size must be >= 1");
  pa_pool* p = new (std::nothrow) pa_pool;
  if (!p) return fail(PA_ERR_OOM, "pa_pool_create: host allocation failed");
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->ref.assign(num_blocks, 0);
  p->cached.assign(num_blocks, 0);
  p->key.assign(num_blocks, 0);
  p->parent_key.assign(num_blocks, 0);
  p->key_tokens.resize(num_blocks);
  p->ev_pos.resize(num_blocks);
  p->free_stack.resize(num_blocks);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete p;
        return fail(PA_ERR_INVALID_ARG, "pa_pool_create: free_order is not a permutation");
      }
      seen[b] = 1;
      p->free_stack[num_blocks - 1 - i] = b;
    }
  } else {
    for (int32_t i = 0; i < num_blocks; ++i) p->free_stack[num_blocks - 1 - i] = i;
  }
  *out = p;
  return PA_OK;
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

pa_status pa_pool_alloc(pa_pool* p, int32_t* block) {
  if (!p || !block) return fail(PA_ERR_INVALID_ARG, "pa_pool_alloc: NULL argument");
  if (p->available() == 0) return fail(PA_ERR_OOM, "pa_pool_alloc: pool exhausted");
  *block = p->pop();
  return PA_OK;
}

pa_status pa_pool_incref(pa_pool* p, int32_t block) {
  if (!p) return fail(PA_ERR_INVALID_ARG, "pa_pool_incref: NULL pool");
  if (!p->valid_block(block)) return fail(PA_ERR_BOUNDS, "pa_pool_incref: block id out of range");
  if (p->ref[block] <= 0) return fail(PA_ERR_REFCOUNT, "pa_pool_incref: block is free");
  p->ref[block] += 1;
  return PA_OK;
}

pa_status pa_pool_decref(pa_pool* p, int32_t block) {
  if (!p) return fail(PA_ERR_INVALID_ARG, "pa_pool_decref: NULL pool");
  if (!p->valid_block(block)) return fail(PA_ERR_BOUNDS, "pa_pool_decref: block id out of range");
  if (p->ref[block] <= 0) return fail(PA_ERR_REFCOUNT, "pa_pool_decref: block is already free");
  p->release(block);
  return PA_OK;
}

int32_t pa_pool_refcount(const pa_pool* p, int32_t block) {
  if (!p || !p->valid_block(block)) return -1;
  return p->ref[block];
}

pa_status pa_pool_stats(const pa_pool* p, pa_pool_stats_t* st) {
  if (!p || !st) return fail(PA_ERR_INVALID_ARG, "pa_pool_stats: NULL argument");
  std::memset(st, 0, sizeof(*st));
  st->num_blocks = p->num_blocks;
  st->block_size = p->block_size;
  st->free_blocks = static_cast<int32_t>(p->available());
  for (int32_t r : p->ref) {
    if (r >= 1) st->used_blocks += 1;
    if (r >= 2) st->shared_blocks += 1;
    if (r > st->max_refcount) st->max_refcount = r;
  }
  st->live_seqs = p->live_seqs;
  return PA_OK;
}

pa_status pa_seq_create(pa_pool* p, int32_t* seq) {
  if (!p || !seq) return fail(PA_ERR_INVALID_ARG, "pa_seq_create: NULL argument");
  p->seqs.emplace_back();
  p->seqs.back().live = true;
  p->live_seqs += 1;
  *seq = static_cast<int32_t>(p->seqs.size()) - 1;
  return PA_OK;
}

pa_status pa_seq_free(pa_pool* p, int32_t seq) {
  if (!p) return fail(PA_ERR_INVALID_ARG, "pa_seq_free: NULL pool");
  if (!p->valid_seq(seq)) return fail(PA_ERR_BOUNDS, "pa_seq_free: unknown sequence");
  pa_pool::Seq& q = p->seqs[seq];
  for (int32_t b : q.table) p->release(b);
  q.table.clear();
  q.table.shrink_to_fit();
  q.len = 0;
  q.live = false;
  p->live_seqs -= 1;
  return PA_OK;
}

pa_status pa_seq_fork(pa_pool* p, int32_t parent, int32_t num_tokens, int32_t* child) {
  if (!p || !child) return fail(PA_ERR_INVALID_ARG, "pa_seq_fork: NULL argument");
  if (!p->valid_seq(parent)) return fail(PA_ERR_BOUNDS, "pa_seq_fork: unknown parent");
  if (num_tokens < 0 || num_tokens > p->seqs[parent].len)
    return fail(PA_ERR_INVALID_ARG, "pa_seq_fork: num_tokens outside [0, parent length]");
  const int32_t n = (num_tokens + p->block_size - 1) / p->block_size;
  pa_pool::Seq c;
  c.live = true;
  c.len = num_tokens;
  c.table.assign(p->seqs[parent].table.begin(), p->seqs[parent].table.begin() + n);
  for (int32_t b : c.table) p->ref[b] += 1;
  p->seqs.push_back(std::move(c));
  p->live_seqs += 1;
  *child = static_cast<int32_t>(p->seqs.size()) - 1;
  return PA_OK;
}

pa_status pa_seq_append_slot(pa_pool* p, int32_t seq, int64_t* slot, int32_t cow_pair[2],
                             int32_t* has_cow) {
  if (!p || !slot) return fail(PA_ERR_INVALID_ARG, "pa_seq_append_slot: NULL argument");
  if (!p->valid_seq(seq)) return fail(PA_ERR_BOUNDS, "pa_seq_append_slot: unknown sequence");
  pa_pool::Seq& q = p->seqs[seq];
  if (q.len == INT32_MAX) return fail(PA_ERR_INVALID_ARG, "pa_seq_append_slot: length overflow");
  if (!append_fits(p, q, 1))
    return fail(PA_ERR_OOM, "pa_seq_append_slot: pool exhausted");
  int32_t src = -1, dst = -1;
  bool cow = false;
  append_one(p, q, slot, &src, &dst, &cow);
  if (has_cow) *has_cow = cow ? 1 : 0;
  if (cow_pair) {
    cow_pair[0] = cow ? src : -1;
    cow_pair[1] = cow ? dst : -1;
  }
  return PA_OK;
}

pa_status pa_seq_append_tokens(pa_pool* p, int32_t seq, int32_t n, int64_t* slots,
                               int32_t* cow_pairs, int32_t* num_cow) {
  if (!p) return fail(PA_ERR_INVALID_ARG, "pa_seq_append_tokens: NULL pool");
  if (!p->valid_seq(seq)) return fail(PA_ERR_BOUNDS, "pa_seq_append_tokens: unknown sequence");
  if (n < 0) return fail(PA_ERR_INVALID_ARG, "pa_seq_append_tokens: n < 0");
  pa_pool::Seq& q = p->seqs[seq];
  if (static_cast<int64_t>(q.len) + n > INT32_MAX)
    return fail(PA_ERR_INVALID_ARG, "pa_seq_append_tokens: length overflow");
  if (!append_fits(p, q, n))
    return fail(PA_ERR_OOM, "pa_seq_append_tokens: pool exhausted");
  int32_t ncow = 0;
  for (int32_t i = 0; i < n; ++i) {
    int64_t s;
    int32_t src, dst;
    bool cow;
    append_one(p, q, &s, &src, &dst, &cow);
    if (slots) slots[i] = s;
    if (cow) {
      if (cow_pairs) {
        cow_pairs[2 * ncow] = src;
        cow_pairs[2 * ncow + 1] = dst;
      }
      ncow += 1;
    }
  }
  if (num_cow) *num_cow = ncow;
  return PA_OK;
}

pa_status pa_seq_length(const pa_pool* p, int32_t seq, int32_t* length) {
  if (!p || !length) return fail(PA_ERR_INVALID_ARG, "pa_seq_length: NULL argument");
  if (!p->valid_seq(seq)) return fail(PA_ERR_BOUNDS, "pa_seq_length: unknown sequence");
  *length = p->seqs[seq].len;
  return PA_OK;
}

pa_status pa_seq_table(const pa_pool* p, int32_t seq, int32_t* out, int32_t cap,
                       int32_t* n_blocks) {
  if (!p || !n_blocks) return fail(PA_ERR_INVALID_ARG, "pa_seq_table: NULL argument");
  if (!p->valid_seq(seq)) return fail(PA_ERR_BOUNDS, "pa_seq_table: unknown sequence");
  const pa_pool::Seq& q = p->seqs[seq];
  const int32_t n = static_cast<int32_t>(q.table.size());
  *n_blocks = n;
  if (out) {
    if (cap < n) return fail(PA_ERR_INVALID_ARG, "pa_seq_table: cap smaller than the table");
    std::memcpy(out, q.table.data(), sizeof(int32_t) * n);
  }
  return PA_OK;
}

pa_status pa_seq_create_prompt(pa_pool* p, const int32_t* tokens, int32_t num_tokens,
                               int32_t* seq, int32_t* cached_tokens, int64_t* slots) {
  if (!p || !seq || !cached_tokens || num_tokens < 0 || (num_tokens > 0 && !tokens))
    return fail(PA_ERR_INVALID_ARG, "pa_seq_create_prompt: bad argument");
  const int32_t bs = p->block_size;
  const int32_t nfull = num_tokens / bs;
  const int32_t nblocks = (num_tokens + bs - 1) / bs;
  // chain keys of the full blocks; the leading run found in the cache
  std::vector<uint64_t> keys(nfull);
  std::vector<int32_t> matched;
  int64_t revive = 0;  // matched blocks now evictable: they stop being available
  uint64_t parent = 0;
  bool matching = true;
  for (int32_t i = 0; i < nfull; ++i) {
    const int32_t* tk = tokens + static_cast<size_t>(i) * bs;
    keys[i] = chain_key(parent, tk, bs);
    if (matching) {
      auto it = p->by_key.find(keys[i]);
      const int32_t b = it == p->by_key.end() ? -1 : it->second;
      if (b >= 0 && p->parent_key[b] == parent &&
          std::memcmp(p->key_tokens[b].data(), tk, sizeof(int32_t) * bs) == 0) {
        matched.push_back(b);
        if (p->ref[b] == 0) revive += 1;
      } else {
        matching = false;
      }
    }
    parent = keys[i];
  }
  const int64_t fresh = nblocks - static_cast<int64_t>(matched.size());
  if (fresh > static_cast<int64_t>(p->available()) - revive)
    return fail(PA_ERR_OOM, "pa_seq_create_prompt: pool exhausted");
  // commit: map the matches, then allocate (and enter into the cache) the rest
  pa_pool::Seq q;
  q.live = true;
  q.len = num_tokens;
  for (int32_t b : matched) {
    if (p->ref[b] == 0) {
      p->evictable.erase(p->ev_pos[b]);
      p->ref[b] = 1;
    } else {
      p->ref[b] += 1;
    }
    q.table.push_back(b);
  }
  for (int32_t i = static_cast<int32_t>(matched.size()); i < nblocks; ++i) {
    const int32_t b = p->pop();
    q.table.push_back(b);
    if (i < nfull && p->by_key.find(keys[i]) == p->by_key.end()) {
      p->cached[b] = 1;
      p->key[b] = keys[i];
      p->parent_key[b] = i > 0 ? keys[i - 1] : 0;
      p->key_tokens[b].assign(tokens + static_cast<size_t>(i) * bs,
                              tokens + static_cast<size_t>(i + 1) * bs);
      p->by_key[keys[i]] = b;
    }
  }
  p->lookups += nfull;
  p->hits += static_cast<int64_t>(matched.size());
  if (slots)
    for (int32_t t = 0; t < num_tokens; ++t)
      slots[t] = static_cast<int64_t>(q.table[t / bs]) * bs + t % bs;
  *cached_tokens = static_cast<int32_t>(matched.size()) * bs;
  p->seqs.push_back(std::move(q));
  p->live_seqs += 1;
  *seq = static_cast<int32_t>(p->seqs.size()) - 1;
  return PA_OK;
}

pa_status pa_pool_prefix_stats(const pa_pool* p, pa_prefix_stats_t* st) {
  if (!p || !st) return fail(PA_ERR_INVALID_ARG, "pa_pool_prefix_stats: NULL argument");
  st->cached_blocks = static_cast<int32_t>(p->by_key.size());
  st->evictable_blocks = static_cast<int32_t>(p->evictable.size());
  st->lookups = p->lookups;
  st->hits = p->hits;
  return PA_OK;
}

pa_status pa_pool_export(const pa_pool* p, const int32_t* seqs, int32_t n, int32_t max_blocks,
                         int32_t* tables, int32_t* lens) {
  if (!p || (n > 0 && (!seqs || !tables || !lens)) || n < 0 || max_blocks < 1)
    return fail(PA_ERR_INVALID_ARG, "pa_pool_export: bad argument");
  for (int32_t i = 0; i < n; ++i) {
    if (!p->valid_seq(seqs[i])) return fail(PA_ERR_BOUNDS, "pa_pool_export: unknown sequence");
    if (static_cast<int32_t>(p->seqs[seqs[i]].table.size()) > max_blocks)
      return fail(PA_ERR_INVALID_ARG, "pa_pool_export: a table exceeds max_blocks");
  }
  for (int32_t i = 0; i < n; ++i) {
    const pa_pool::Seq& q = p->seqs[seqs[i]];
    int32_t* row = tables + static_cast<size_t>(i) * max_blocks;
    const int32_t nb = static_cast<int32_t>(q.table.size());
    std::memcpy(row, q.table.data(), sizeof(int32_t) * nb);
    for (int32_t j = nb; j < max_blocks; ++j) row[j] = -1;
    lens[i] = q.len;
  }
  return PA_OK;
}

}  // extern "C"
