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
// Policy choices the pages leave open, stated in pagedkv.h: the free list is
// a stack seeded from a caller-given order; a fresh block is taken when the
// length is a multiple of the block size before the append; a failing call
// leaves the pool unchanged.
#include <cstdint>
#include <cstring>
#include <new>
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

  bool valid_block(int32_t b) const { return b >= 0 && b < num_blocks; }
  bool valid_seq(int32_t s) const {
    return s >= 0 && s < static_cast<int32_t>(seqs.size()) && seqs[s].live;
  }
  int32_t pop() {
    int32_t b = free_stack.back();
    free_stack.pop_back();
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) free_stack.push_back(b);
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
    if (p->ref[old] > 1) {
      const int32_t fresh = p->pop();
      p->ref[old] -= 1;  // was > 1, stays >= 1
      q.table[j] = fresh;
      *cow = true;
      *src = old;
      *dst = fresh;
    }
  }
  q.len = pos + 1;
  *slot = static_cast<int64_t>(q.table[j]) * bs + pos % bs;
}

// Blocks that appending n tokens to q would take from the free list.
int64_t blocks_for_append(const pa_pool* p, const pa_pool::Seq& q, int32_t n) {
  if (n <= 0) return 0;
  const int32_t bs = p->block_size;
  int64_t need = 0;
  // the partially filled last block, if shared, costs one copy-on-write block
  if (q.len % bs != 0 && p->ref[q.table[q.len / bs]] > 1) need += 1;
  // fresh blocks for every boundary crossed: positions len..len+n-1 that are multiples of bs
  const int64_t first = q.len, last = static_cast<int64_t>(q.len) + n - 1;
  need += last / bs - (first + bs - 1) / bs + 1;
  return need;
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
  if (p->free_stack.empty()) return fail(PA_ERR_OOM, "pa_pool_alloc: pool exhausted");
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
  st->free_blocks = static_cast<int32_t>(p->free_stack.size());
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
  if (blocks_for_append(p, q, 1) > static_cast<int64_t>(p->free_stack.size()))
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
  if (blocks_for_append(p, q, n) > static_cast<int64_t>(p->free_stack.size()))
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
