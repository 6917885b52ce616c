// Launch rules of the query-major tensor-core kernel (pa_prefill_tc.cu), the
// path for many new tokens per sequence. Not part of the public ABI.
#pragma once

#include "pa_internal.h"

namespace pa {

// A unit of work is (sequence, group of KV heads, tile of 128 query rows =
// tokens x G heads of each head in the group, split of the keys); one
// persistent CTA per SM takes its share of them.
inline int query_major_tiles(const pa_decode_params* p) {
  const int rows = query_len_of(p) * (p->num_q_heads / p->num_kv_heads);
  return (rows + 127) / 128;
}
// KV heads per CTA: two (adjacent in a block, one 4 KiB box per half) when a
// head has at most 64 rows and the head count is even, else one.
inline int query_major_heads(const pa_decode_params* p) {
  const int rows = query_len_of(p) * (p->num_q_heads / p->num_kv_heads);
  return rows <= 64 && p->num_kv_heads % 2 == 0 ? 2 : 1;
}
// Splits of each item's keys: enough to bring small batches to 256 items,
// each split at least 4 chunks long (a chunk is 64 / heads-per-item keys),
// at most 16. The partials of a split live in the workspace.
inline int query_major_splits(const pa_decode_params* p) {
  const int hb = query_major_heads(p);
  const int64_t units = int64_t(p->num_seqs) * (p->num_kv_heads / hb) * query_major_tiles(p);
  if (units <= 0 || units >= 256) return 1;
  const int chunks = (p->max_context_len + 64 / hb - 1) / (64 / hb);
  int ns = int((256 + units - 1) / units);
  if (ns > chunks / 4) ns = chunks / 4;
  if (ns > 16) ns = 16;
  return ns < 1 ? 1 : ns;
}
// It takes the bf16 cache at head_dim 128 and block size 16 or 32 when the
// column-group decode would split the new tokens into several groups (each
// re-reading the keys), or when a KV head has at least 16 query rows (new
// tokens x G) and the batch gives it 128 (sequence, KV head, tile) units.
inline bool use_query_major(const pa_decode_params* p) {
  const int g = p->num_q_heads / p->num_kv_heads;
  return p->variant == PA_DECODE_TENSOR_CORE && p->kv_dtype == PA_KV_BF16 && p->head_dim == 128 &&
         (p->block_size == 16 || p->block_size == 32) && query_len_of(p) > 1 &&
         (g == 1 || g == 2 || g == 4 || g == 8) &&
         (tc_n_groups(p) > 1 ||
          (query_len_of(p) * g >= 16 &&
           int64_t(p->num_seqs) * p->num_kv_heads * query_major_tiles(p) >= 128));
}

// part_ml / part_o: the workspace's partials when query_major_splits(p) > 1
// ([B*Q*Hq][splits][2] and [B*Q*Hq][splits][128] floats), else unused.
// dependent: launch as a programmatic dependent of the previous kernel (its
// set-up overlaps that kernel; every thread waits for it before touching the
// cache or the outputs) -- after the step's KV write, or when the caller says
// the tables and lengths were final before the previous kernel began.
int launch_query_major_tc(const pa_decode_params* p, void* stream, float* part_ml, float* part_o,
                          bool dependent);
// Its device error word shares the tensor-core decode's.
int read_and_clear_query_major_errors(uint32_t* flags);

}  // namespace pa
