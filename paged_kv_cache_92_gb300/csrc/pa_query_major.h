// Launch rules of the query-major tensor-core kernel (pa_prefill_tc.cu), the
// path for many new tokens per sequence. Not part of the public ABI.
#pragma once

#include "pa_internal.h"

namespace pa {

// A unit of work is (sequence, group of KV heads, tile of 128 query rows =
// tokens x G heads of each head in the group); one persistent CTA per SM takes
// its share of them.
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
// It takes the bf16 cache at head_dim 128 and block size 16 when a KV head has
// at least 16 query rows (new tokens x G) or the column-group decode would
// split the new tokens into several groups (each re-reading the keys), and
// the batch gives it at least 128 (sequence, KV head, tile) units of work.
inline bool use_query_major(const pa_decode_params* p) {
  const int g = p->num_q_heads / p->num_kv_heads;
  return p->variant == PA_DECODE_TENSOR_CORE && p->kv_dtype == PA_KV_BF16 && p->head_dim == 128 &&
         p->block_size == 16 && query_len_of(p) > 1 && (g == 1 || g == 2 || g == 4 || g == 8) &&
         (tc_n_groups(p) > 1 || query_len_of(p) * g >= 16) &&
         int64_t(p->num_seqs) * p->num_kv_heads * query_major_tiles(p) >= 128;
}

int launch_query_major_tc(const pa_decode_params* p, void* stream);
// Its device error word shares the tensor-core decode's.
int read_and_clear_query_major_errors(uint32_t* flags);

}  // namespace pa
