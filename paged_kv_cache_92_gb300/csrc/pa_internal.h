// Internal declarations shared by the host-side translation units of
// libpagedkv.so. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/pagedkv.h"

namespace pa {

// Record a thread-local error message and return `s` (for PA_OK the message is untouched).
pa_status set_error(pa_status s, const char* msg);
pa_status set_cuda_error(const char* where, int cuda_err);

constexpr int kBlockSize = 16;  // the CUDA-core decode's block size
// Block sizes the cache kernels and the tensor-core decode take.
inline bool block_size_ok(int bs) { return bs == 8 || bs == 16 || bs == 32; }
constexpr int kDefaultPartitionTokens = 512;
constexpr int kMaxPartitionTokens = 4096;
// The tensor-core decode kernel plans its stream-K split in shared memory
// (one int per sequence); larger batches run on the CUDA-core kernel.
constexpr int kTcMaxSeqs = 16384;

// Resolved decode launch parameters (host validated).
struct DecodeLaunch {
  const pa_decode_params* p;
  int partition_tokens;  // CUDA-core kernel: split-K partition length
  int num_partitions;    // CUDA-core kernel: max partitions over sequences
  int grid;              // tensor-core kernel: persistent CTAs (one per SM)
  float* part_m;         // partial maxima (layout depends on the kernel)
  float* part_l;         // partial sums
  float* part_acc;       // partial weighted sums
  int* plan;             // tensor-core kernel: stream-K plan for its merge
  const pa_append_params* append;  // non-null: write each sequence's new token first
  unsigned char* q8;     // 8-bit cache: split queries [B][2N][D] (workspace)
  float* q_inv_alpha;    // 8-bit cache: [B][N] (workspace)
  void* qp;              // bf16, query_len > 1: queries in column order [B][N][D] (workspace)
};

// New tokens per sequence (query_len 0 means 1).
inline int query_len_of(const pa_decode_params* p) {
  return p->query_len > 1 ? p->query_len : 1;
}

// Tensor-core column layout. The kernel's query rows ("columns": the N side
// of its MMAs) are grouped by KV head: head g owns columns [g*GE, (g+1)*GE),
// column g*GE + i*G + j being query token i of query head g*G + j. GE is G
// times the tokens of a column group rounded up to a power of two; columns
// whose token index is past the group's tokens are unused. With one token per
// sequence GE = G and the column of query head h is h itself.
//
// A column group holds at most tc_max_group_tokens() query tokens: GE <= 16
// (8 at block size 8) and num_kv_heads * GE <= 128 (64 for the 8-bit cache).
// A sequence with more new tokens is split into n_groups groups of that many
// (the last one possibly shorter), each decoded as a virtual sequence of its
// own that streams the keys its last token can see.
inline int pow2_ceil(int x) {
  int q = 1;
  while (q < x) q <<= 1;
  return q;
}
inline int tc_max_group_tokens(const pa_decode_params* p) {
  const int g = p->num_q_heads / p->num_kv_heads;
  int cols = p->block_size == 8 ? 8 : 16;  // columns per KV head
  const int total = p->kv_dtype == PA_KV_FP8_E4M3 ? 64 : 128;
  if (cols * p->num_kv_heads > total) cols = total / p->num_kv_heads;
  return cols >= g ? cols / g : 0;
}
inline int tc_q_group(const pa_decode_params* p) {
  const int q = query_len_of(p), cap = tc_max_group_tokens(p);
  return q <= cap ? q : cap;
}
inline int tc_n_groups(const pa_decode_params* p) {
  const int qg = tc_q_group(p);
  return qg > 0 ? (query_len_of(p) + qg - 1) / qg : 0;
}
inline int tc_group_cols(const pa_decode_params* p) {
  return (p->num_q_heads / p->num_kv_heads) * pow2_ceil(tc_q_group(p));
}
inline int tc_cols(const pa_decode_params* p) { return p->num_kv_heads * tc_group_cols(p); }
// Virtual sequences of the tensor-core decode: num_seqs * n_groups.
inline int64_t tc_virtual_seqs(const pa_decode_params* p) {
  return int64_t(p->num_seqs) * tc_n_groups(p);
}

// Columns padded to the tensor-core N (16, 32, 64 or 128).
inline int tc_n_pad(int cols) {
  return cols <= 16 ? 16 : (cols <= 32 ? 32 : (cols <= 64 ? 64 : 128));
}

inline int log2_of(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

// Where the query rows of one virtual sequence sit in the column layout
// above. Virtual sequence v is column group v % n_groups (tokens
// [g * q_group, g * q_group + q_group) of query_len) of sequence v / n_groups.
struct QueryMap {
  int num_seqs;       // virtual sequences (sequences x n_groups)
  int num_real_seqs;  // sequences
  int num_q_heads, query_len, q_group, n_groups, g_log2, group_cols, num_cols, n_pad, head_dim;
};
inline QueryMap query_map(const pa_decode_params* p) {
  QueryMap m;
  m.num_real_seqs = p->num_seqs;
  m.n_groups = tc_n_groups(p);
  m.num_seqs = int(tc_virtual_seqs(p));
  m.num_q_heads = p->num_q_heads;
  m.query_len = query_len_of(p);
  m.q_group = tc_q_group(p);
  m.g_log2 = log2_of(p->num_q_heads / p->num_kv_heads);
  m.group_cols = tc_group_cols(p);
  m.num_cols = tc_cols(p);
  m.n_pad = tc_n_pad(m.num_cols);
  m.head_dim = p->head_dim;
  return m;
}
#ifdef __CUDACC__
// Row of q ([B][query_len][Hq][D]) that column n of virtual sequence v holds, or -1.
__device__ __forceinline__ int64_t query_source_row(const QueryMap& m, int v, int n) {
  if (n >= m.num_cols) return -1;
  const int b = v / m.n_groups, grp = v - b * m.n_groups;
  const int g = n / m.group_cols, r = n - g * m.group_cols;
  const int il = r >> m.g_log2, j = r & ((1 << m.g_log2) - 1);
  const int i = grp * m.q_group + il;
  if (il >= m.q_group || i >= m.query_len) return -1;
  return (int64_t(b) * m.query_len + i) * m.num_q_heads + (g << m.g_log2) + j;
}
#endif

// Bytes at the start of every decode workspace (reserved).
constexpr size_t kWorkspaceHeaderBytes = 256;

// Workspace carve-up of the kernel a call will run (decode_uses_tc: the
// tensor-core kernel; otherwise the CUDA-core one), after the header. The
// other kernel's fields are zero.
struct WorkspaceLayout {
  size_t total;
  size_t simt_m, simt_l, simt_acc;    // [seqs][q heads][partitions](+[dim])
  size_t tc_plan, tc_m, tc_l, tc_acc; // plan, then [seqs + grid][q heads](+[dim])
  size_t tc_q8, tc_qa;                // 8-bit cache: split queries, their 1/alpha
  size_t tc_qp;                       // bf16, query_len > 1: queries in column order
};
WorkspaceLayout decode_workspace_layout(const pa_decode_params* p, int num_partitions,
                                        int tc_grid);

// Tensor-core kernel: shapes it handles, and its grid (SM count of the current
// device, or 0 if that cannot be queried).
bool tc_supports(const pa_decode_params* p);
int tc_grid();
// The decode runs on the tensor-core kernel: variant PA_DECODE_TENSOR_CORE and
// a shape it handles (else the CUDA-core kernel runs).
bool decode_uses_tc(const pa_decode_params* p);

// Kernel launchers (pa_decode.cu / pa_cache.cu). Return a cudaError_t as int.
int launch_decode(const DecodeLaunch& L, void* stream);      // CUDA-core decode kernel
int launch_decode_tc(const DecodeLaunch& L, void* stream);   // tensor-core decode kernel
// its shares by translation unit: bf16 head_dim 64; the 8-bit cache; block
// size 8; block size 32 (bf16, 8-bit); block sizes 8 and 32 at head_dim 64
int launch_decode_tc_d64(const DecodeLaunch& L, void* stream);
int launch_decode_tc_fp8(const DecodeLaunch& L, void* stream);
int launch_decode_tc_bs8(const DecodeLaunch& L, void* stream);
int launch_decode_tc_bs32(const DecodeLaunch& L, void* stream);
int launch_decode_tc_bs32_fp8(const DecodeLaunch& L, void* stream);
int launch_decode_tc_bs8_d64(const DecodeLaunch& L, void* stream);   // bf16 head_dim 64
int launch_decode_tc_bs32_d64(const DecodeLaunch& L, void* stream);
int launch_merge(const DecodeLaunch& L, void* stream);       // split-K merge (if needed)
// Decode-step check (block_tables non-null): token t is sequence t's newest
// token; it is written only if slot_mapping[t] is the slot of token
// min(context_lens[t], cap) - 1 of sequence t (else PA_DEVERR_APPEND_SLOT),
// and not at all for an empty sequence.
struct AppendCheck {
  const int32_t* block_tables = nullptr;
  const int32_t* context_lens = nullptr;
  int max_blocks_per_seq = 0;
  int cap = 0;
  int q_len = 1;  // new tokens per sequence: token row t is token t % q_len of sequence t / q_len
};
int launch_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, int32_t num_blocks, void* stream,
                             const AppendCheck& check = AppendCheck());
// 8-bit cache (pa_fp8.cu)
int launch_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, const float* k_scale,
                                 const float* v_scale, int32_t num_tokens, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                 void* stream);
int read_and_clear_fp8_errors(uint32_t* flags);
// Query preparation for the bf16 tensor-core decode with several new tokens
// per sequence (pa_query.cu): the rows of q ([B][query_len][Hq][D] bf16) in
// the column layout, padded to n_pad rows with zeros ([B][n_pad][D]).
int launch_permute_q(const void* q, void* qp, const QueryMap& m, void* stream);
// The 8-bit decode's preparation launch (pa_fp8.cu): the rows of q split into
// two E4M3 terms in the column layout ([B][2*n_pad][D] bytes, hi rows then lo
// rows, and [B][n_pad] floats 1/alpha), and -- with `append` (pa_append_decode)
// -- the quantising KV write of the step's new tokens, checked against their
// positions like the fused bf16 write. With q == nullptr only the write runs
// (the CUDA-core decode of the 8-bit cache).
int launch_quantize_q(const void* q, void* q8, float* inv_alpha, const QueryMap& m,
                      const pa_decode_params* p, const pa_append_params* append, void* stream);
// Copy `bytes` from src -- host memory the GPU can address (pinned, mapped
// under unified addressing), 16-byte aligned -- to device memory dst (16-byte
// aligned), with a kernel rather than a DMA copy (pa_cache.cu).
int launch_stage_in(const void* src, void* dst, size_t bytes, void* stream);
int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int32_t num_blocks, void* stream);

// Device error words, one per kernel translation unit: read and clear.
int read_and_clear_decode_errors(uint32_t* flags);
int read_and_clear_decode_tc_errors(uint32_t* flags);  // all three shares below
int read_and_clear_decode_tc_d64_errors(uint32_t* flags);
int read_and_clear_decode_tc_fp8_errors(uint32_t* flags);
int read_and_clear_decode_tc_bs8_errors(uint32_t* flags);
int read_and_clear_decode_tc_bs32_errors(uint32_t* flags);
int read_and_clear_decode_tc_bs32_fp8_errors(uint32_t* flags);
int read_and_clear_decode_tc_bs8_d64_errors(uint32_t* flags);
int read_and_clear_decode_tc_bs32_d64_errors(uint32_t* flags);

// Size of the library-owned device scratch used by pa_decode_noalloc.
constexpr size_t kNoAllocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
// Device address of that scratch on the current device (looked up on first use).
int decode_scratch_address(void** addr);
int read_and_clear_cache_errors(uint32_t* flags);

}  // namespace pa
