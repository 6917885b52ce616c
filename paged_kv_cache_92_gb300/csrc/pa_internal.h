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

constexpr int kBlockSize = 16;
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
};

// Query heads padded to the tensor-core N (16, 32 or 64).
inline int tc_n_pad(int num_q_heads) {
  return num_q_heads <= 16 ? 16 : (num_q_heads <= 32 ? 32 : 64);
}

// Bytes at the start of every decode workspace (reserved).
constexpr size_t kWorkspaceHeaderBytes = 256;

// Workspace carve-up. Both kernels start after the header; a call uses one.
struct WorkspaceLayout {
  size_t total;
  size_t simt_m, simt_l, simt_acc;    // [seqs][q heads][partitions](+[dim])
  size_t tc_plan, tc_m, tc_l, tc_acc; // plan, then [seqs + grid][q heads](+[dim])
  size_t tc_q8, tc_qa;                // 8-bit cache: split queries, their 1/alpha
};
WorkspaceLayout decode_workspace_layout(const pa_decode_params* p, int num_partitions,
                                        int tc_grid);

// Tensor-core kernel: shapes it handles, and its grid (SM count of the current
// device, or 0 if that cannot be queried).
bool tc_supports(const pa_decode_params* p);
int tc_grid();

// Kernel launchers (pa_decode.cu / pa_cache.cu). Return a cudaError_t as int.
int launch_decode(const DecodeLaunch& L, void* stream);      // CUDA-core decode kernel
int launch_decode_tc(const DecodeLaunch& L, void* stream);   // tensor-core decode kernel
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
};
int launch_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                             int32_t head_dim, int32_t num_blocks, void* stream,
                             const AppendCheck& check = AppendCheck());
// 8-bit cache (pa_fp8.cu)
int launch_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, const float* k_scale,
                                 const float* v_scale, int32_t num_tokens, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t num_blocks, void* stream);
int launch_quantize_q(const void* q, void* q8, float* inv_alpha, int32_t num_seqs,
                      int32_t num_q_heads, int32_t n_pad, int32_t head_dim, void* stream);
int read_and_clear_fp8_errors(uint32_t* flags);
int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                       int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, void* stream);

// Device error words, one per kernel translation unit: read and clear.
int read_and_clear_decode_errors(uint32_t* flags);
int read_and_clear_decode_tc_errors(uint32_t* flags);

// Size of the library-owned device scratch used by pa_decode_noalloc.
constexpr size_t kNoAllocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
// Device address of that scratch on the current device (looked up on first use).
int decode_scratch_address(void** addr);
int read_and_clear_cache_errors(uint32_t* flags);

}  // namespace pa
