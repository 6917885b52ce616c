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

// Resolved decode launch parameters (host validated).
struct DecodeLaunch {
  const pa_decode_params* p;
  int partition_tokens;
  int num_partitions;  // max over sequences, from max_context_len
  float* part_m;       // [num_seqs][num_q_heads][num_partitions]
  float* part_l;       // same
  float* part_acc;     // [num_seqs][num_q_heads][num_partitions][head_dim]
  unsigned int* counters;  // work counter of the tensor-core kernel (zero at launch)
};

// Bytes at the start of every decode workspace holding the work counter.
constexpr size_t kWorkspaceHeaderBytes = 256;

// Workspace carve-up: counter header, then split-K partials. Returns total bytes.
size_t decode_workspace_layout(const pa_decode_params* p, int num_partitions, size_t* off_m,
                               size_t* off_l, size_t* off_acc);

// Kernel launchers (pa_decode.cu / pa_cache.cu). Return a cudaError_t as int.
int launch_decode(const DecodeLaunch& L, void* stream);      // CUDA-core decode kernel
int launch_decode_tc(const DecodeLaunch& L, void* stream);   // tensor-core decode kernel
int launch_merge(const DecodeLaunch& L, void* stream);       // split-K merge (if needed)
int launch_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                             int32_t head_dim, int32_t num_blocks, void* stream);
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
