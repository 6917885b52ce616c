// Cache-writing kernels for sm_103a: the new token's K/V written through the
// slot mapping, and the whole-block copy of copy-on-write. Both are plain
// 16-byte vector copies (bit-exact); each thread moves one 16-byte chunk, so
// consecutive threads touch consecutive addresses on both sides.
//
// Sources: "How Paged Attention and Continuous Batching Actually Work",
// §One step, end to end (write KV through the slot-mapping formula);
// "Paged Attention as a Memory Manager", §Prefix Caching and Copy-on-Write
// (allocate a fresh block, copy the existing content). The block size is a
// power of two ("Paged Attention as a Memory Manager", §PagedAttention: 8, 16
// or 32 tokens); slots split into (block, offset) by shift and mask.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_cache_errors;

// One thread per 16-byte chunk of one (token, KV head) row, for K and V.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                             uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                             const int64_t* __restrict__ slot_mapping, int64_t num_chunks,
                             int num_kv_heads, int chunks_per_row, int64_t num_slots, int bs_log2,
                             AppendCheck check) {
  const int BS = 1 << bs_log2;
  // a decode launched as a programmatic dependent may start its set-up now;
  // it waits for this kernel before it reads the cache
  dev::griddep_launch_dependents();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= num_chunks) return;
  const int c = int(idx % chunks_per_row);
  const int64_t row = idx / chunks_per_row;  // t * num_kv_heads + h
  const int h = int(row % num_kv_heads);
  const int64_t t = row / num_kv_heads;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;  // padding token: no write
  if (slot >= num_slots) {
    atomicOr(&g_cache_errors, PA_DEVERR_SLOT);
    return;
  }
  if (check.block_tables) {
    // decode step: token t is new token i of sequence b, written only at its
    // position's slot (the last q_len tokens of the sequence)
    const int64_t b = t / check.q_len;
    const int i = int(t - b * check.q_len);
    const int L = min(check.context_lens[b], check.cap);
    if (L < check.q_len) return;  // no room for the new tokens: the decode flags the length
    const int pos = L - check.q_len + i;
    const int e = check.block_tables[b * check.max_blocks_per_seq + pos / BS];
    if (slot != int64_t(e) * BS + pos % BS) {
      if (h == 0 && c == 0) atomicOr(&g_cache_errors, PA_DEVERR_APPEND_SLOT);
      return;
    }
  }
  const int64_t blk = slot >> bs_log2;
  const int64_t off = slot & (BS - 1);
  const int64_t dst = ((blk * num_kv_heads + h) * BS + off) * chunks_per_row + c;
  k_cache[dst] = k_new[idx];
  v_cache[dst] = v_new[idx];
}

// grid = (chunk blocks, num_pairs, 2): z selects the K or V cache.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ pairs, int64_t block_chunks, int num_blocks) {
  const int pair = blockIdx.y;
  const int src = pairs[2 * pair];
  const int dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_cache_errors, PA_DEVERR_COPY_PAIR);
    return;
  }
  uint4* cache = blockIdx.z == 0 ? k_cache : v_cache;
  const uint4* s = cache + int64_t(src) * block_chunks;
  uint4* d = cache + int64_t(dst) * block_chunks;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < block_chunks;
       i += int64_t(gridDim.x) * blockDim.x)
    d[i] = s[i];
}

// A plain copy of n16 16-byte chunks (then `tail` bytes) from memory the GPU
// reads over the host link -- pinned host memory -- into device memory: the
// staging of a host-driven step's packed inputs. Each thread issues its two
// loads before its stores, so a warp has two link round trips in flight.
__global__ void __launch_bounds__(256)
    stage_in_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16,
                    int tail) {
  // a decode launched as a programmatic dependent may start its set-up now;
  // it waits for this kernel before it reads what this kernel writes
  dev::griddep_launch_dependents();
  const int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 2;
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
  if (i < n16) a = src[i];
  if (i + 1 < n16) b = src[i + 1];
  if (i < n16) dst[i] = a;
  if (i + 1 < n16) dst[i + 1] = b;
  if (i == 0)
    for (int t = 0; t < tail; ++t)
      reinterpret_cast<uint8_t*>(dst + n16)[t] = reinterpret_cast<const uint8_t*>(src + n16)[t];
}

}  // namespace

int launch_stage_in(const void* src, void* dst, size_t bytes, void* stream) {
  if (bytes == 0) return int(cudaSuccess);
  const int64_t n16 = int64_t(bytes / 16);
  const int tail = int(bytes % 16);
  const int threads = 256;
  const int64_t blocks = (n16 + 2 * threads - 1) / (2 * threads);
  stage_in_kernel<<<unsigned(blocks > 0 ? blocks : 1), threads, 0,
                    static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(src),
                                                         static_cast<uint4*>(dst), n16, tail);
  return int(cudaGetLastError());
}

int launch_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, int32_t num_blocks, void* stream,
                             const AppendCheck& check) {
  const int chunks_per_row = head_dim * 2 / 16;
  const int64_t num_chunks = int64_t(num_tokens) * num_kv_heads * chunks_per_row;
  if (num_chunks == 0) return int(cudaSuccess);
  const int threads = 256;
  const int64_t blocks = (num_chunks + threads - 1) / threads;
  reshape_and_cache_kernel<<<unsigned(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, num_chunks,
      num_kv_heads, chunks_per_row, int64_t(num_blocks) * block_size, log2_of(block_size), check);
  return int(cudaGetLastError());
}

int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int32_t num_blocks, void* stream) {
  if (num_pairs == 0) return int(cudaSuccess);
  const int64_t block_chunks = int64_t(num_kv_heads) * block_size * head_dim * 2 / 16;
  const int threads = 256;
  int64_t gx = (block_chunks + threads - 1) / threads;
  if (gx > 64) gx = 64;
  dim3 grid(unsigned(gx), unsigned(num_pairs), 2);
  copy_blocks_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, block_chunks, num_blocks);
  return int(cudaGetLastError());
}

int read_and_clear_cache_errors(uint32_t* flags) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_cache_errors, sizeof(v));
  if (e != cudaSuccess) return int(e);
  e = cudaMemcpyToSymbol(g_cache_errors, &zero, sizeof(zero));
  *flags = v;
  return int(e);
}

}  // namespace pa
