// 8-bit (FP8 E4M3) KV cache support for sm_103a: the quantising KV write.
// (The split of the queries into two E4M3 terms is in pa_query.cu.)
//
// The pages say only that paging combines with 8-bit KV quantisation, which
// halves the bytes per block ("PagedAttention" glossary page, §What paging
// costs). The format is this library's reading:
//  - OCP E4M3 codes, one dequantisation scale per KV head for K and for V;
//  - write: code = E4M3(float32(x) / scale[h]), round to nearest even,
//    saturating to +-448 (the CUDA conversion intrinsic with satfinite);
//  - layout: K [block][head][offset][d] like the bf16 cache; V transposed
//    inside each (block, head) tile in sub-tiles of 16 keys,
//    [block][head][offset / 16][d][offset % 16] (one [d][16] sub-tile at block
//    size 16, two at 32), so that the value product reads V^T K-major (16
//    contiguous keys per row) on the tensor cores.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_fp8_errors;

using dev::to_e4m3;

// One thread per 8 elements (one 16-byte chunk of the bf16 input) of one
// (token, KV head) row, for K and V.
__global__ void __launch_bounds__(256)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                 uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                 const int64_t* __restrict__ slot_mapping,
                                 const float* __restrict__ k_scale,
                                 const float* __restrict__ v_scale, int64_t num_chunks,
                                 int num_kv_heads, int head_dim, int64_t num_slots, int bs_log2) {
  const int BS = 1 << bs_log2;
  dev::griddep_launch_dependents();
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= num_chunks) return;
  const int cpr = head_dim / 8;
  const int c = int(idx % cpr);
  const int64_t row = idx / cpr;  // t * num_kv_heads + h
  const int h = int(row % num_kv_heads);
  const int64_t t = row / num_kv_heads;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;  // padding token: no write
  if (slot >= num_slots) {
    if (h == 0 && c == 0) atomicOr(&g_fp8_errors, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot >> bs_log2;
  const int off = int(slot & (BS - 1));
  const float ks = k_scale[h], vs = v_scale[h];
  const uint4 kr = k_new[idx], vr = v_new[idx];
  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kr);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vr);
  uint8_t kq[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) kq[i] = to_e4m3(__fdiv_rn(__bfloat162float(kb[i]), ks));
  const int64_t tile = (blk * num_kv_heads + h) * int64_t(BS) * head_dim;
  // K row: 8 contiguous bytes
  uint2 kw;
  kw.x = uint32_t(kq[0]) | uint32_t(kq[1]) << 8 | uint32_t(kq[2]) << 16 | uint32_t(kq[3]) << 24;
  kw.y = uint32_t(kq[4]) | uint32_t(kq[5]) << 8 | uint32_t(kq[6]) << 16 | uint32_t(kq[7]) << 24;
  *reinterpret_cast<uint2*>(k_cache + tile + int64_t(off) * head_dim + c * 8) = kw;
  // V column: element d of the row goes to byte d * 16 + off % 16 of the
  // tile's sub-tile off / 16
  const int64_t sub = tile + int64_t(off >> 4) * 16 * head_dim + (off & 15);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    v_cache[sub + int64_t(c * 8 + i) * 16] = to_e4m3(__fdiv_rn(__bfloat162float(vb[i]), vs));
}

}  // namespace

int launch_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, const float* k_scale,
                                 const float* v_scale, int32_t num_tokens, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                 void* stream) {
  const int64_t num_chunks = int64_t(num_tokens) * num_kv_heads * (head_dim / 8);
  if (num_chunks == 0) return int(cudaSuccess);
  const int threads = 256;
  const int64_t blocks = (num_chunks + threads - 1) / threads;
  reshape_and_cache_fp8_kernel<<<unsigned(blocks), threads, 0,
                                 static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), slot_mapping, k_scale,
      v_scale, num_chunks, num_kv_heads, head_dim, int64_t(num_blocks) * block_size,
      log2_of(block_size));
  return int(cudaGetLastError());
}

int read_and_clear_fp8_errors(uint32_t* flags) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_fp8_errors, sizeof(v));
  if (e != cudaSuccess) return int(e);
  e = cudaMemcpyToSymbol(g_fp8_errors, &zero, sizeof(zero));
  *flags = v;
  return int(e);
}

}  // namespace pa
