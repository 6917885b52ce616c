// 8-bit (FP8 E4M3) KV cache support for sm_103a: the quantising KV write,
// and the decode's preparation launch (the split of the queries into two
// E4M3 terms, with the step's quantising KV write in the same launch).
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

#include <algorithm>
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
  const int W = BS < 16 ? BS : 16;  // keys of one V^T sub-tile
  const int64_t sub = tile + int64_t(off / W) * W * head_dim + (off % W);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    v_cache[sub + int64_t(c * 8 + i) * W] = to_e4m3(__fdiv_rn(__bfloat162float(vb[i]), vs));
}

// Queries for the E4M3 tensor-core decode. For every (sequence b, column n)
// the row is scaled by a power of two alpha (its largest magnitude lands in
// [64, 128)), split into hi = E4M3(q * alpha) and lo = E4M3(q * alpha - hi),
// which together carry about 8 significant bits (the scores use hi + lo), and
// 1/alpha is kept for the softmax. Output rows: q8[b][n] = hi, q8[b][N + n] =
// lo; inv_alpha[b][n] (zero rows and 1 for columns without a query). One warp
// per (b, n).
__device__ __forceinline__ void split_query_row(const __nv_bfloat16* __restrict__ q,
                                                uint8_t* __restrict__ q8,
                                                float* __restrict__ inv_alpha,
                                                const QueryMap& m, int64_t gw, int lane) {
  const int N = m.n_pad;
  if (gw >= int64_t(m.num_seqs) * N) return;
  const int b = int(gw / N), n = int(gw % N);
  const int per = m.head_dim / 32;  // elements per lane (4 at head_dim 128)
  uint8_t* hi_row = q8 + (int64_t(b) * 2 * N + n) * m.head_dim;
  uint8_t* lo_row = q8 + (int64_t(b) * 2 * N + N + n) * m.head_dim;
  const int64_t src_row = query_source_row(m, b, n);
  if (src_row < 0) {
    for (int i = 0; i < per; ++i) {
      hi_row[lane * per + i] = 0;
      lo_row[lane * per + i] = 0;
    }
    if (lane == 0) inv_alpha[int64_t(b) * N + n] = 1.0f;
    return;
  }
  const __nv_bfloat16* src = q + src_row * m.head_dim + lane * per;
  float v[4];
  float amax = 0.0f;
  for (int i = 0; i < per; ++i) {
    v[i] = __bfloat162float(src[i]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int e = 0;
  if (amax > 0.0f) (void)frexpf(amax, &e);  // amax < 2^e
  e = max(e, -100);
  const float alpha = ldexpf(1.0f, 7 - e);  // a power of two: exact
  for (int i = 0; i < per; ++i) {
    const float y = v[i] * alpha;
    const uint8_t h = dev::to_e4m3(y);
    hi_row[lane * per + i] = h;
    lo_row[lane * per + i] = dev::to_e4m3(y - dev::from_e4m3(h));
  }
  if (lane == 0) inv_alpha[int64_t(b) * N + n] = ldexpf(1.0f, e - 7);
}


// The step's new tokens for pa_append_decode on the 8-bit cache: token row
// t = b * q_len + i is position L_b - q_len + i of sequence b, and is written
// only at that position's slot (a negative slot: no write; an out-of-range
// slot: PA_DEVERR_SLOT; another slot: PA_DEVERR_APPEND_SLOT, no write).
struct Fp8Append {
  const uint4* k_new;
  const uint4* v_new;
  const int64_t* slot_mapping;
  uint8_t* k_cache;
  uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int64_t num_chunks;  // rows x (head_dim / 8); 0 = nothing to write
  int64_t num_slots;
  int num_kv_heads, head_dim, max_blocks_per_seq, cap, q_len, bs_log2;
  int early;  // lengths and tables final before the previous kernel began (overlap_prologue)
};

// One launch ahead of the 8-bit decode. The first blocks write the new
// tokens, one thread per 8 elements of a (token, KV head) row, dividing by
// the head's scale with a reciprocal and Markstein's correction step (the
// same codes as the division); the last q_blocks split the queries (one warp
// per (sequence, column)). The write blocks go first because they wait on
// two memory round trips (the table entry needs the length): dispatched after
// the split blocks, they ended the launch later, and the decode waits for its
// end (measured on the 64-sequence 8B layer: 45.9 against 42.0 us per step).
__global__ void __launch_bounds__(128)
    prep_fp8_kernel(const __nv_bfloat16* __restrict__ q, uint8_t* __restrict__ q8,
                    float* __restrict__ inv_alpha, const QueryMap m, int q_blocks,
                    const Fp8Append a) {
  dev::griddep_launch_dependents();
  const int w_blocks = int(gridDim.x) - q_blocks;
  if (int(blockIdx.x) >= w_blocks) {
    dev::griddep_wait();  // q may come from the previous kernel
    split_query_row(q, q8, inv_alpha, m,
                    int64_t(blockIdx.x - w_blocks) * 4 + (threadIdx.x >> 5), threadIdx.x & 31);
    return;
  }
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= a.num_chunks) return;
  const int BS = 1 << a.bs_log2;
  const int cpr = a.head_dim / 8;
  const int c = int(idx % cpr);
  const int64_t row = idx / cpr;  // t * num_kv_heads + h
  const int h = int(row % a.num_kv_heads);
  const int64_t t = row / a.num_kv_heads;
  const int b = int(t / a.q_len), i = int(t % a.q_len);
  // The token's position (from its sequence's length) and that position's
  // table entry: two dependent loads. When the lengths and tables were final
  // before the previous kernel began they are taken before waiting for it,
  // and only the loads of this step's inputs remain after the wait (one
  // round trip on the decode's critical path instead of two).
  int L = 0, e = -1;
  auto locate = [&]() {
    L = min(a.context_lens[b], a.cap);
    if (L >= a.q_len)
      e = a.block_tables[int64_t(b) * a.max_blocks_per_seq + ((L - a.q_len + i) >> a.bs_log2)];
  };
  if (a.early) locate();
  dev::griddep_wait();  // the slots and the new rows may come from the previous kernel
  if (!a.early) locate();
  const int64_t slot = a.slot_mapping[t];
  const uint4 kr = a.k_new[idx], vr = a.v_new[idx];
  const float ks = a.k_scale[h], vs = a.v_scale[h];
  if (slot < 0) return;  // padding token: no write
  if (slot >= a.num_slots) {
    if (h == 0 && c == 0) atomicOr(&g_fp8_errors, PA_DEVERR_SLOT);
    return;
  }
  if (L < a.q_len) return;  // no room for the new tokens: the decode flags the length
  const int pos = L - a.q_len + i;
  if (e < 0 || slot != int64_t(e) * BS + (pos & (BS - 1))) {
    if (h == 0 && c == 0) atomicOr(&g_fp8_errors, PA_DEVERR_APPEND_SLOT);
    return;
  }
  const float rk = __frcp_rn(ks), rv = __frcp_rn(vs);
  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kr);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vr);
  uint32_t kw[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j)
    kw[j >> 2] |= uint32_t(to_e4m3(dev::div_rn_by(__bfloat162float(kb[j]), ks, rk)))
                  << (8 * (j & 3));
  const int off = pos & (BS - 1);
  const int64_t tile = (int64_t(e) * a.num_kv_heads + h) * int64_t(BS) * a.head_dim;
  *reinterpret_cast<uint2*>(a.k_cache + tile + int64_t(off) * a.head_dim + c * 8) =
      make_uint2(kw[0], kw[1]);
  const int W = BS < 16 ? BS : 16;  // keys of one V^T sub-tile
  const int64_t sub = tile + int64_t(off / W) * W * a.head_dim + (off % W);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    a.v_cache[sub + int64_t(c * 8 + j) * W] =
        to_e4m3(dev::div_rn_by(__bfloat162float(vb[j]), vs, rv));
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

int launch_quantize_q(const void* q, void* q8, float* inv_alpha, const QueryMap& m,
                      const pa_decode_params* p, const pa_append_params* ap, void* stream) {
  if (q != nullptr && m.head_dim != 128) return int(cudaErrorInvalidValue);
  Fp8Append a = {};
  if (ap) {
    a.k_new = static_cast<const uint4*>(ap->k_new);
    a.v_new = static_cast<const uint4*>(ap->v_new);
    a.slot_mapping = ap->slot_mapping;
    a.k_cache = static_cast<uint8_t*>(ap->k_cache);
    a.v_cache = static_cast<uint8_t*>(ap->v_cache);
    a.k_scale = p->k_scale;
    a.v_scale = p->v_scale;
    a.block_tables = p->block_tables;
    a.context_lens = p->context_lens;
    a.num_kv_heads = p->num_kv_heads;
    a.head_dim = p->head_dim;
    a.max_blocks_per_seq = p->max_blocks_per_seq;
    a.cap = std::min(p->max_blocks_per_seq * p->block_size, p->max_context_len);
    a.q_len = m.query_len;
    a.bs_log2 = log2_of(p->block_size);
    a.num_slots = int64_t(p->num_blocks) * p->block_size;
    a.num_chunks = int64_t(m.num_real_seqs) * m.query_len * p->num_kv_heads * (p->head_dim / 8);
    a.early = p->overlap_prologue ? 1 : 0;
  }
  const int64_t q_blocks = q != nullptr ? (int64_t(m.num_seqs) * m.n_pad + 3) / 4 : 0;
  const int64_t w_blocks = (a.num_chunks + 127) / 128;
  if (q_blocks + w_blocks == 0) return int(cudaSuccess);
  // a programmatic dependent of the previous kernel on the stream (it waits
  // before it reads q or the new rows)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(q_blocks + w_blocks));
  cfg.blockDim = dim3(128);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, prep_fp8_kernel, static_cast<const __nv_bfloat16*>(q),
                                static_cast<uint8_t*>(q8), inv_alpha, m, int(q_blocks), a));
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
