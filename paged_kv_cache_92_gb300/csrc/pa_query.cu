// Query preparation for the tensor-core decode: the rows of q placed in the
// kernel's column order (grouped by KV head, then query token, then query
// head within the group), as bf16 or split into two E4M3 terms for the 8-bit
// cache. Columns that hold no query (padding, or a token index past the
// sequence's new tokens) are zero.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Row of q ([B][query_len][Hq][D]) that column n of sequence b holds, or -1.
__device__ __forceinline__ int64_t source_row(const QueryMap& m, int b, int n) {
  if (n >= m.num_cols) return -1;
  const int g = n / m.group_cols, r = n - g * m.group_cols;
  const int i = r >> m.g_log2, j = r & ((1 << m.g_log2) - 1);
  if (i >= m.query_len) return -1;
  return (int64_t(b) * m.query_len + i) * m.num_q_heads + (g << m.g_log2) + j;
}

// One warp per (sequence, column): a row of head_dim bf16 values.
__global__ void __launch_bounds__(128)
    permute_q_kernel(const uint4* __restrict__ q, uint4* __restrict__ qp, const QueryMap m) {
  dev::griddep_launch_dependents();
  dev::griddep_wait();  // q may come from the previous kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * 4 + warp;
  if (gw >= int64_t(m.num_seqs) * m.n_pad) return;
  const int b = int(gw / m.n_pad), n = int(gw % m.n_pad);
  const int cpr = m.head_dim / 8;  // 16-byte chunks per row
  if (lane >= cpr) return;
  const int64_t src = source_row(m, b, n);
  qp[gw * cpr + lane] = src >= 0 ? q[src * cpr + lane] : make_uint4(0u, 0u, 0u, 0u);
}

// Queries for the E4M3 tensor-core decode. For every (sequence b, column n)
// the row is scaled by a power of two alpha (its largest magnitude lands in
// [64, 128)), split into hi = E4M3(q * alpha) and lo = E4M3(q * alpha - hi),
// which together carry about 8 significant bits (the scores use hi + lo), and
// 1/alpha is kept for the softmax. Output rows: q8[b][n] = hi, q8[b][N + n] =
// lo; inv_alpha[b][n] (zero rows and 1 for columns without a query). One warp
// per (b, n).
__global__ void __launch_bounds__(128)
    quantize_q_kernel(const __nv_bfloat16* __restrict__ q, uint8_t* __restrict__ q8,
                      float* __restrict__ inv_alpha, const QueryMap m) {
  dev::griddep_launch_dependents();
  dev::griddep_wait();  // q may come from the previous kernel
  const int N = m.n_pad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * 4 + warp;
  if (gw >= int64_t(m.num_seqs) * N) return;
  const int b = int(gw / N), n = int(gw % N);
  const int per = m.head_dim / 32;  // elements per lane (4 at head_dim 128)
  uint8_t* hi_row = q8 + (int64_t(b) * 2 * N + n) * m.head_dim;
  uint8_t* lo_row = q8 + (int64_t(b) * 2 * N + N + n) * m.head_dim;
  const int64_t src_row = source_row(m, b, n);
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

// One warp per (sequence, column), launched as a programmatic dependent of
// the previous kernel on the stream (each kernel waits before reading q).
template <typename K, typename... A>
int launch_rows(K kernel, const QueryMap& m, void* stream, A... args) {
  const int64_t warps = int64_t(m.num_seqs) * m.n_pad;
  if (warps == 0) return int(cudaSuccess);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((warps + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, kernel, args..., m));
}

}  // namespace

int launch_permute_q(const void* q, void* qp, const QueryMap& m, void* stream) {
  if (m.head_dim % 8 != 0 || m.head_dim > 256) return int(cudaErrorInvalidValue);
  return launch_rows(permute_q_kernel, m, stream, static_cast<const uint4*>(q),
                     static_cast<uint4*>(qp));
}

int launch_quantize_q(const void* q, void* q8, float* inv_alpha, const QueryMap& m,
                      void* stream) {
  if (m.head_dim != 128) return int(cudaErrorInvalidValue);
  return launch_rows(quantize_q_kernel, m, stream, static_cast<const __nv_bfloat16*>(q),
                     static_cast<uint8_t*>(q8), inv_alpha);
}

}  // namespace pa
