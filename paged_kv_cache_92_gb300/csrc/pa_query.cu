// Query preparation for the bf16 tensor-core decode with several new tokens
// per sequence: the rows of q placed in the kernel's column order (grouped by
// KV head, then query token, then query head within the group). Columns that
// hold no query (padding, or a token index past the sequence's new tokens)
// are zero. (The 8-bit path's split queries are made in pa_fp8.cu.)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

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
  const int64_t src = query_source_row(m, b, n);
  qp[gw * cpr + lane] = src >= 0 ? q[src * cpr + lane] : make_uint4(0u, 0u, 0u, 0u);
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

}  // namespace pa
