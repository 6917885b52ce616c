// Tensor-core paged decode: the bf16 head_dim 128 instances and the entry
// points shared by all instances (shape rules, grid, dispatch, error words).
// The kernels themselves are in pa_decode_tc.cuh.
#include "pa_decode_tc.cuh"

namespace pa {

bool tc_supports(const pa_decode_params* p) {
  const int H = p->num_kv_heads;
  const int G = p->num_q_heads / H;
  if (!(H == 1 || H == 2 || H == 4 || H == 8) || !(G == 1 || G == 2 || G == 4 || G == 8) ||
      p->num_seqs > kTcMaxSeqs || query_len_of(p) > kMaxGE)
    return false;
  return tc_group_cols(p) <= kMaxGE &&
         tc_cols(p) <= (p->kv_dtype == PA_KV_FP8_E4M3 ? 64 : 128);
}

int tc_grid() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int launch_decode_tc(const DecodeLaunch& Lc, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Lc.p->kv_dtype == PA_KV_FP8_E4M3)
    return Lc.p->head_dim == 128 ? launch_decode_tc_fp8(Lc, s) : int(cudaErrorInvalidValue);
  switch (Lc.p->head_dim) {
    case 64: return launch_decode_tc_d64(Lc, s);
    case 128: return dispatch_tc<128, false>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

int read_and_clear_decode_tc_errors(uint32_t* flags) {
  uint32_t a = 0, b = 0, c = 0;
  int r = read_and_clear_tc_error_word(&a);
  if (r == 0) r = read_and_clear_decode_tc_d64_errors(&b);
  if (r == 0) r = read_and_clear_decode_tc_fp8_errors(&c);
  *flags = a | b | c;
  return r;
}

}  // namespace pa
