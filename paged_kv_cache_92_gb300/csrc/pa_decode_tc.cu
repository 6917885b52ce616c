// Tensor-core paged decode: the bf16 head_dim 128 block-size-16 instances and
// the entry points shared by all instances (shape rules, grid, dispatch by
// block size and cache type, error words). The kernels themselves are in
// pa_decode_tc.cuh.
#include "pa_decode_tc.cuh"

namespace pa {

bool tc_supports(const pa_decode_params* p) {
  const int H = p->num_kv_heads;
  const int G = p->num_q_heads / H;
  if (!(H == 1 || H == 2 || H == 4 || H == 8) || !(G == 1 || G == 2 || G == 4 || G == 8))
    return false;
  const bool fp8 = p->kv_dtype == PA_KV_FP8_E4M3;
  if (fp8 && p->head_dim != 128) return false;  // (the CUDA-core kernel takes head_dim 64)
  if (p->block_size != 16) {  // block sizes 8 and 32: bf16 head_dim 64 or 128, the
                              // 8-bit cache at 32 only (head_dim 128)
    if ((p->head_dim != 128 && p->head_dim != 64) || (p->block_size == 8 && fp8)) return false;
  }
  // column groups within the column budget (always, for these shapes), and
  // every virtual sequence (sequence x column group) in the kernel's plan
  return tc_max_group_tokens(p) >= 1 && tc_group_cols(p) <= kMaxGE &&
         tc_cols(p) <= (fp8 ? 64 : 128) && tc_virtual_seqs(p) <= kTcMaxSeqs;
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
  const pa_decode_params* p = Lc.p;
  const bool fp8 = p->kv_dtype == PA_KV_FP8_E4M3;
  switch (p->block_size) {
    case 8:
      if (fp8) return int(cudaErrorInvalidValue);
      return p->head_dim == 128 ? launch_decode_tc_bs8(Lc, s)
                                : (p->head_dim == 64 ? launch_decode_tc_bs8_d64(Lc, s)
                                                     : int(cudaErrorInvalidValue));
    case 32:
      if (fp8) return p->head_dim == 128 ? launch_decode_tc_bs32_fp8(Lc, s)
                                         : int(cudaErrorInvalidValue);
      return p->head_dim == 128 ? launch_decode_tc_bs32(Lc, s)
                                : (p->head_dim == 64 ? launch_decode_tc_bs32_d64(Lc, s)
                                                     : int(cudaErrorInvalidValue));
    case 16:
      if (fp8)
        return p->head_dim == 128 ? launch_decode_tc_fp8(Lc, s) : int(cudaErrorInvalidValue);
      switch (p->head_dim) {
        case 64: return launch_decode_tc_d64(Lc, s);
        case 128: return dispatch_tc<128, false, 16>(Lc, s);
        default: return int(cudaErrorInvalidValue);
      }
    default: return int(cudaErrorInvalidValue);
  }
}

int read_and_clear_decode_tc_errors(uint32_t* flags) {
  uint32_t f[8] = {};
  int r = read_and_clear_tc_error_word(&f[0]);
  if (r == 0) r = read_and_clear_decode_tc_d64_errors(&f[1]);
  if (r == 0) r = read_and_clear_decode_tc_fp8_errors(&f[2]);
  if (r == 0) r = read_and_clear_decode_tc_bs8_errors(&f[3]);
  if (r == 0) r = read_and_clear_decode_tc_bs32_errors(&f[4]);
  if (r == 0) r = read_and_clear_decode_tc_bs32_fp8_errors(&f[5]);
  if (r == 0) r = read_and_clear_decode_tc_bs8_d64_errors(&f[6]);
  if (r == 0) r = read_and_clear_decode_tc_bs32_d64_errors(&f[7]);
  *flags = f[0] | f[1] | f[2] | f[3] | f[4] | f[5] | f[6] | f[7];
  return r;
}

}  // namespace pa
