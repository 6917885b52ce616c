// Tensor-core paged decode: the bf16 head_dim 64, block size 32 instances
// (kernels in pa_decode_tc.cuh).
#include "pa_decode_tc.cuh"

namespace pa {

int launch_decode_tc_bs32_d64(const DecodeLaunch& Lc, void* stream) {
  return dispatch_tc<64, false, 32>(Lc, static_cast<cudaStream_t>(stream));
}

int read_and_clear_decode_tc_bs32_d64_errors(uint32_t* flags) {
  return read_and_clear_tc_error_word(flags);
}

}  // namespace pa
