// Tensor-core paged decode over the 8-bit (E4M3) cache: the head_dim 128
// instances (kernels in pa_decode_tc.cuh).
#include "pa_decode_tc.cuh"

namespace pa {

int launch_decode_tc_fp8(const DecodeLaunch& Lc, void* stream) {
  return dispatch_tc<128, true, 16>(Lc, static_cast<cudaStream_t>(stream));
}

int read_and_clear_decode_tc_fp8_errors(uint32_t* flags) {
  return read_and_clear_tc_error_word(flags);
}

}  // namespace pa
