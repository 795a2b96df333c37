// pa_decode_fp8.cu -- the decode kernels for E4M3 caches with __half queries
// (split-K partials go through the float16 reduce of pa_decode_f16.cu).
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_f16_e4m3(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_typed<__half, E4M3>(a, stream);
}

}  // namespace pa
