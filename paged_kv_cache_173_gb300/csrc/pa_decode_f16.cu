// pa_decode_f16.cu -- the decode and reduce kernels for __half caches.
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_f16(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_typed<__half>(a, stream);
}

cudaError_t launch_splitk_reduce_f16(const ReduceArgs& a, cudaStream_t stream) {
  return launch_splitk_reduce_typed<__half>(a, stream);
}

}  // namespace pa
