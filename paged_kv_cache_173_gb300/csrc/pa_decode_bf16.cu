// pa_decode_bf16.cu -- the decode and reduce kernels for __nv_bfloat16 caches.
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_typed<__nv_bfloat16>(a, stream);
}

cudaError_t launch_splitk_reduce_bf16(const ReduceArgs& a, cudaStream_t stream) {
  return launch_splitk_reduce_typed<__nv_bfloat16>(a, stream);
}

}  // namespace pa
