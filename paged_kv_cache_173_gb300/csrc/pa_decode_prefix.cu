// pa_decode_prefix.cu -- shared-prefix split-K decode: the shared pass over
// each group's common prompt blocks, then the per-sequence pass over the
// rest, for every query / cache type.
#include "pa_decode.cuh"
#include "pagedattn.h"

namespace pa {

cudaError_t launch_decode_prefix(const DecodeArgs& a, cudaStream_t stream) {
  if (a.kv_dtype == PA_FP8_E4M3) return launch_decode_prefix_typed<__half, E4M3>(a, stream);
  if (a.dtype == PA_BF16) return launch_decode_prefix_typed<__nv_bfloat16>(a, stream);
  return launch_decode_prefix_typed<__half>(a, stream);
}

}  // namespace pa
