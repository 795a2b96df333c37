// pa_prefill.cu -- the paged prefill kernels for __half and __nv_bfloat16.
#include "pa_prefill.cuh"
#include "pagedattn.h"

namespace pa {

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? launch_prefill_typed<__nv_bfloat16>(a, stream)
                            : launch_prefill_typed<__half>(a, stream);
}

}  // namespace pa
