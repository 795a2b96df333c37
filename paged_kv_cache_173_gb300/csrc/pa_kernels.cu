// pa_kernels.cu -- the cache write (reshape_and_cache) and the dispatch of
// the decode kernels by element type.
//
//  reshape_and_cache_kernel   scatter new tokens' K/V rows into their slots
//                             ("vLLM PagedAttention source walk-through",
//                             section 3.2: append_token writes the token's KV
//                             at block_table[pos / B], offset pos % B)
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_launch.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {

namespace {

// ============================================================ reshape_and_cache
struct ReshapeParams {
  const uint4* key;
  const uint4* value;
  uint4* k_cache;
  uint4* v_cache;
  const int64_t* slot_mapping;
  int64_t num_slots;  // num_blocks * block_size
  int num_tokens;
  int num_kv_heads;
  int row_vecs;  // head_dim * 2 / 16
};

// One warp per (token, KV head): lanes 0-15 copy the K row, lanes 16-31 the V
// row, 16 bytes per lane per step.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const __grid_constant__ ReshapeParams p) {
  grid_dependency_wait();     // inputs may come from the previous kernel on the stream
  allow_dependent_launch();   // the decode may start its prologue; it waits for this grid
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.num_tokens * p.num_kv_heads) return;
  const int t = wid / p.num_kv_heads;
  const int h = wid - t * p.num_kv_heads;
  const int64_t slot = __ldg(p.slot_mapping + t);
  if (slot < 0 || slot >= p.num_slots) return;  // padding, or out of the pool
  const bool is_v = lane >= 16;
  const uint4* src = (is_v ? p.value : p.key) + (static_cast<int64_t>(t) * p.num_kv_heads + h) * p.row_vecs;
  uint4* dst = (is_v ? p.v_cache : p.k_cache) + (slot * p.num_kv_heads + h) * p.row_vecs;
  for (int i = lane & 15; i < p.row_vecs; i += 16) dst[i] = __ldg(src + i);
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  ReshapeParams p;
  p.key = static_cast<const uint4*>(a.key);
  p.value = static_cast<const uint4*>(a.value);
  p.k_cache = static_cast<uint4*>(a.k_cache);
  p.v_cache = static_cast<uint4*>(a.v_cache);
  p.slot_mapping = a.slot_mapping;
  p.num_slots = static_cast<int64_t>(a.num_blocks) * a.block_size;
  p.num_tokens = a.num_tokens;
  p.num_kv_heads = a.num_kv_heads;
  p.row_vecs = a.head_dim * 2 / 16;
  const int64_t warps = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads;
  const int blocks = static_cast<int>((warps + 7) / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? launch_decode_bf16(a, stream) : launch_decode_f16(a, stream);
}

cudaError_t launch_splitk_reduce(const ReduceArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? launch_splitk_reduce_bf16(a, stream) : launch_splitk_reduce_f16(a, stream);
}

}  // namespace pa
