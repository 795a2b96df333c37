// pa_kernels.cu -- the cache write (reshape_and_cache) and the dispatch of
// the decode kernels by element type.
//
//  reshape_and_cache_kernel   scatter new tokens' K/V rows into their slots
//                             ("vLLM PagedAttention source walk-through",
//                             section 3.2: append_token writes the token's KV
//                             at block_table[pos / B], offset pos % B)
//  reshape_and_cache_e4m3_kernel
//                             the same into E4M3 caches: each element is
//                             stored as the code nearest to x / scale ("when
//                             the KV cache meets OS paging", section 6:
//                             compression inside the block)
//  copy_blocks_kernel         whole-block copies, the copy step of
//                             copy-on-write
//  wait_selftest_kernel       one warp through the bounded mbarrier wait that
//                             every pipeline of the library uses: a wait on a
//                             phase nothing completes must give up after its
//                             limit, and a completed phase must be seen
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

// ======================================================= reshape_and_cache, E4M3
struct ReshapeE4m3Params {
  const uint4* key;  // 8 elements of 16 bits per vector
  const uint4* value;
  uint2* k_cache;    // 8 codes per vector
  uint2* v_cache;
  const int64_t* slot_mapping;
  int64_t num_slots;
  int num_tokens;
  int num_kv_heads;
  int row_vecs;  // head_dim / 8
  float k_scale;
  float v_scale;
};

// One warp per (token, KV head), lanes 0-15 on K and 16-31 on V: each lane
// turns 8 elements (16 bytes) into 8 codes (8 bytes) per step.  The quotient
// x / scale is rounded once to float32 (IEEE division), then to E4M3.
template <typename T>
__global__ void __launch_bounds__(256) reshape_and_cache_e4m3_kernel(const __grid_constant__ ReshapeE4m3Params p) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.num_tokens * p.num_kv_heads) return;
  const int t = wid / p.num_kv_heads;
  const int h = wid - t * p.num_kv_heads;
  const int64_t slot = __ldg(p.slot_mapping + t);
  if (slot < 0 || slot >= p.num_slots) return;  // padding, or out of the pool
  const bool is_v = lane >= 16;
  const float sc = is_v ? p.v_scale : p.k_scale;
  const uint4* src = (is_v ? p.value : p.key) + (static_cast<int64_t>(t) * p.num_kv_heads + h) * p.row_vecs;
  uint2* dst = (is_v ? p.v_cache : p.k_cache) + (slot * p.num_kv_heads + h) * p.row_vecs;
  for (int i = lane & 15; i < p.row_vecs; i += 16) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack2<T>(w[j]);
      const uint32_t c0 = float_to_e4m3_sat(__fdiv_rn(f.x, sc));
      const uint32_t c1 = float_to_e4m3_sat(__fdiv_rn(f.y, sc));
      o[j >> 1] |= (c0 | (c1 << 8)) << ((j & 1) * 16);
    }
    dst[i] = make_uint2(o[0], o[1]);
  }
}

// ================================================================ copy_blocks
struct CopyBlocksParams {
  uint4* k_cache;
  uint4* v_cache;
  const int64_t* block_mapping;
  int num_blocks;
  int64_t block_vecs;  // 16-byte vectors per block
  int64_t slice_vecs;  // vectors per CTA slice of a block
};

// grid (pair, K or V, slice of the block): each CTA copies one slice of one
// block with 16-byte loads and stores.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const __grid_constant__ CopyBlocksParams p) {
  grid_dependency_wait();
  const int64_t src = __ldg(p.block_mapping + 2 * static_cast<int64_t>(blockIdx.x));
  const int64_t dst = __ldg(p.block_mapping + 2 * static_cast<int64_t>(blockIdx.x) + 1);
  if (src < 0 || dst < 0 || src >= p.num_blocks || dst >= p.num_blocks || src == dst) return;
  uint4* pool = blockIdx.y == 0 ? p.k_cache : p.v_cache;
  const int64_t begin = static_cast<int64_t>(blockIdx.z) * p.slice_vecs;
  const int64_t end = begin + p.slice_vecs < p.block_vecs ? begin + p.slice_vecs : p.block_vecs;
  const uint4* from = pool + src * p.block_vecs;
  uint4* to = pool + dst * p.block_vecs;
  for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) to[i] = __ldg(from + i);
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream) {
  if (a.num_pairs == 0) return cudaSuccess;
  CopyBlocksParams p;
  p.k_cache = static_cast<uint4*>(a.k_cache);
  p.v_cache = static_cast<uint4*>(a.v_cache);
  p.block_mapping = a.block_mapping;
  p.num_blocks = a.num_blocks;
  p.block_vecs = a.block_bytes / 16;
  p.slice_vecs = 2048;  // 32 KB per CTA
  const int64_t slices = (p.block_vecs + p.slice_vecs - 1) / p.slice_vecs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_pairs, 2, static_cast<unsigned>(slices));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, copy_blocks_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

namespace {

cudaError_t launch_reshape_e4m3(const ReshapeArgs& a, cudaStream_t stream) {
  ReshapeE4m3Params p;
  p.key = static_cast<const uint4*>(a.key);
  p.value = static_cast<const uint4*>(a.value);
  p.k_cache = static_cast<uint2*>(a.k_cache);
  p.v_cache = static_cast<uint2*>(a.v_cache);
  p.slot_mapping = a.slot_mapping;
  p.num_slots = static_cast<int64_t>(a.num_blocks) * a.block_size;
  p.num_tokens = a.num_tokens;
  p.num_kv_heads = a.num_kv_heads;
  p.row_vecs = a.head_dim / 8;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  const int64_t warps = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = a.dtype == PA_BF16 ? cudaLaunchKernelEx(&cfg, reshape_and_cache_e4m3_kernel<__nv_bfloat16>, p)
                                     : cudaLaunchKernelEx(&cfg, reshape_and_cache_e4m3_kernel<__half>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  if (a.kv_dtype == PA_FP8_E4M3) return launch_reshape_e4m3(a, stream);
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

namespace {

// result[0] = 1 if the wait on a phase that nothing completes gave up, result[1]
// = 1 if the wait on a phase completed by one arrival returned, result[2] = the
// microseconds the first wait took.
__global__ void wait_selftest_kernel(int32_t* result, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar[2];
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);  // nothing arrives here
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&bar[1])) : "memory");
  }
  __syncwarp();
  const uint64_t t0 = global_timer_ns();
  const bool never = mbar_wait_bounded(&bar[0], 0, limit_ns);
  const uint64_t t1 = global_timer_ns();
  const bool done = mbar_wait_bounded(&bar[1], 0, limit_ns);
  if (threadIdx.x == 0) {
    result[0] = never ? 0 : 1;
    result[1] = done ? 1 : 0;
    result[2] = static_cast<int32_t>((t1 - t0) / 1000u);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* result, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(result, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.kv_dtype == PA_FP8_E4M3) return launch_decode_f16_e4m3(a, stream);
  return a.dtype == PA_BF16 ? launch_decode_bf16(a, stream) : launch_decode_f16(a, stream);
}

cudaError_t launch_splitk_reduce(const ReduceArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? launch_splitk_reduce_bf16(a, stream) : launch_splitk_reduce_f16(a, stream);
}

}  // namespace pa
