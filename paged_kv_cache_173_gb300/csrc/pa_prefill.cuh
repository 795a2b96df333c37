// pa_prefill.cuh -- host side of the paged prefill (whole prompts and chunks
// of them) over the K/V pools: the Q tensor map and the launch of
// paged_prefill_tc_kernel (pa_prefill_tc.cuh), templated on the element type
// T (__half or __nv_bfloat16) and the head size.
//
// The method: each new token attends to every earlier position of its
// sequence and to its own ("Efficient Memory Management for LLM Serving with
// PagedAttention -- in-depth reading", section 5.1, item 5: chunked prefill;
// "vAttention: dynamic memory management without PagedAttention": paged
// prefill kernels read K/V through the block table); the block walk and the
// online softmax follow "vLLM PagedAttention source walk-through", section 3.4.
#pragma once

#include "pa_decode.cuh"
#include "pa_prefill_tc.cuh"

namespace pa {

namespace {

// q as [rows][H][d] with a box of 64 dims x G heads x (128 / G) rows, 128-byte
// swizzled: the box lands as the 128-row tile (token, head) of a CTA.
template <typename T>
cudaError_t make_q_map(CUtensorMap* map, const void* q, int head_dim, int num_heads, int group, int64_t rows) {
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encode_fn(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(num_heads) * head_dim * 2};
  const cuuint32_t box[3] = {BOX_DIMS, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(TC_ROWS / group)};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = enc(map, tma_dtype<T>(), 3, const_cast<void*>(q), dims, strides, box, estride,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename T, int HEAD_DIM>
cudaError_t launch_prefill_tc_t(const PrefillArgs& a, cudaStream_t stream) {
  using C = TcCfg<T, HEAD_DIM>;
  auto kern = paged_prefill_tc_kernel<T, HEAD_DIM>;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_smem(kern, C::SMEM_BYTES, smem_set);
  if (e != cudaSuccess) return e;
  PrefillTcParams p;
  const int group = a.num_heads / a.num_kv_heads;
  e = make_q_map<T>(&p.tmap_q, a.q, HEAD_DIM, a.num_heads, group, a.num_rows);
  if (e != cudaSuccess) return e;
  const int64_t pool_rows = static_cast<int64_t>(a.num_blocks) * a.block_size;
  e = make_pool_map<T, HEAD_DIM>(&p.tmap_k, a.k_cache, a.num_kv_heads, pool_rows);
  if (e != cudaSuccess) return e;
  e = make_pool_map<T, HEAD_DIM>(&p.tmap_v, a.v_cache, a.num_kv_heads, pool_rows);
  if (e != cudaSuccess) return e;
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.query_start_loc = a.query_start_loc;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_heads = a.num_heads;
  p.group = group;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.tile_tokens = TC_ROWS / group;
  const int tiles = (a.max_query_len + p.tile_tokens - 1) / p.tile_tokens;
  p.pairs = (tiles + TC_TILES - 1) / TC_TILES;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (p.pairs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.pairs, a.num_kv_heads, a.num_seqs);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_typed(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_rows == 0) return cudaSuccess;
  switch (a.head_dim) {
    case 64: return launch_prefill_tc_t<T, 64>(a, stream);
    case 128: return launch_prefill_tc_t<T, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

}  // namespace pa
