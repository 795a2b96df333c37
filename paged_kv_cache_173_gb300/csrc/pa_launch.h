// pa_launch.h -- internal interface between the C entry points (pa_abi.cu)
// and the kernel launchers (pa_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

struct ReshapeArgs {
  const void* key;
  const void* value;
  void* k_cache;
  void* v_cache;
  const int64_t* slot_mapping;
  int num_tokens;
  int num_blocks;
  int block_size;
  int num_kv_heads;
  int head_dim;
  int dtype;      // key / value: PA_FP16 or PA_BF16
  int kv_dtype;   // the caches: dtype (a plain copy) or PA_FP8_E4M3
  float k_scale;  // E4M3 caches: the stored code is the one nearest to x / scale
  float v_scale;
};

struct CopyBlocksArgs {
  void* k_cache;
  void* v_cache;
  const int64_t* block_mapping;
  int num_pairs;
  int num_blocks;
  int64_t block_bytes;  // block_size * num_kv_heads * head_dim * element size
};

struct DecodeArgs {
  int dtype;     // q and out: PA_FP16 or PA_BF16
  int kv_dtype;  // the caches: dtype, or PA_FP8_E4M3 (values = code * k_scale / v_scale)
  float k_scale;
  float v_scale;
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws;  // split-K workspace (nullptr for single-pass decode)
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  float scale;
  int partition_size;      // tokens; single-pass decode uses max_blocks_per_seq * block_size
  int max_num_partitions;  // grid extent along partitions (split-K)
  int cluster_size;        // > 0: one cluster of this many CTAs per (sequence, KV head);
                           // 0: plain grid; < 0: chosen from occupancy
  const int32_t* prefix_lens;  // shared-prefix split-K: [ceil(num_seqs / seqs_per_group)], else null
  int seqs_per_group;
  // Append: one new token per sequence, [S][Hk][d] of `dtype`, written into
  // the pools at the slot of position ctx - 1 by the decode itself (null: none).
  const void* new_key;
  const void* new_value;
};

struct ReduceArgs {
  int dtype;  // PA_FP16 or PA_BF16
  void* out;
  const float* ws;
  const int32_t* context_lens;
  int max_blocks_per_seq;
  int block_size;
  int num_seqs;
  int num_heads;
  int head_dim;
  int partition_size;
  int max_num_partitions;
};

struct PrefillArgs {
  int dtype;  // PA_FP16 or PA_BF16
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int max_blocks_per_seq;
  int num_seqs;
  int num_rows;
  int max_query_len;
  int num_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  float scale;
};

// Record a formatted message as the calling thread's last error; returns status.
int set_last_error(int status, const char* fmt, ...);

// The host checks of a split-K decode call except those of its workspace
// (shapes, types, pointers, partition_size a positive multiple of
// block_size); PA_OK or the status and last-error text of the first failure.
int check_splitk_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int dtype, int partition_size);

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream);
cudaError_t launch_wait_selftest(int32_t* result, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const ReduceArgs& a, cudaStream_t stream);

// per element type (pa_decode_f16.cu, pa_decode_bf16.cu)
cudaError_t launch_decode_f16(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_splitk_reduce_f16(const ReduceArgs& a, cudaStream_t stream);
cudaError_t launch_splitk_reduce_bf16(const ReduceArgs& a, cudaStream_t stream);
// E4M3 caches with float16 queries (pa_decode_fp8.cu)
cudaError_t launch_decode_f16_e4m3(const DecodeArgs& a, cudaStream_t stream);
// paged prefill (pa_prefill.cu)
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// shared-prefix split-K (pa_decode_prefix.cu): the shared pass, then the
// per-sequence pass
cudaError_t launch_decode_prefix(const DecodeArgs& a, cudaStream_t stream);

// Workspace geometry shared by the partition kernel and the reduce kernel:
// o [S][H][P][d], then m [S][H][P], then l [S][H][P], float32.
inline size_t ws_rows(int num_seqs, int num_heads, int max_num_partitions) {
  return static_cast<size_t>(num_seqs) * num_heads * max_num_partitions;
}

}  // namespace pa
