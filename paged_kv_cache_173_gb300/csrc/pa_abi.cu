// pa_abi.cu -- the extern "C" entry points of libpagedattn.so.
//
// Host-side argument checks, then one launch per kernel on the caller's
// stream.  Semantics and argument layouts are stated in include/pagedattn.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdint>

#include "pa_launch.h"
#include "pagedattn.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int ok() {
  g_last_error[0] = '\0';
  return PA_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  // a launch-configuration error is not sticky: clear it so that it is not
  // reported again by the caller's next launch
  (void)cudaGetLastError();
  return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 16, 32, 64, 128 or 256 tokens per block.
bool block_size_supported(int b) { return b >= 16 && b <= 256 && (b & (b - 1)) == 0; }

// Shape checks shared by every decode entry point.
int check_decode(const void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                 int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                 int num_blocks, float scale, int dtype) {
  if (dtype != PA_FP16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "dtype %d is not supported (PA_FP16 or PA_BF16)", dtype);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not supported (64, 128 or 256)", head_dim);
  if (!block_size_supported(block_size))
    return fail(PA_ERR_UNSUPPORTED, "block_size %d is not supported (16, 32, 64, 128 or 256)",
                block_size);
  if (num_heads <= 0 || num_kv_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_heads (%d) and num_kv_heads (%d) must be positive", num_heads,
                num_kv_heads);
  if (num_heads % num_kv_heads != 0)
    return fail(PA_ERR_UNSUPPORTED, "num_heads %d is not a multiple of num_kv_heads %d", num_heads,
                num_kv_heads);
  if (num_heads / num_kv_heads > 16)
    return fail(PA_ERR_UNSUPPORTED, "query group size %d exceeds 16", num_heads / num_kv_heads);
  if (head_dim == 256 && num_heads / num_kv_heads > 8)
    return fail(PA_ERR_UNSUPPORTED, "head_dim 256 supports query groups of at most 8 (got %d)",
                num_heads / num_kv_heads);
  if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs %d is negative", num_seqs);
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "num_seqs %d exceeds 65535", num_seqs);
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d must be positive", max_blocks_per_seq);
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq * block_size exceeds 2^31 - 1");
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks %d must be positive", num_blocks);
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * block_size exceeds 2^31 - 1 token slots");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PA_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PA_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  return PA_OK;
}

int needed_partitions(int max_blocks_per_seq, int block_size, int partition_size) {
  const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  return static_cast<int>((cap + partition_size - 1) / partition_size);
}

int check_splitk(int max_blocks_per_seq, int block_size, int partition_size, int max_num_partitions,
                 const void* workspace, size_t workspace_bytes, int num_seqs, int num_heads,
                 int head_dim) {
  if (partition_size <= 0 || partition_size % block_size != 0)
    return fail(PA_ERR_INVALID_ARG, "partition_size %d must be a positive multiple of block_size %d",
                partition_size, block_size);
  const int need = needed_partitions(max_blocks_per_seq, block_size, partition_size);
  if (max_num_partitions < need)
    return fail(PA_ERR_INVALID_ARG, "max_num_partitions %d < ceil(max_blocks_per_seq * block_size / "
                "partition_size) = %d", max_num_partitions, need);
  if (max_num_partitions > 65535)
    return fail(PA_ERR_UNSUPPORTED, "max_num_partitions %d exceeds 65535", max_num_partitions);
  if (num_seqs == 0) return PA_OK;
  const size_t bytes = pa_splitk_workspace_bytes(num_seqs, num_heads, head_dim, max_num_partitions);
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(PA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (workspace_bytes < bytes)
    return fail(PA_ERR_INVALID_ARG, "workspace_bytes %zu < %zu required", workspace_bytes, bytes);
  return PA_OK;
}

int check_kv_scales(float k_scale, float v_scale) {
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
    return fail(PA_ERR_INVALID_ARG, "k_scale (%g) and v_scale (%g) must be finite and positive",
                static_cast<double>(k_scale), static_cast<double>(v_scale));
  return PA_OK;
}

// The cache type of an E4M3 decode and the query types it takes.
int check_fp8_decode(int dtype, float k_scale, float v_scale) {
  if (dtype != PA_FP16)
    return fail(PA_ERR_UNSUPPORTED, "E4M3 caches take PA_FP16 queries (got dtype %d)", dtype);
  return check_kv_scales(k_scale, v_scale);
}

pa::DecodeArgs decode_args(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, float scale, int dtype, int kv_dtype, float k_scale,
                           float v_scale) {
  pa::DecodeArgs a{};
  a.prefix_lens = nullptr;
  a.seqs_per_group = 1;
  a.dtype = dtype;
  a.kv_dtype = kv_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.ws = nullptr;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  return a;
}

// pa_decode / pa_decode_fp8 after their own dtype checks.
int decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                int num_blocks, float scale, int dtype, int kv_dtype, float k_scale, float v_scale,
                void* stream) {
  int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        dtype);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return ok();
  pa::DecodeArgs a = decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                 num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 dtype, kv_dtype, k_scale, v_scale);
  // One CTA per (sequence, KV head) when the pairs fill the GPU; otherwise a
  // cluster of up to 8 CTAs per pair that split the sequence and merge
  // through distributed shared memory (chosen by the launcher).
  a.cluster_size = -1;
  a.partition_size = max_blocks_per_seq * block_size;
  a.max_num_partitions = 1;
  return cuda_status(pa::launch_decode(a, static_cast<cudaStream_t>(stream)), "decode launch");
}

// pa_decode_splitk / pa_decode_splitk_fp8 after their own dtype checks.
int splitk_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                int num_blocks, float scale, int dtype, int kv_dtype, float k_scale, float v_scale,
                int partition_size, int max_num_partitions, void* workspace, size_t workspace_bytes,
                void* stream) {
  int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        dtype);
  if (st != PA_OK) return st;
  st = check_splitk(max_blocks_per_seq, block_size, partition_size, max_num_partitions, workspace,
                    workspace_bytes, num_seqs, num_heads, head_dim);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return ok();
  pa::DecodeArgs a = decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                 num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 dtype, kv_dtype, k_scale, v_scale);
  a.ws = static_cast<float*>(workspace);
  a.partition_size = partition_size;
  a.max_num_partitions = max_num_partitions;
  a.cluster_size = 0;
  return cuda_status(pa::launch_decode(a, static_cast<cudaStream_t>(stream)), "split-K decode launch");
}

// The new-token arguments and cache types of the append entry points.
int check_append(const void* key, const void* value, int num_seqs, int dtype, int kv_dtype, float k_scale,
                 float v_scale) {
  if (kv_dtype == PA_FP8_E4M3) {
    const int st = check_fp8_decode(dtype, k_scale, v_scale);
    if (st != PA_OK) return st;
  } else if (kv_dtype != dtype) {
    return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d must equal dtype %d or be PA_FP8_E4M3", kv_dtype, dtype);
  }
  if (num_seqs == 0) return PA_OK;
  if (!key || !value) return fail(PA_ERR_INVALID_ARG, "key and value must not be NULL");
  if (!aligned(key, 16) || !aligned(value, 16))
    return fail(PA_ERR_INVALID_ARG, "key and value must be 16-byte aligned");
  return PA_OK;
}

// pa_append_and_decode / pa_append_and_decode_splitk: the decode arguments
// with the new tokens' rows; workspace == NULL selects the single pass.
int append_impl(void* out, const void* q, const void* key, const void* value, void* k_cache, void* v_cache,
                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                int dtype, int kv_dtype, float k_scale, float v_scale, bool splitk, int partition_size,
                int max_num_partitions, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_append(key, value, num_seqs, dtype, kv_dtype, k_scale, v_scale);
  if (st != PA_OK) return st;
  st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                    num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype);
  if (st != PA_OK) return st;
  if (splitk) {
    st = check_splitk(max_blocks_per_seq, block_size, partition_size, max_num_partitions, workspace,
                      workspace_bytes, num_seqs, num_heads, head_dim);
    if (st != PA_OK) return st;
  }
  if (num_seqs == 0) return ok();
  const bool fp8 = kv_dtype == PA_FP8_E4M3;
  pa::DecodeArgs a = decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                 num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 dtype, kv_dtype, fp8 ? k_scale : 1.f, fp8 ? v_scale : 1.f);
  a.new_key = key;
  a.new_value = value;
  if (splitk) {
    a.ws = static_cast<float*>(workspace);
    a.partition_size = partition_size;
    a.max_num_partitions = max_num_partitions;
    a.cluster_size = 0;
  } else {
    a.cluster_size = -1;
    a.partition_size = max_blocks_per_seq * block_size;
    a.max_num_partitions = 1;
  }
  return cuda_status(pa::launch_decode(a, static_cast<cudaStream_t>(stream)),
                     splitk ? "append + split-K decode launch" : "append + decode launch");
}

// The checks shared by both cache writes.
int check_reshape(const void* key, const void* value, const void* k_cache, const void* v_cache,
                  const int64_t* slot_mapping, int num_tokens, int num_blocks, int block_size,
                  int num_kv_heads, int head_dim, int dtype) {
  if (dtype != PA_FP16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "dtype %d is not supported (PA_FP16 or PA_BF16)", dtype);
  if (head_dim <= 0 || head_dim % 8 != 0 || head_dim > 1024)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not supported (a multiple of 8, at most 1024)",
                head_dim);
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens %d is negative", num_tokens);
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_blocks, block_size and num_kv_heads must be positive");
  if (static_cast<int64_t>(num_tokens) * num_kv_heads > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "num_tokens * num_kv_heads exceeds 2^31 - 1");
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(PA_ERR_INVALID_ARG, "key, value and the caches must be 16-byte aligned, "
                "slot_mapping 8-byte aligned");
  return PA_OK;
}

}  // namespace

namespace pa {

int check_splitk_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int dtype, int partition_size) {
  const int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                              num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype);
  if (st != PA_OK) return st;
  if (partition_size <= 0 || partition_size % block_size != 0)
    return fail(PA_ERR_INVALID_ARG, "partition_size %d must be a positive multiple of block_size %d",
                partition_size, block_size);
  return PA_OK;
}

int set_last_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

}  // namespace pa

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    default: return "PA_UNKNOWN_STATUS";
  }
}

const char* pa_last_error(void) { return g_last_error; }

int pa_selftest_wait(int32_t* result, unsigned limit_us, void* stream) {
  if (!result) return fail(PA_ERR_INVALID_ARG, "result is NULL");
  if (!aligned(result, 4)) return fail(PA_ERR_INVALID_ARG, "result must be 4-byte aligned");
  if (limit_us == 0 || limit_us > 10000000u)
    return fail(PA_ERR_INVALID_ARG, "limit_us %u must be in 1 .. 10,000,000", limit_us);
  return cuda_status(pa::launch_wait_selftest(result, static_cast<uint64_t>(limit_us) * 1000u,
                                              static_cast<cudaStream_t>(stream)),
                     "wait self-test launch");
}

size_t pa_splitk_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_num_partitions) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_num_partitions <= 0) return 0;
  const size_t rows = pa::ws_rows(num_seqs, num_heads, max_num_partitions);
  return rows * (static_cast<size_t>(head_dim) + 2) * sizeof(float);
}

int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_blocks,
                         int block_size, int num_kv_heads, int head_dim, int dtype, void* stream) {
  const int st = check_reshape(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                               block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_tokens == 0) return ok();
  pa::ReshapeArgs a{key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks, block_size,
                    num_kv_heads, head_dim, dtype, dtype, 1.f, 1.f};
  return cuda_status(pa::launch_reshape_and_cache(a, static_cast<cudaStream_t>(stream)),
                     "reshape_and_cache launch");
}

int pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim, int dtype,
                             float k_scale, float v_scale, void* stream) {
  int st = check_reshape(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks, block_size,
                         num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (head_dim % 16 != 0)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not supported for E4M3 caches (a multiple of 16)",
                head_dim);
  st = check_kv_scales(k_scale, v_scale);
  if (st != PA_OK) return st;
  if (num_tokens == 0) return ok();
  pa::ReshapeArgs a{key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks, block_size,
                    num_kv_heads, head_dim, dtype, PA_FP8_E4M3, k_scale, v_scale};
  return cuda_status(pa::launch_reshape_and_cache(a, static_cast<cudaStream_t>(stream)),
                     "reshape_and_cache_fp8 launch");
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int num_pairs,
                   int num_blocks, int block_size, int num_kv_heads, int head_dim, int dtype,
                   void* stream) {
  if (dtype != PA_FP16 && dtype != PA_BF16 && dtype != PA_FP8_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "dtype %d is not supported (PA_FP16, PA_BF16 or PA_FP8_E4M3)", dtype);
  if (num_pairs < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs %d is negative", num_pairs);
  if (num_pairs > INT32_MAX / 2) return fail(PA_ERR_UNSUPPORTED, "num_pairs %d is too large", num_pairs);
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_blocks, block_size, num_kv_heads and head_dim must be positive");
  const int64_t block_bytes =
      static_cast<int64_t>(block_size) * num_kv_heads * head_dim * (dtype == PA_FP8_E4M3 ? 1 : 2);
  if (block_bytes % 16 != 0)
    return fail(PA_ERR_UNSUPPORTED, "block bytes %lld are not a multiple of 16", (long long)block_bytes);
  if (num_pairs == 0) return ok();
  if (!k_cache || !v_cache || !block_mapping) return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_mapping, 8))
    return fail(PA_ERR_INVALID_ARG, "the caches must be 16-byte aligned, block_mapping 8-byte aligned");
  pa::CopyBlocksArgs a{k_cache, v_cache, block_mapping, num_pairs, num_blocks, block_bytes};
  return cuda_status(pa::launch_copy_blocks(a, static_cast<cudaStream_t>(stream)), "copy_blocks launch");
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
              int num_blocks, float scale, int dtype, void* stream) {
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, dtype, 1.f,
                     1.f, stream);
}

int pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                  int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int dtype, float k_scale, float v_scale,
                  void* stream) {
  const int st = check_fp8_decode(dtype, k_scale, v_scale);
  if (st != PA_OK) return st;
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, PA_FP8_E4M3,
                     k_scale, v_scale, stream);
}

int pa_decode_splitk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                     int head_dim, int block_size, int num_blocks, float scale, int dtype,
                     int partition_size, int max_num_partitions, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return splitk_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, dtype, 1.f,
                     1.f, partition_size, max_num_partitions, workspace, workspace_bytes, stream);
}

int pa_decode_splitk_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, int dtype, float k_scale, float v_scale, int partition_size,
                         int max_num_partitions, void* workspace, size_t workspace_bytes,
                         void* stream) {
  const int st = check_fp8_decode(dtype, k_scale, v_scale);
  if (st != PA_OK) return st;
  return splitk_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, PA_FP8_E4M3,
                     k_scale, v_scale, partition_size, max_num_partitions, workspace, workspace_bytes,
                     stream);
}

int pa_decode_prefix_splitk(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            float scale, int dtype, int kv_dtype, float k_scale, float v_scale,
                            int seqs_per_group, const int32_t* prefix_lens, int partition_size,
                            int max_num_partitions, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (kv_dtype == PA_FP8_E4M3) {
    const int st = check_fp8_decode(dtype, k_scale, v_scale);
    if (st != PA_OK) return st;
  } else if (kv_dtype != dtype) {
    return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d must equal dtype %d or be PA_FP8_E4M3", kv_dtype, dtype);
  }
  int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        dtype);
  if (st != PA_OK) return st;
  st = check_splitk(max_blocks_per_seq, block_size, partition_size, max_num_partitions, workspace,
                    workspace_bytes, num_seqs, num_heads, head_dim);
  if (st != PA_OK) return st;
  if (seqs_per_group <= 0) return fail(PA_ERR_INVALID_ARG, "seqs_per_group %d must be positive", seqs_per_group);
  if (num_seqs == 0) return ok();
  if (!prefix_lens) return fail(PA_ERR_INVALID_ARG, "prefix_lens is NULL");
  if (!aligned(prefix_lens, 4)) return fail(PA_ERR_INVALID_ARG, "prefix_lens must be 4-byte aligned");
  pa::DecodeArgs a = decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                 num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 dtype, kv_dtype, kv_dtype == PA_FP8_E4M3 ? k_scale : 1.f,
                                 kv_dtype == PA_FP8_E4M3 ? v_scale : 1.f);
  a.ws = static_cast<float*>(workspace);
  a.partition_size = partition_size;
  a.max_num_partitions = max_num_partitions;
  a.cluster_size = 0;
  a.prefix_lens = prefix_lens;
  a.seqs_per_group = seqs_per_group;
  return cuda_status(pa::launch_decode_prefix(a, static_cast<cudaStream_t>(stream)),
                     "shared-prefix decode launch");
}

int pa_append_and_decode(void* out, const void* q, const void* key, const void* value, void* k_cache,
                         void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, float scale, int dtype, int kv_dtype,
                         float k_scale, float v_scale, void* stream) {
  return append_impl(out, q, key, value, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, kv_dtype,
                     k_scale, v_scale, false, 0, 1, nullptr, 0, stream);
}

int pa_append_and_decode_splitk(void* out, const void* q, const void* key, const void* value, void* k_cache,
                                void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, int num_blocks, float scale, int dtype,
                                int kv_dtype, float k_scale, float v_scale, int partition_size,
                                int max_num_partitions, void* workspace, size_t workspace_bytes, void* stream) {
  return append_impl(out, q, key, value, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, kv_dtype,
                     k_scale, v_scale, true, partition_size, max_num_partitions, workspace, workspace_bytes,
                     stream);
}

int pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
               const int32_t* query_start_loc, int num_seqs, int num_rows, int max_query_len,
               int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
               float scale, int dtype, void* stream) {
  int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        dtype);
  if (st != PA_OK) return st;
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "prefill supports head_dim 64 or 128 (got %d)", head_dim);
  const int G = num_heads / num_kv_heads;
  if (128 % G != 0)
    return fail(PA_ERR_UNSUPPORTED, "prefill needs a query group size dividing 128 (got %d)", G);
  if (max_query_len < 0 || num_rows < 0)
    return fail(PA_ERR_INVALID_ARG, "max_query_len (%d) and num_rows (%d) must be >= 0", max_query_len, num_rows);
  if (num_seqs == 0 || max_query_len == 0 || num_rows == 0) return ok();
  if (!query_start_loc) return fail(PA_ERR_INVALID_ARG, "query_start_loc is NULL");
  if (!aligned(query_start_loc, 4)) return fail(PA_ERR_INVALID_ARG, "query_start_loc must be 4-byte aligned");
  pa::PrefillArgs a{dtype,      out,       q,           k_cache,      v_cache,      block_tables,
                    context_lens, query_start_loc, max_blocks_per_seq, num_seqs, num_rows,
                    max_query_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale};
  return cuda_status(pa::launch_prefill(a, static_cast<cudaStream_t>(stream)), "prefill launch");
}

int pa_splitk_reduce(void* out, const void* workspace, size_t workspace_bytes,
                     const int32_t* context_lens, int max_blocks_per_seq, int block_size,
                     int num_seqs, int num_heads, int head_dim, int partition_size,
                     int max_num_partitions, int dtype, void* stream) {
  if (dtype != PA_FP16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "dtype %d is not supported (PA_FP16 or PA_BF16)", dtype);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not supported (64, 128 or 256)", head_dim);
  if (!block_size_supported(block_size))
    return fail(PA_ERR_UNSUPPORTED, "block_size %d is not supported", block_size);
  if (num_seqs < 0 || num_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_seqs must be >= 0 and num_heads > 0");
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "num_seqs %d exceeds 65535", num_seqs);
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d must be positive", max_blocks_per_seq);
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq * block_size exceeds 2^31 - 1");
  int st = check_splitk(max_blocks_per_seq, block_size, partition_size, max_num_partitions, workspace,
                        workspace_bytes, num_seqs, num_heads, head_dim);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return ok();
  if (!out || !context_lens) return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(out, 16) || !aligned(context_lens, 4))
    return fail(PA_ERR_INVALID_ARG, "out must be 16-byte aligned, context_lens 4-byte aligned");
  pa::ReduceArgs a{dtype, out, static_cast<const float*>(workspace), context_lens, max_blocks_per_seq,
                   block_size, num_seqs, num_heads, head_dim, partition_size, max_num_partitions};
  return cuda_status(pa::launch_splitk_reduce(a, static_cast<cudaStream_t>(stream)),
                     "split-K reduce launch");
}

}  // extern "C"
