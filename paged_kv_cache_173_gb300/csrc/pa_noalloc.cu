// pa_noalloc.cu -- split-K decode for callers that cannot allocate device
// memory: the partials live in a fixed array inside the library.
//
// Who needs it: a serving runtime that reserves (nearly) all device memory
// for its KV-cache pool at start-up and hands out no scratch afterwards; a
// host program that reaches the library only through this C ABI and owns no
// GPU allocator of its own; and any decode loop that must not call cudaMalloc,
// which can synchronise the whole device.  Such a caller passes its inputs and
// outputs only; this entry point brings its own workspace.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "pa_launch.h"
#include "pagedattn.h"

namespace {

// The split-K workspace (partition outputs o, maxima m and sums l, float32).
// One copy per GPU that loads the library, held until the process exits.
static __device__ __align__(256) float g_static_scratch[PA_STATIC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
std::atomic<float*> g_scratch_addr[kMaxDevices];

// The device address of g_static_scratch on the current device, looked up once
// per device.  In host code the symbol is only a host-side stand-in; passing it
// to a kernel would address the wrong memory.
int scratch_on_current_device(float** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return pa::set_last_error(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pa::set_last_error(PA_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  float* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* sym = nullptr;
    e = cudaGetSymbolAddress(&sym, g_static_scratch);
    if (e != cudaSuccess || sym == nullptr)
      return pa::set_last_error(PA_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s",
                                cudaGetErrorString(e));
    p = static_cast<float*>(sym);
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *addr = p;
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_splitk_static(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, float scale, int dtype,
                                       int partition_size, void* stream) {
  // the arguments first, so that an invalid call is reported as such and not
  // as a batch too large for the scratch
  const int chk = pa::check_splitk_decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                               context_lens, num_seqs, num_heads, num_kv_heads, head_dim,
                                               block_size, num_blocks, scale, dtype, partition_size);
  if (chk != PA_OK) return chk;
  const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  const int64_t parts = (cap + partition_size - 1) / partition_size;
  const int max_num_partitions = parts > INT32_MAX ? INT32_MAX : static_cast<int>(parts);
  const size_t need = pa_splitk_workspace_bytes(num_seqs, num_heads, head_dim, max_num_partitions);
  if (need > PA_STATIC_SCRATCH_BYTES)
    return pa::set_last_error(PA_ERR_UNSUPPORTED,
                              "this batch needs %zu bytes of split-K scratch; the static scratch holds "
                              "%zu bytes (use pa_decode_splitk with a caller workspace, or a larger "
                              "partition_size)",
                              need, static_cast<size_t>(PA_STATIC_SCRATCH_BYTES));
  float* ws = nullptr;
  if (num_seqs > 0) {
    const int st = scratch_on_current_device(&ws);
    if (st != PA_OK) return st;
  }
  // The partition kernel writes every workspace row that the reduce reads in
  // this call, so stale contents from an earlier call need no clearing.
  int st = pa_decode_splitk(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                            dtype, partition_size, max_num_partitions, ws, PA_STATIC_SCRATCH_BYTES,
                            stream);
  if (st != PA_OK) return st;
  return pa_splitk_reduce(out, ws, PA_STATIC_SCRATCH_BYTES, context_lens, max_blocks_per_seq,
                          block_size, num_seqs, num_heads, head_dim, partition_size,
                          max_num_partitions, dtype, stream);
}
