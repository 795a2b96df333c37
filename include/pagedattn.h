/*
 * pagedattn.h -- C ABI of libpagedattn.so: PagedAttention decode for GB300
 * (sm_103a).
 *
 * The KV cache of one layer lives in two preallocated pools of fixed-size
 * blocks, one for keys and one for values, each laid out
 *
 *     [num_blocks][block_size][num_kv_heads][head_dim]      (row-major)
 *
 * A sequence's tokens are scattered over physical blocks; its block table
 * row maps logical block i to a physical block id, and its context length
 * bounds the valid slots of its last block.  ("PagedAttention: when the KV
 * cache meets OS paging", section 3.1; "Efficient Memory Management for LLM
 * Serving with PagedAttention -- in-depth reading", sections 2.3 and 3.2.)
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller.  The library allocates
 *    nothing and keeps no state between calls except a per-thread text of
 *    the last error (pa_last_error), a per-device record of which kernel
 *    attributes it has already set, a per-thread cache of the TMA
 *    descriptors it encoded for recently seen pools (a descriptor depends
 *    only on the pool's address and shape, so a cached one is always the one
 *    a fresh encoding gives), and the fixed device array that
 *    pa_decode_splitk_static uses as its workspace.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream).  The caller synchronises.
 *  - The return value is a pa_status.  Arguments are checked on the host
 *    before any launch; on an error nothing is launched.  Values that live in
 *    device memory (slot ids, block ids, context lengths) cannot be read by
 *    the host without a synchronisation, so the kernels check them instead
 *    and never read or write outside the buffers whose sizes the call states:
 *    the documented outcome of a bad device value is given with each call.
 *  - Tensor pointers must be 16-byte aligned and the tensors contiguous in
 *    the layouts given.  Element type (dtype): PA_FP16 or PA_BF16, the same
 *    for q, the caches, the new tokens and out.  Scores, softmax and
 *    accumulation are float32; the attention weights enter the P.V product
 *    as fp16, or for bf16 as a rounded value plus its rounded residual.
 *  - Supported shapes: head_dim in {64, 128, 256}; block_size in {16, 32,
 *    64, 128, 256}; num_heads a multiple of num_kv_heads with
 *    num_heads / num_kv_heads <= 16 (<= 8 for head_dim 256);
 *    num_seqs <= 65535.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, inconsistent sizes  */
  PA_ERR_UNSUPPORTED = -2, /* a shape or dtype outside the supported set  */
  PA_ERR_CUDA = -3         /* a CUDA runtime error; see pa_last_error()   */
} pa_status;

typedef enum pa_dtype {
  PA_FP16 = 0,    /* IEEE binary16 */
  PA_BF16 = 1,    /* bfloat16 (the upper half of an IEEE binary32) */
  PA_FP8_E4M3 = 2 /* a cache of OCP E4M3 codes (pa_*_fp8 entry points and
                     pa_copy_blocks only) */
} pa_dtype;

/*
 * pa_reshape_and_cache -- write each new token's key and value into its slot.
 *
 * Defined by the cache write of "vLLM PagedAttention source walk-through",
 * section 3.2 (append_token computes block_idx = pos / block_size and
 * block_offset = pos % block_size and writes the token's KV there) and
 * "in-depth reading", section 3.4, step 1.  The slot is passed flattened:
 *
 *     slot = physical_block * block_size + block_offset
 *
 * For every token t < num_tokens with slot_mapping[t] >= 0 and every KV head
 * h:  k_cache[slot / block_size][slot % block_size][h][:] = key[t][h][:],
 * likewise v_cache from value.  The copy is bit-exact.
 *
 *   key, value     [num_tokens][num_kv_heads][head_dim], read only
 *   k_cache,
 *   v_cache        [num_blocks][block_size][num_kv_heads][head_dim], written
 *                  in place at the mapped slots only
 *   slot_mapping   [num_tokens] int64.  Negative: padding, skipped.  A slot
 *                  >= num_blocks * block_size is a caller error; it is
 *                  skipped (nothing is written out of bounds).  Slots must be
 *                  distinct: with duplicates the surviving value is undefined.
 *   num_tokens     >= 0 (0 is a no-op)
 *
 * Copy-on-write of a block shared by several sequences is the caller's job
 * (the write goes to whatever block the slot names).
 */
int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_blocks,
                         int block_size, int num_kv_heads, int head_dim, int dtype,
                         void* stream);

/*
 * pa_copy_blocks -- copy whole KV blocks, the copy step of copy-on-write.
 *
 * Sequences may share physical blocks (parallel sampling from one prompt:
 * their block tables point at the same ids, with a reference count); before
 * one of them writes into a shared block, its runtime copies the block to a
 * free one and repoints that sequence's table entry.  ("Unveiling the NVIDIA
 * driver stack: GPU page tables and vLLM PagedAttention", section 4:
 * reference counts and copy-on-write protect writes to shared blocks;
 * "PagedAttention: when the KV cache meets OS paging", section 4.3;
 * "Efficient Memory Management for LLM Serving with PagedAttention --
 * in-depth reading", section 2.4.)
 *
 * For every pair i < num_pairs with src = block_mapping[2i] and
 * dst = block_mapping[2i + 1]:
 *     k_cache[dst][:][:][:] = k_cache[src][:][:][:], likewise v_cache,
 * a bit-exact copy of block_size * num_kv_heads * head_dim elements.
 *
 *   k_cache, v_cache  [num_blocks][block_size][num_kv_heads][head_dim]
 *   block_mapping     [num_pairs][2] int64 (src, dst)
 *   dtype             PA_FP16, PA_BF16 or PA_FP8_E4M3 (the copy moves
 *                     bytes; only the element size matters)
 *
 * Device-value outcomes: a pair with an id outside [0, num_blocks), or with
 * src == dst, is skipped.  Destinations must be distinct and no destination
 * may be the source of another pair in the same call (otherwise the result
 * depends on the order of the copies).
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int num_pairs,
                   int num_blocks, int block_size, int num_kv_heads, int head_dim, int dtype,
                   void* stream);

/*
 * pa_decode -- single-pass paged decode attention, one query token per
 * sequence.
 *
 * Defined by "vLLM PagedAttention source walk-through", section 3.4 (walk the
 * block table, load each block's K and V, score q against K scaled by
 * `scale`, mask the slots past the context, online softmax with a running
 * maximum and sum, accumulate the probabilities times V, normalise by the
 * running sum) and "PagedAttention: when the KV cache meets OS paging",
 * section 3.2.  The result equals ordinary softmax attention over the
 * sequence's first context_lens[s] tokens:
 *
 *   out[s][h][:] = sum_i softmax_i(scale * q[s][h] . K_i) * V_i,
 *   K_i, V_i     = pool rows of token i of sequence s, KV head h / G,
 *   G            = num_heads / num_kv_heads (consecutive query heads share a
 *                  KV head).
 *
 *   out            [num_seqs][num_heads][head_dim], written (fp16, rounded
 *                  to nearest even)
 *   q              [num_seqs][num_heads][head_dim]
 *   k_cache,
 *   v_cache        [num_blocks][block_size][num_kv_heads][head_dim]
 *   block_tables   [num_seqs][max_blocks_per_seq] int32 physical block ids;
 *                  only the first ceil(context_lens[s] / block_size) entries
 *                  of a row are read
 *   context_lens   [num_seqs] int32, the number of valid tokens, including
 *                  the token being decoded
 *
 * Device-value outcomes: context_lens[s] == 0 gives out[s] = 0;
 * context_lens[s] < 0 or > max_blocks_per_seq * block_size, or a block id
 * read from the table outside [0, num_blocks), gives NaN in out for the
 * affected (sequence, KV-head group).  Nothing is read out of bounds.
 */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
              int num_blocks, float scale, int dtype, void* stream);

/*
 * pa_splitk_workspace_bytes -- size of the split-K workspace.
 *
 * The workspace holds, per (sequence, query head, partition), the
 * partition's normalised output o_p [head_dim] and its log-sum-exp pair
 * (m_p, l_p), all float32:  num_seqs * num_heads * max_num_partitions *
 * (head_dim + 2) * 4 bytes.  Returns 0 for non-positive arguments.
 */
size_t pa_splitk_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_num_partitions);

/*
 * pa_decode_splitk -- the same attention as pa_decode, with each sequence's
 * context cut into partitions of partition_size tokens that run in parallel.
 *
 * Partition p of sequence s covers tokens [p * partition_size,
 * min((p + 1) * partition_size, context_lens[s])).  Each runs the online
 * softmax of "vLLM PagedAttention source walk-through", section 3.4 over its
 * tokens and stores o_p = acc_p / l_p together with its running maximum m_p
 * (in log2 units: m_p = max_i scale * log2(e) * q . K_i) and sum
 * l_p = sum_i 2^(scale * log2(e) * q . K_i - m_p).  pa_splitk_reduce merges
 * the partitions with the same correction factor the walk-through's online
 * softmax applies between blocks.
 *
 * Sequences with at most one partition are finished here: out[s] is written
 * directly and they leave nothing in the workspace.  Calling
 * pa_splitk_reduce afterwards is always required and always correct.
 *
 *   partition_size      tokens per partition, a positive multiple of
 *                       block_size
 *   max_num_partitions  >= ceil(max_blocks_per_seq * block_size /
 *                       partition_size)
 *   workspace           device buffer of workspace_bytes >=
 *                       pa_splitk_workspace_bytes(num_seqs, num_heads,
 *                       head_dim, max_num_partitions); scratch owned by the
 *                       caller, contents on entry ignored
 *
 * Other arguments and device-value outcomes as pa_decode.
 */
int pa_decode_splitk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                     int head_dim, int block_size, int num_blocks, float scale, int dtype,
                     int partition_size, int max_num_partitions, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * pa_decode_prefix_splitk -- pa_decode_splitk for batches whose sequences
 * share prompt blocks: each shared block is read once per group instead of
 * once per sequence.
 *
 * Parallel sampling (several outputs from one prompt) and shared prefixes
 * let several block tables point at the same physical blocks ("Unveiling
 * the NVIDIA driver stack: GPU page tables and vLLM PagedAttention",
 * section 4; "PagedAttention: when the KV cache meets OS paging", section
 * 4.3; "in-depth reading", section 2.4).  The result is the attention that
 * pa_decode_splitk computes.  What changes is the bytes read: a shared
 * prompt block is read once per group and KV head (for up to 16 / G
 * sequences of the group per read, 8 / G at head_dim 256).
 *
 * Groups: sequences [j * seqs_per_group, min((j + 1) * seqs_per_group,
 * num_seqs)) form group j; callers order the batch so that the sequences of
 * one prompt are consecutive.  prefix_lens[j] (device, int32,
 * ceil(num_seqs / seqs_per_group) entries) is the number of leading tokens
 * that the group's sequences hold in the same physical blocks (the first
 * prefix_lens[j] / block_size entries of their table rows are equal).
 *
 * Sequence s of group j has its first L = prefix_lens[j] tokens computed by
 * the group's shared pass when L is a positive multiple of partition_size,
 * L <= context_lens[s], and L <= the context length of the group's first
 * sequence (both within max_blocks_per_seq * block_size).  Otherwise the
 * whole sequence is computed on its own, exactly as by pa_decode_splitk.
 * The shared pass reads the prefix through the group's first table row.
 *
 *   dtype, kv_dtype   PA_FP16 or PA_BF16 with kv_dtype == dtype, or dtype
 *                     PA_FP16 with kv_dtype PA_FP8_E4M3 and the pool scales
 *                     k_scale, v_scale (ignored for 16-bit caches)
 *   seqs_per_group    >= 1
 *
 * Follow with pa_splitk_reduce (same partition_size, max_num_partitions,
 * workspace; dtype of out) on the same stream.  Other arguments as
 * pa_decode_splitk.
 *
 * Device-value outcomes: as pa_decode_splitk.  In addition, a sequence whose
 * table entries over the shared prefix differ from the group's first row
 * gets NaN.
 */
int pa_decode_prefix_splitk(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            float scale, int dtype, int kv_dtype, float k_scale, float v_scale,
                            int seqs_per_group, const int32_t* prefix_lens, int partition_size,
                            int max_num_partitions, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * pa_append_and_decode -- one decode step in one launch: each sequence's
 * new token is written into the cache and attention is computed over the
 * whole context, new token included.
 *
 * A decode step first appends the new token's K/V to the sequence's last
 * block and then attends over every valid slot ("Efficient Memory
 * Management for LLM Serving with PagedAttention -- in-depth reading",
 * section 3.4, steps 1 and 3; "vLLM PagedAttention source walk-through",
 * section 3.2, append_token: block table[pos / block_size], offset
 * pos % block_size).  This call does both for one new token per sequence at
 * position pos = context_lens[s] - 1, so the result, pools included, is the
 * one of
 *
 *   pa_reshape_and_cache (or pa_reshape_and_cache_fp8) with
 *       slot_mapping[s] = block_tables[s][pos / block_size] * block_size
 *                         + pos % block_size,
 *   then pa_decode (or pa_decode_fp8).
 *
 * The decode's CTA that reads position pos writes the row into the pools
 * and uses it directly, so no separate cache-write launch precedes the
 * decode.
 *
 *   key, value     [num_seqs][num_kv_heads][head_dim] of dtype, the new
 *                  token of each sequence (read only)
 *   k_cache,
 *   v_cache        the pools; the new tokens' slots are written
 *   dtype, kv_dtype, k_scale, v_scale
 *                  as pa_decode_prefix_splitk: 16-bit pools of the query
 *                  type, or E4M3 pools with PA_FP16 queries and new tokens;
 *                  an E4M3 pool stores the code nearest to the float32
 *                  quotient key / k_scale (value / v_scale), as
 *                  pa_reshape_and_cache_fp8 does
 *
 * Precondition: the slot written for sequence s is read by no other
 * sequence of the call (copy-on-write has given a shared block its own copy
 * before a sequence appends to it: "Unveiling the NVIDIA driver stack",
 * section 4; pa_copy_blocks).  Otherwise that other sequence may see the old
 * or the new row.
 *
 * Other arguments as pa_decode.  Device-value outcomes as pa_decode; a
 * sequence with context_lens[s] <= 0, a context length past the table's
 * capacity, or an out-of-pool block id at position pos writes nothing into
 * the pools.
 */
int pa_append_and_decode(void* out, const void* q, const void* key, const void* value, void* k_cache,
                         void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, float scale, int dtype, int kv_dtype,
                         float k_scale, float v_scale, void* stream);

/*
 * pa_append_and_decode_splitk -- pa_append_and_decode with the split-K
 * decode: the new tokens' cache write, then the partitions of
 * pa_decode_splitk, in one launch.  The partition covering position
 * context_lens[s] - 1 writes the row.  Follow with pa_splitk_reduce (same
 * partition_size, max_num_partitions, workspace) on the same stream.
 *
 * Arguments as pa_append_and_decode plus the split-K arguments of
 * pa_decode_splitk; outcomes and precondition as pa_append_and_decode.
 */
int pa_append_and_decode_splitk(void* out, const void* q, const void* key, const void* value, void* k_cache,
                                void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, int num_blocks, float scale, int dtype,
                                int kv_dtype, float k_scale, float v_scale, int partition_size,
                                int max_num_partitions, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill -- paged attention for prompt tokens: whole prompts, or chunks
 * of them appended to a cached context (chunked prefill).
 *
 * Prefill computes attention for many new tokens of a sequence at once; each
 * attends to every earlier position of its sequence and to its own ("in-depth
 * reading", section 5.1, item 5: chunked prefill; "vAttention: dynamic memory
 * management without PagedAttention", the paged prefill kernels it measures).
 * The keys and values come from the pools through the block table, as in
 * decode; write the new tokens' K/V first with pa_reshape_and_cache.
 *
 * Sequence s owns query rows [query_start_loc[s], query_start_loc[s + 1]) of
 * q and out (qlen rows, 0 <= qlen <= context_lens[s]); its last qlen
 * positions are those rows' tokens.  Row i sits at position
 * p = context_lens[s] - qlen + i, and
 *
 *   out[row][h][:] = sum_{k <= p} softmax_k(scale * q[row][h] . K_k) * V_k,
 *
 * with K_k, V_k the pool rows of position k of sequence s, KV head h / G.
 *
 *   q, out            [num_rows][num_heads][head_dim] of dtype, num_rows =
 *                     query_start_loc[num_seqs]
 *   query_start_loc   [num_seqs + 1] int32, non-decreasing, starting at 0
 *   max_query_len     >= every qlen (sizes the grid; rows past it are not
 *                     computed)
 *   head_dim          64 or 128; num_heads / num_kv_heads must divide 128
 *
 * Other arguments as pa_decode.  Scores, softmax and accumulation are
 * float32 (the products accumulate in tensor memory); the attention weights
 * enter P.V rounded to fp16, or for bf16 as a rounded value plus its rounded
 * residual.
 *
 * Device-value outcomes: a context length below qlen or above
 * max_blocks_per_seq * block_size gives NaN in every row of that sequence.  A
 * block id read from the table outside [0, num_blocks) gives NaN in every row
 * of the CTA that reads it: two consecutive tiles of 128 rows (128 / G tokens
 * times the G query heads of a KV head each), so rows of that pair that stop
 * before the bad block are NaN too.  A sequence with qlen <= 0 writes
 * nothing.  Nothing is read out of bounds.
 */
int pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
               const int32_t* query_start_loc, int num_seqs, int num_rows, int max_query_len,
               int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
               float scale, int dtype, void* stream);

/*
 * pa_splitk_reduce -- merge the partitions left by pa_decode_splitk.
 *
 * For each (s, h) whose sequence has P = ceil(context_lens[s] /
 * partition_size) >= 2 partitions:
 *
 *   M = max_p m_p,  w_p = l_p * 2^(m_p - M),
 *   out[s][h][:] = fp16( sum_p w_p * o_p[:] / sum_p w_p ).
 *
 * This is the correction factor exp(old_max - new_max) of the online softmax
 * in "vLLM PagedAttention source walk-through", section 3.4, applied between
 * partitions instead of between blocks.  Sequences with P <= 1, or with an
 * out-of-range context length, are left untouched (pa_decode_splitk already
 * wrote them).  The arguments must match the pa_decode_splitk call that
 * filled the workspace, on the same stream (or ordered after it).
 */
int pa_splitk_reduce(void* out, const void* workspace, size_t workspace_bytes,
                     const int32_t* context_lens, int max_blocks_per_seq, int block_size,
                     int num_seqs, int num_heads, int head_dim, int partition_size,
                     int max_num_partitions, int dtype, void* stream);

/*
 * pa_decode_splitk_static -- pa_decode_splitk followed by pa_splitk_reduce,
 * with the split-K workspace taken from a fixed array inside the library
 * instead of from the caller.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory -- a serving
 * runtime that has reserved nearly all device memory for its KV-cache pool
 * and hands out no scratch, a host program that reaches the library only
 * through this C ABI and owns no GPU allocator, or a decode loop that must
 * not call cudaMalloc (which can synchronise the device).  It allocates
 * nothing: the caller passes inputs and outputs as for pa_decode_splitk
 * (with max_num_partitions = ceil(max_blocks_per_seq * block_size /
 * partition_size)), and the partials go to a file-scope device array of
 * PA_STATIC_SCRATCH_BYTES, which every GPU that loads the library holds
 * until the process exits.
 *
 *  - A batch whose workspace (pa_splitk_workspace_bytes) exceeds
 *    PA_STATIC_SCRATCH_BYTES is rejected with PA_ERR_UNSUPPORTED and a
 *    message; nothing is launched.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and remembers it;
 *    make that first call before any stream capture.  The address is
 *    remembered for the life of the process: after cudaDeviceReset (or
 *    anything else that destroys the device's primary context) it no longer
 *    names the array, so do not call this entry point on that device again.
 *  - Arguments are checked as for pa_decode_splitk first; a valid batch that
 *    is too large for the array is then rejected as below.
 *  - Every call on a device shares the one array and leaves its partials
 *    there.  Nothing in it needs to start at zero: each call writes every
 *    row it later reads.  Calls whose kernels overlap on the GPU (different
 *    streams, or concurrent host threads) race on the array: order them.
 *
 * Result, arguments and device-value outcomes as pa_decode_splitk + reduce.
 */
#define PA_STATIC_SCRATCH_BYTES ((size_t)32 * 1024 * 1024)

int pa_decode_splitk_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            float scale, int dtype, int partition_size, void* stream);

/*
 * FP8 caches.  "PagedAttention: when the KV cache meets OS paging", section
 * 6, stacks FP8 quantisation of the KV cache on the block abstraction: the
 * data are compressed inside each block and the attention kernel
 * dequantises them.  The page fixes no format or scale; these entry points
 * use OCP E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7, 3 fraction
 * bits, no infinities, 0x7F/0xFF NaN, largest finite 448) and one float
 * scale per pool: the element stored for x is
 *
 *     code = E4M3_satfinite( fp32(x) / k_scale )   (v_scale for V),
 *
 * the IEEE float32 quotient rounded to the nearest code, ties to even,
 * finite values beyond 448 saturating to +-448; the element read back is
 * value(code) * k_scale (v_scale).  The pools have the layout of the 16-bit
 * caches with one byte per element.  Queries, new tokens and outputs stay
 * 16-bit.  Scales must be finite and positive (else PA_ERR_INVALID_ARG).
 */

/*
 * pa_reshape_and_cache_fp8 -- pa_reshape_and_cache into E4M3 pools.
 *
 *   key, value        [num_tokens][num_kv_heads][head_dim] of dtype
 *                     (PA_FP16 or PA_BF16)
 *   k_cache, v_cache  [num_blocks][block_size][num_kv_heads][head_dim]
 *                     uint8 E4M3 codes; head_dim a multiple of 16
 *
 * Slots and device-value outcomes as pa_reshape_and_cache.
 */
int pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim, int dtype,
                             float k_scale, float v_scale, void* stream);

/*
 * pa_decode_fp8 -- pa_decode over E4M3 pools: the same attention with
 * K_i = value(k code) * k_scale and V_i = value(v code) * v_scale.  The
 * codes are widened exactly to fp16 inside the kernel; k_scale multiplies
 * the scores and v_scale the output, both in float32.
 *
 *   q, out   [num_seqs][num_heads][head_dim], dtype PA_FP16 (PA_BF16 is
 *            PA_ERR_UNSUPPORTED)
 *
 * Other arguments, supported shapes and device-value outcomes as pa_decode
 * (a NaN code in a valid slot gives NaN in the affected output).
 */
int pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                  int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int dtype, float k_scale, float v_scale,
                  void* stream);

/*
 * pa_decode_splitk_fp8 -- pa_decode_splitk over E4M3 pools.  The workspace
 * holds the scaled float32 partials, so pa_splitk_reduce (dtype PA_FP16)
 * finishes the call unchanged.
 */
int pa_decode_splitk_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, int dtype, float k_scale, float v_scale, int partition_size,
                         int max_num_partitions, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * pa_selftest_wait -- checks, on the device, the bounded wait that every
 * pipeline of this library uses on its mbarriers (TMA copies landing, MMAs
 * completing, softmax threads handing over P): a wait that runs past its
 * limit gives up and reports instead of spinning, so a stage that never
 * completes cannot hang the GPU; the library's kernels then write NaN rows.
 *
 * One warp waits on a phase that nothing completes, with a limit of
 * limit_us microseconds, then on a phase completed by one arrival.
 *
 *   result    device int32 [3], 4-byte aligned: [0] = 1 if the first wait
 *             gave up, [1] = 1 if the second wait returned, [2] = the
 *             microseconds the first wait took (>= limit_us when it gave up)
 *   limit_us  1 .. 10,000,000
 *
 * Asynchronous on `stream`; the device context stays usable afterwards.
 */
int pa_selftest_wait(int32_t* result, unsigned limit_us, void* stream);

/* Fixed text naming a status code. */
const char* pa_status_string(int status);

/* Text of the last error raised on the calling thread ("" if none). */
const char* pa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
