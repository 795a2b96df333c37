// pa_decode.cuh -- paged decode and split-K reduce kernels, templated on the
// element type T (__half or __nv_bfloat16).  Included by one translation unit
// per element type (pa_decode_f16.cu, pa_decode_bf16.cu); everything here has
// internal linkage except what those units export.
//
//  paged_decode_kernel        one CTA per (KV head, partition, sequence);
//                             each warp streams 16-token chunks of its share
//                             of the partition through a private ring of
//                             shared-memory stages filled by TMA tensor copies,
//                             scores the G query heads of the group against
//                             K with m16n8k16 MMAs, runs the online softmax in
//                             float32 and accumulates P.V with MMAs; the warps
//                             are merged in shared memory at the end.  Run as
//                             thread-block clusters, the CTAs of a cluster
//                             split one (sequence, KV head) and merge through
//                             distributed shared memory.
//  splitk_reduce_*_kernel     log-sum-exp merge of the split-K partitions
//
// The method: "vLLM PagedAttention source walk-through", section 3.4 (block
// walk, mask, online softmax with correction factor exp(old_max - new_max));
// "PagedAttention: when the KV cache meets OS paging", sections 3.2 and 5.1
// (the kernel translates logical to physical blocks itself; table entries are
// prefetched so the lookups hide under memory latency); "Unveiling the NVIDIA
// driver stack: GPU page tables and vLLM PagedAttention", sections 6 and 7.3
// (address arithmetic from the physical block id; adjacent threads read
// adjacent bytes).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cooperative_groups.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <type_traits>

#include "pa_launch.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr int CHUNK = 16;                       // tokens per pipeline stage
constexpr int kLongestFirstMax = 256;           // batches the single launch ranks longest first
constexpr uint64_t WAIT_LIMIT_NS = 2000000000;  // 2 s: a stage that takes longer is an error

// ================================================================ decode
struct DecodeParams {
  // Tensor maps over the K and V pools viewed as [N*B rows][Hk][d] (3-D,
  // innermost first: d, Hk, rows) with a box of one 128-byte row segment (64
  // bytes for 64 one-byte dims) x 1 head x 16 rows, swizzled over its width.
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  void* out;        // [S][H][d] of T
  const void* q;    // [S][H][d] of T
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_o;
  float* ws_m;
  float* ws_l;
  int max_blocks_per_seq;
  int num_heads;
  int num_kv_heads;
  int group;
  int block_size;
  int chunks_per_block_log2;  // block_size / 16 is a power of two
  int num_blocks;
  int partition_chunks;
  int max_num_partitions;
  float scale_log2;  // scale * k_scale * log2(e): scores are kept in base-2 units
  float out_scale;   // v_scale of an E4M3 V pool (1 otherwise)
  // Shared-prefix decode: sequences [j * seqs_per_group, (j + 1) * seqs_per_group)
  // form group j, whose first prefix_lens[j] tokens sit in the same blocks.
  const int32_t* prefix_lens;  // null: no shared pass
  int seqs_per_group;
  int members_per_cta;  // shared pass: sequences of a group per CTA
  int subgroups;        // shared pass: CTAs per group along grid z
  int num_seqs;
  // Append (the cache write fused into the decode): sequence s's new token,
  // rows new_k / new_v [S][Hk][d] of T, goes into the pools k_pool / v_pool
  // at the slot of position ctx - 1; E4M3 pools store the code nearest to
  // x / k_scale (x / v_scale).
  const void* new_k;
  const void* new_v;
  void* k_pool;
  void* v_pool;
  float k_scale;
  float v_scale;
};

// MODE_LONGEST_FIRST: a single launch (one CTA per (KV head, sequence)) over
// at most kLongestFirstMax sequences in which CTA z takes the sequence of
// rank z in decreasing context length (ties by index), so that the CTAs left
// for a second wave are the shortest.  Otherwise it is MODE_GRID.  (Llama-3-
// 8B-shaped batch, 64 sequences x 8 KV heads on 456 slots: E4M3 fused step
// 32.7 -> 29.8 us, fp16 decode 52.9 -> 51.9 us.)
enum DecodeMode { MODE_GRID = 0, MODE_CLUSTER = 1, MODE_SHARED = 2, MODE_LONGEST_FIRST = 3 };

// Tokens of a sequence that its group's shared pass covers: the group's
// prefix length lp when it is a positive multiple of the partition size that
// both the sequence and the group's first sequence reach (within the
// table's capacity), else 0.  The shared pass and the per-sequence pass
// both decide with this function, so they always agree.
__device__ __forceinline__ int shared_len(int lp, int ctx, int ctx_lead, int cap, int partition_tokens) {
  const bool ok = lp > 0 && lp % partition_tokens == 0 && lp <= ctx && lp <= ctx_lead && ctx <= cap &&
                  ctx_lead <= cap;
  return ok ? lp : 0;
}

// Shared-memory stage of one 16-token chunk of one KV head: TMA boxes of 16
// rows x 64 dims (128 bytes per row, 2 KB per box), 128-byte swizzled: the
// 16-byte unit u of row r sits at unit u ^ (r % 8).  K boxes first (dims
// 0-63, 64-127, ...), then V boxes.
// E4M3 caches use the same 128-byte box rows (128 dims; 64-byte rows of 64
// dims with a 64-byte swizzle: unit u of row r at u ^ ((r / 2) % 4)).
constexpr int BOX_DIMS = 64;
constexpr int BOX_BYTES = CHUNK * BOX_DIMS * 2;

// Cache element tag for E4M3 codes: one byte per element, one float scale
// per pool.  A 16-bit cache uses the query type T itself.
struct E4M3 {};
template <typename KV>
constexpr bool kIsFp8 = std::is_same<KV, E4M3>::value;
template <typename KV>
constexpr int kElemBytes = kIsFp8<KV> ? 1 : 2;

template <int HEAD_DIM, int NT, int WARPS, int STAGES, int ELEM = 2>
struct DecodeCfg {
  static constexpr int ROW_BYTES = HEAD_DIM * ELEM < 128 ? HEAD_DIM * ELEM : 128;  // bytes per box row
  static constexpr int BOX_ELEMS = ROW_BYTES / ELEM;
  static constexpr int BOX_B = CHUNK * ROW_BYTES;
  static constexpr int DBOX = HEAD_DIM / BOX_ELEMS;  // boxes per row of K (or V)
  static constexpr int HALF_BYTES = DBOX * BOX_B;
  static constexpr int CHUNK_BYTES = 2 * HALF_BYTES;   // K and V of one 16-token chunk
  // chunks per stage: E4M3 stages up to d = 128 hold two chunks (8 KB);
  // d = 256 chunks are 8 KB already
  static constexpr int CPS = (ELEM == 1 && HEAD_DIM <= 128) ? 2 : 1;
  static constexpr int STAGE_BYTES = CPS * CHUNK_BYTES;
  static constexpr int RING_BYTES = WARPS * STAGES * STAGE_BYTES;
  static constexpr int GMAX = NT * 8;
  static constexpr int MO_PITCH = HEAD_DIM + 4;  // floats; spreads the merge writes over banks
  static constexpr int MERGE_BYTES = WARPS * GMAX * MO_PITCH * 4 + 2 * WARPS * GMAX * 4 + WARPS * 4;
  // CTA result shared with the other CTAs of a cluster: o [GMAX][HEAD_DIM], m, l [GMAX]
  static constexpr int CTA_OFFSET = (MERGE_BYTES + 15) / 16 * 16;
  static constexpr int CTA_BYTES = GMAX * HEAD_DIM * 4 + 2 * GMAX * 4;
  static constexpr int TAIL_BYTES = CTA_OFFSET + CTA_BYTES;
  static constexpr int BAR_BYTES = 1024;  // the ring that follows is 1024-byte aligned
  static_assert(WARPS * STAGES * 8 <= BAR_BYTES, "barrier area");
  static_assert(RING_BYTES >= (kLongestFirstMax + 1) * 4, "the longest-first ranking fits in the ring");
  // + 1024 so that the ring can be aligned whatever the base alignment is
  static constexpr int SMEM_BYTES = 1024 + BAR_BYTES + (RING_BYTES > TAIL_BYTES ? RING_BYTES : TAIL_BYTES);
};

// ------------------------------------------------- per-warp attention state
// One warp's running softmax state for the 8*NT query heads of a KV head:
// maxima m and sums l (base 2) per head, and the unnormalised output O^T as
// m16n8k16 accumulator fragments (rows = dims, columns = heads).
template <int HEAD_DIM, int NT>
struct WarpAcc {
  static constexpr int KSTEPS = HEAD_DIM / 16;
  float m[NT][2];
  float l[NT][2];
  float o[KSTEPS][NT][4];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int dm = 0; dm < KSTEPS; ++dm)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[dm][nt][i] = 0.f;
    }
  }
};

// Row of q (and of out) of query j of a CTA whose queries start at sequence
// s0: sequence s0 + j / G, head kvh * G + j % G.  A per-sequence CTA has
// queries j < G, the heads of one group.
__device__ __forceinline__ size_t query_row(int s0, int j, int H, int kvh, int G) {
  return static_cast<size_t>(s0 + j / G) * H + kvh * G + j % G;
}

// Query fragments (B operand of S = K Q^T): lane holds query nt*8 + lane/4,
// dims ks*16 + {2c, 2c+1} and ks*16 + {2c+8, 2c+9} with c = lane % 4;
// queries past nq are zero.
template <int HEAD_DIM, int NT>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[HEAD_DIM / 16][NT][2], const void* q,
                                             int s0, int H, int kvh, int G, int nq, int lane) {
  const int g = lane >> 2;
  const int c4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hq = nt * 8 + g;
    const bool hv = hq < nq;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const uint16_t*>(q) + query_row(s0, hv ? hq : 0, H, kvh, G) * HEAD_DIM);
#pragma unroll
    for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
      qf[ks][nt][0] = hv ? __ldg(qrow + ks * 8 + c4) : 0u;
      qf[ks][nt][1] = hv ? __ldg(qrow + ks * 8 + c4 + 4) : 0u;
    }
  }
}

// Query fragments for E4M3 keys: k-step ks pairs the MMA's k indices
// {2c, 2c+1, 2c+8, 2c+9} with dims ks*16 + 4c .. 4c+3, the order in which
// the key fragments arrive (attend_chunk_e4m3), so each lane loads four
// consecutive dims at once.
template <int HEAD_DIM, int NT>
__device__ __forceinline__ void load_q_frags_e4m3(uint32_t (&qf)[HEAD_DIM / 16][NT][2], const void* q, int s0,
                                                  int H, int kvh, int G, int nq, int lane) {
  const int g = lane >> 2;
  const int c4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hq = nt * 8 + g;
    const bool hv = hq < nq;
    const uint2* qrow = reinterpret_cast<const uint2*>(
        static_cast<const uint16_t*>(q) + query_row(s0, hv ? hq : 0, H, kvh, G) * HEAD_DIM);
#pragma unroll
    for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
      const uint2 v = hv ? __ldg(qrow + ks * 4 + c4) : make_uint2(0u, 0u);
      qf[ks][nt][0] = v.x;
      qf[ks][nt][1] = v.y;
    }
  }
}

// Online-softmax step over NSUB 16-token chunks whose scores S[16 tokens][8*NT
// heads] are in sacc[sb] (m16n8 accumulator layout: token g holds elements
// 0-1, token g + 8 elements 2-3), of which the first valid[sb] tokens belong
// to the sequence: updates the running maxima and sums once for all of them,
// rescales the accumulators when a maximum moves, and returns each chunk's
// P^T as B fragments (bf16: also the residual P - bf16(P) in `pl`).
template <typename T, int HEAD_DIM, int NT, int NSUB>
__device__ __forceinline__ void softmax_step(WarpAcc<HEAD_DIM, NT>& acc, const float (&sacc)[NSUB][NT][4],
                                             const int (&valid)[NSUB], float sl2, int lane,
                                             uint32_t (&pb)[NSUB][NT][2], uint32_t (&pl)[NSUB][NT][2]) {
  constexpr int KSTEPS = HEAD_DIM / 16;
  const int g = lane >> 2;
  constexpr bool kSplitP = !std::is_same<T, __half>::value;  // bf16: P = P_hi + P_lo
  static_assert(!kSplitP || NSUB == 1, "bf16 takes one chunk per step");
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // base 2; slots past the context are excluded by select
    float x[NSUB][4];
#pragma unroll
    for (int sb = 0; sb < NSUB; ++sb) {
      const bool v0 = g < valid[sb];
      const bool v1 = g + 8 < valid[sb];
      x[sb][0] = v0 ? sacc[sb][nt][0] * sl2 : -INFINITY;
      x[sb][1] = v0 ? sacc[sb][nt][1] * sl2 : -INFINITY;
      x[sb][2] = v1 ? sacc[sb][nt][2] * sl2 : -INFINITY;
      x[sb][3] = v1 ? sacc[sb][nt][3] * sl2 : -INFINITY;
    }
    float mx0 = fmaxf(x[0][0], x[0][2]);
    float mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
    for (int sb = 1; sb < NSUB; ++sb) {
      mx0 = fmaxf(mx0, fmaxf(x[sb][0], x[sb][2]));
      mx1 = fmaxf(mx1, fmaxf(x[sb][1], x[sb][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, off));
    }
    const float mn0 = fmaxf(acc.m[nt][0], mx0);
    const float mn1 = fmaxf(acc.m[nt][1], mx1);
    const float cr0 = ex2(acc.m[nt][0] - mn0);
    const float cr1 = ex2(acc.m[nt][1] - mn1);
    const bool grew = __any_sync(FULL_MASK, (mn0 != acc.m[nt][0]) | (mn1 != acc.m[nt][1]));
    acc.m[nt][0] = mn0;
    acc.m[nt][1] = mn1;
    float sum0 = 0.f, sum1 = 0.f;
    uint32_t lo[NSUB], hi[NSUB];
#pragma unroll
    for (int sb = 0; sb < NSUB; ++sb) {
      const float p0 = ex2(x[sb][0] - mn0), p1 = ex2(x[sb][1] - mn1);  // token g
      const float p2 = ex2(x[sb][2] - mn0), p3 = ex2(x[sb][3] - mn1);  // token g + 8
      lo[sb] = pack2<T>(p0, p1);
      hi[sb] = pack2<T>(p2, p3);
      const float2 flo = unpack2<T>(lo[sb]);
      const float2 fhi = unpack2<T>(hi[sb]);
      if constexpr (kSplitP) {
        // bf16 keeps 8 significant bits: P also goes in as the rounded residual,
        // so P_hi + P_lo carries about 16 bits and the sum uses P itself
        pl[sb][nt][0] = movmatrix_trans(pack2<T>(p0 - flo.x, p1 - flo.y));
        pl[sb][nt][1] = movmatrix_trans(pack2<T>(p2 - fhi.x, p3 - fhi.y));
        sum0 = sb == 0 ? (p0 + p2) : sum0 + (p0 + p2);
        sum1 = sb == 0 ? (p1 + p3) : sum1 + (p1 + p3);
      } else {
        // the running sum adds the same rounded weights that multiply V
        sum0 = sb == 0 ? (flo.x + fhi.x) : sum0 + (flo.x + fhi.x);
        sum1 = sb == 0 ? (flo.y + fhi.y) : sum1 + (flo.y + fhi.y);
      }
    }
    acc.l[nt][0] = acc.l[nt][0] * cr0 + sum0;
    acc.l[nt][1] = acc.l[nt][1] * cr1 + sum1;
    if (grew) {  // a running maximum moved: rescale the accumulators
#pragma unroll
      for (int dm = 0; dm < KSTEPS; ++dm) {
        acc.o[dm][nt][0] *= cr0;
        acc.o[dm][nt][1] *= cr1;
        acc.o[dm][nt][2] *= cr0;
        acc.o[dm][nt][3] *= cr1;
      }
    }
#pragma unroll
    for (int sb = 0; sb < NSUB; ++sb) {
      pb[sb][nt][0] = movmatrix_trans(lo[sb]);  // P^T tokens 0-7 as the B fragment
      pb[sb][nt][1] = movmatrix_trans(hi[sb]);  // P^T tokens 8-15
    }
  }
}

// Attend one 16-token chunk held in shared memory at `kb` (K boxes, then V
// boxes at kb + half_bytes; 128-byte swizzle), of which the first `valid`
// tokens belong to the sequence.  Updates the warp's running state.
template <typename T, int HEAD_DIM, int NT>
__device__ __forceinline__ void attend_chunk(WarpAcc<HEAD_DIM, NT>& acc,
                                             const uint32_t (&qf)[HEAD_DIM / 16][NT][2], uint32_t kb,
                                             uint32_t half_bytes, int valid, float sl2, int lane) {
  constexpr int KSTEPS = HEAD_DIM / 16;
  const int c4 = lane & 3;
  const uint32_t vb = kb + half_bytes;
  constexpr bool kSplitP = !std::is_same<T, __half>::value;

  // S[16 tokens][8*NT heads] = K Q^T, as two independent MMA chains (even
  // and odd k-steps) that are added at the end
  float sacc[1][NT][4], sacc2[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[0][nt][i] = sacc2[nt][i] = 0.f;
  // lane supplies row (lane & 15) at 16-byte unit 2*(ks%4) + lane/16 of box ks/4
  const uint32_t ka = kb + (lane & 15) * 128;
  const uint32_t kx = lane & 7;
#pragma unroll
  for (int ks = 0; ks < KSTEPS; ++ks) {
    uint32_t a[4];
    const uint32_t unit = ((ks & 3) * 2 + (lane >> 4)) ^ kx;
    ldsm_x4(a, ka + (ks >> 2) * BOX_BYTES + unit * 16);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      mma_16816<T>((ks & 1) ? sacc2[nt] : sacc[0][nt], a, qf[ks][nt][0], qf[ks][nt][1]);
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[0][nt][i] += sacc2[nt][i];

  uint32_t pb1[1][NT][2], pl1[1][NT][2];
  const int valid1[1] = {valid};
  softmax_step<T, HEAD_DIM, NT, 1>(acc, sacc, valid1, sl2, lane, pb1, pl1);
  const uint32_t(&pb)[NT][2] = pb1[0];
  const uint32_t(&pl)[NT][2] = pl1[0];

  // O^T[d][heads] += V^T P^T; V rows past the context are zeroed by select
  const int t0 = 2 * c4;
  const uint32_t mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
  const uint32_t mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
  // lane supplies token row (lane & 7) + 8*(lane/16) at unit 2*(dm%4) + (lane/8)%2
  const uint32_t va = vb + ((lane & 7) + ((lane >> 4) << 3)) * 128;
  const uint32_t vsel = (lane >> 3) & 1;
  const uint32_t vx = lane & 7;
  if (valid == CHUNK) {
#pragma unroll
    for (int dm = 0; dm < KSTEPS; ++dm) {
      uint32_t a[4];
      ldsm_x4_trans(a, va + (dm >> 2) * BOX_BYTES + ((((dm & 3) * 2) + vsel) ^ vx) * 16);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_16816<T>(acc.o[dm][nt], a, pb[nt][0], pb[nt][1]);
        if constexpr (kSplitP) mma_16816<T>(acc.o[dm][nt], a, pl[nt][0], pl[nt][1]);
      }
    }
  } else {  // the last chunk of the sequence
#pragma unroll
    for (int dm = 0; dm < KSTEPS; ++dm) {
      uint32_t a[4];
      ldsm_x4_trans(a, va + (dm >> 2) * BOX_BYTES + ((((dm & 3) * 2) + vsel) ^ vx) * 16);
      a[0] &= mlo;
      a[1] &= mlo;
      a[2] &= mhi;
      a[3] &= mhi;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_16816<T>(acc.o[dm][nt], a, pb[nt][0], pb[nt][1]);
        if constexpr (kSplitP) mma_16816<T>(acc.o[dm][nt], a, pl[nt][0], pl[nt][1]);
      }
    }
  }
}

// Byte offset of 16-byte unit `unit` of row `row` in a swizzled box of
// ROW_BYTES-byte rows.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swizzled(uint32_t row, uint32_t unit) {
  if constexpr (ROW_BYTES == 128) {
    return row * 128u + ((unit ^ (row & 7u)) << 4);
  } else {
    return row * 64u + ((unit ^ ((row >> 1) & 3u)) << 4);
  }
}

// O^T += V^T P^T over E4M3 codes.  ldmatrix.trans of 16-bit pairs hands a
// lane the codes of tokens 2c, 2c+1 at dims 2g, 2g+1 of a 16-dim unit; a byte
// permute regroups them by dim, so MMA row g stands for dim 2g of the unit and
// row g + 8 for dim 2g + 1.  MASK: tokens past `valid` are zeroed by select.
template <int HEAD_DIM, int NT, int ROW_BYTES, bool MASK>
__device__ __forceinline__ void pv_e4m3(WarpAcc<HEAD_DIM, NT>& acc, const uint32_t (&pb)[NT][2], uint32_t vaddr,
                                        uint32_t tok, uint32_t uo, uint32_t mlo, uint32_t mhi) {
  constexpr int UNITS = ROW_BYTES / 16;
  constexpr int BOXB = CHUNK * ROW_BYTES;
#pragma unroll
  for (int u = 0; u < HEAD_DIM / 16; u += 2) {
    uint32_t r[4];  // tokens 0-7 / 8-15 of unit u, then of unit u + 1
    ldsm_x4_trans(r, vaddr + (u / UNITS) * BOXB + swizzled<ROW_BYTES>(tok, (u % UNITS) + uo));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t a[4];  // (tok 2c, 2c+1) at dim 2g, at dim 2g+1; then tokens 2c+8, 2c+9
      e4m3x4_to_half2x2(__byte_perm(r[2 * h], 0u, 0x3120), a[0], a[1]);
      e4m3x4_to_half2x2(__byte_perm(r[2 * h + 1], 0u, 0x3120), a[2], a[3]);
      if constexpr (MASK) {
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_f16_16816(acc.o[u + h][nt], a, pb[nt][0], pb[nt][1]);
    }
  }
}

// S = K Q^T for one 16-token chunk of E4M3 keys at `kb`.  A lane receives
// the codes of tokens g and g + 8 at dims 4c .. 4c+3 of a unit; their low
// pair fills k indices 2c, 2c+1 and their high pair 2c+8, 2c+9
// (load_q_frags_e4m3 orders q the same way).  Even and odd k-steps run as
// two MMA chains that are added at the end.
template <int HEAD_DIM, int NT, int ROW_BYTES>
__device__ __forceinline__ void qk_e4m3(float (&sacc)[NT][4], const uint32_t (&qf)[HEAD_DIM / 16][NT][2],
                                        uint32_t kb, uint32_t tok, uint32_t uo) {
  constexpr int UNITS = ROW_BYTES / 16;
  constexpr int BOXB = CHUNK * ROW_BYTES;
  float sacc2[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[nt][i] = sacc2[nt][i] = 0.f;
#pragma unroll
  for (int u = 0; u < HEAD_DIM / 16; u += 2) {
    uint32_t r[4];
    ldsm_x4(r, kb + (u / UNITS) * BOXB + swizzled<ROW_BYTES>(tok, (u % UNITS) + uo));
    uint32_t a[4], b[4];  // k-step u from r[0], r[1]; k-step u + 1 from r[2], r[3]
    e4m3x4_to_half2x2(r[0], a[0], a[2]);
    e4m3x4_to_half2x2(r[1], a[1], a[3]);
    e4m3x4_to_half2x2(r[2], b[0], b[2]);
    e4m3x4_to_half2x2(r[3], b[1], b[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_f16_16816(sacc[nt], a, qf[u][nt][0], qf[u][nt][1]);
      mma_f16_16816(sacc2[nt], b, qf[u + 1][nt][0], qf[u + 1][nt][1]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[nt][i] += sacc2[nt][i];
}

// Lane roles shared by the E4M3 ldmatrix loads: a lane supplies token row
// `tok` of unit (u + uo), so the four matrices are tokens {0-7, 8-15} x
// units {u, u + 1}.
__device__ __forceinline__ uint32_t e4m3_tok(int lane) { return (lane & 7) + (((lane >> 3) & 1) << 3); }
__device__ __forceinline__ uint32_t e4m3_uo(int lane) { return static_cast<uint32_t>(lane) >> 4; }

// Select masks for the V fragments of a chunk with `valid` tokens: the
// halves of tokens (2c, 2c+1) and (2c+8, 2c+9).
__device__ __forceinline__ void v_masks(int valid, int lane, uint32_t& mlo, uint32_t& mhi) {
  const int t0 = 2 * (lane & 3);
  mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
  mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
}

// attend_chunk for one 16-token chunk of E4M3 K and V boxes (codes widened
// exactly to float16 in registers; the pool scales are applied outside:
// k_scale in `sl2`, v_scale to the final output).  K boxes at `kb`, V boxes
// at kb + half_bytes.
template <int HEAD_DIM, int NT, int ROW_BYTES>
__device__ __forceinline__ void attend_chunk_e4m3(WarpAcc<HEAD_DIM, NT>& acc,
                                                  const uint32_t (&qf)[HEAD_DIM / 16][NT][2], uint32_t kb,
                                                  uint32_t half_bytes, int valid, float sl2, int lane) {
  const uint32_t tok = e4m3_tok(lane), uo = e4m3_uo(lane);
  float sacc[1][NT][4];
  qk_e4m3<HEAD_DIM, NT, ROW_BYTES>(sacc[0], qf, kb, tok, uo);
  uint32_t pb[1][NT][2], pl[1][NT][2];
  const int valid1[1] = {valid};
  softmax_step<__half, HEAD_DIM, NT, 1>(acc, sacc, valid1, sl2, lane, pb, pl);
  uint32_t mlo, mhi;
  v_masks(valid, lane, mlo, mhi);
  if (valid == CHUNK) {
    pv_e4m3<HEAD_DIM, NT, ROW_BYTES, false>(acc, pb[0], kb + half_bytes, tok, uo, mlo, mhi);
  } else {  // the last chunk of the sequence
    pv_e4m3<HEAD_DIM, NT, ROW_BYTES, true>(acc, pb[0], kb + half_bytes, tok, uo, mlo, mhi);
  }
}

// Two 16-token chunks of E4M3 codes in one stage (the first at `kb`, the
// second at kb + chunk_bytes; K then V boxes in each), scored and folded
// into the running softmax in one step.  The first chunk is full; the second
// has `valid2` tokens.
template <int HEAD_DIM, int NT, int ROW_BYTES>
__device__ __forceinline__ void attend_pair_e4m3(WarpAcc<HEAD_DIM, NT>& acc,
                                                 const uint32_t (&qf)[HEAD_DIM / 16][NT][2], uint32_t kb,
                                                 uint32_t chunk_bytes, uint32_t half_bytes, int valid2, float sl2,
                                                 int lane) {
  const uint32_t tok = e4m3_tok(lane), uo = e4m3_uo(lane);
  const uint32_t kb2 = kb + chunk_bytes;
  float sacc[2][NT][4];
  qk_e4m3<HEAD_DIM, NT, ROW_BYTES>(sacc[0], qf, kb, tok, uo);
  qk_e4m3<HEAD_DIM, NT, ROW_BYTES>(sacc[1], qf, kb2, tok, uo);
  uint32_t pb[2][NT][2], pl[2][NT][2];
  const int valid[2] = {CHUNK, valid2};
  softmax_step<__half, HEAD_DIM, NT, 2>(acc, sacc, valid, sl2, lane, pb, pl);
  uint32_t mlo, mhi;
  v_masks(valid2, lane, mlo, mhi);
  pv_e4m3<HEAD_DIM, NT, ROW_BYTES, false>(acc, pb[0], kb + half_bytes, tok, uo, mlo, mhi);
  if (valid2 == CHUNK) {
    pv_e4m3<HEAD_DIM, NT, ROW_BYTES, false>(acc, pb[1], kb2 + half_bytes, tok, uo, mlo, mhi);
  } else {
    pv_e4m3<HEAD_DIM, NT, ROW_BYTES, true>(acc, pb[1], kb2 + half_bytes, tok, uo, mlo, mhi);
  }
}

// ------------------------------------------------------- the fused append
// A sequence's new K and V rows for one KV head, as the 16-byte units (8
// elements of T) that the lanes of one warp hold: unit x < U of the K row,
// then the V row; lane i holds units i, i + 32, ...
template <int HEAD_DIM>
struct AppendRow {
  static constexpr int U = HEAD_DIM / 8;        // units per row
  static constexpr int NV = (2 * U + 31) / 32;  // units per lane
  uint4 v[NV];
};

template <int HEAD_DIM>
__device__ __forceinline__ void append_load(AppendRow<HEAD_DIM>& a, const DecodeParams& p, int s, int kvh,
                                            int lane) {
  constexpr int U = AppendRow<HEAD_DIM>::U;
  const size_t row = (static_cast<size_t>(s) * p.num_kv_heads + kvh) * U;
  const uint4* k = static_cast<const uint4*>(p.new_k) + row;
  const uint4* v = static_cast<const uint4*>(p.new_v) + row;
#pragma unroll
  for (int j = 0; j < AppendRow<HEAD_DIM>::NV; ++j) {
    const int x = lane + 32 * j;
    if (x < 2 * U) a.v[j] = __ldg((x < U ? k : v) + (x % U));
  }
}

// Write the rows into the pools at pool row `prow` (block * B + offset) and
// into the landed shared-memory chunk at `cbase` (K boxes, V boxes at
// + half_bytes), token row r, where TMA put what the pool held before the
// write.  16-bit pools take the bits; E4M3 pools take, per element, the code
// nearest to the float32 quotient x / scale (the conversion the E4M3 cache
// write uses), so both hold what a separate cache write would leave.
template <typename KV, int HEAD_DIM, int ROW_BYTES, int BOX_B, int HALF_BYTES>
__device__ __forceinline__ void append_store(const AppendRow<HEAD_DIM>& a, const DecodeParams& p, int64_t prow,
                                             int kvh, uint32_t cbase, uint32_t r, int lane) {
  constexpr int U = AppendRow<HEAD_DIM>::U;
  constexpr int UPB = ROW_BYTES / 16;  // 16-byte units per box row
#pragma unroll
  for (int j = 0; j < AppendRow<HEAD_DIM>::NV; ++j) {
    const int x = lane + 32 * j;
    if (x >= 2 * U) continue;
    const int which = x >= U ? 1 : 0;  // 0: K, 1: V
    const int u = x % U;
    const int64_t grow = prow * p.num_kv_heads + kvh;  // the (slot, head) row of the pool
    if constexpr (!kIsFp8<KV>) {
      uint4* g = static_cast<uint4*>(which ? p.v_pool : p.k_pool) + grow * U + u;
      *g = a.v[j];
      const uint32_t sa = cbase + which * HALF_BYTES + (u / UPB) * BOX_B + swizzled<ROW_BYTES>(r, u % UPB);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sa), "r"(a.v[j].x), "r"(a.v[j].y),
                   "r"(a.v[j].z), "r"(a.v[j].w)
                   : "memory");
    } else {
      const float sc = which ? p.v_scale : p.k_scale;
      const uint32_t w[4] = {a.v[j].x, a.v[j].y, a.v[j].z, a.v[j].w};
      uint32_t o[2] = {0u, 0u};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float2 f = unpack_half2(w[jj]);
        const uint32_t c0 = float_to_e4m3_sat(__fdiv_rn(f.x, sc));
        const uint32_t c1 = float_to_e4m3_sat(__fdiv_rn(f.y, sc));
        o[jj >> 1] |= (c0 | (c1 << 8)) << ((jj & 1) * 16);
      }
      uint2* g = static_cast<uint2*>(which ? p.v_pool : p.k_pool) + grow * U + u;  // 8 codes per unit
      *g = make_uint2(o[0], o[1]);
      const int cu = u >> 1;  // the 16-code unit of the row holding these 8 codes
      const uint32_t sa =
          cbase + which * HALF_BYTES + (cu / UPB) * BOX_B + swizzled<ROW_BYTES>(r, cu % UPB) + (u & 1) * 8;
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(sa), "r"(o[0]), "r"(o[1]) : "memory");
    }
  }
}

// The fused cache write of one warp's new-token chunk: load the rows, store
// them into the pools and over row r of the landed chunk at `cbase`.  Kept
// out of line: it runs once per (sequence, KV head), and inlined into the
// chunk loop it would raise the register count of the whole kernel.
template <typename KV, int HEAD_DIM, int ROW_BYTES, int BOX_B, int HALF_BYTES>
__device__ __noinline__ void append_chunk_row(const DecodeParams& p, int s, int kvh, int64_t prow, uint32_t cbase,
                                              uint32_t r, int lane) {
  AppendRow<HEAD_DIM> nv;
  append_load<HEAD_DIM>(nv, p, s, kvh, lane);
  append_store<KV, HEAD_DIM, ROW_BYTES, BOX_B, HALF_BYTES>(nv, p, prow, kvh, cbase, r, lane);
}

// Sum the per-lane partial running sums over the 8 row groups of the warp.
template <int HEAD_DIM, int NT>
__device__ __forceinline__ void reduce_warp_sums(WarpAcc<HEAD_DIM, NT>& acc) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) acc.l[nt][j] += __shfl_xor_sync(FULL_MASK, acc.l[nt][j], off);
}

// Store one warp's state in the merge area: o [GMAX][mo_pitch] floats, m and
// l [GMAX] (call after reduce_warp_sums).  Accumulator row r of k-step dm is
// dim dm*16 + r, or with E4M3 values (DIM_PAIRS) dim dm*16 + 2(r % 8) + r / 8.
template <int HEAD_DIM, int NT, bool DIM_PAIRS = false>
__device__ __forceinline__ void store_warp_state(const WarpAcc<HEAD_DIM, NT>& acc, float* mo, float* mm,
                                                 float* ml, int mo_pitch, int lane) {
  const int g = lane >> 2;
  const int c4 = lane & 3;
#pragma unroll
  for (int dm = 0; dm < HEAD_DIM / 16; ++dm)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int head = nt * 8 + 2 * c4 + (i & 1);
        const int d = DIM_PAIRS ? dm * 16 + 2 * g + (i >> 1) : dm * 16 + g + (i >> 1) * 8;
        mo[head * mo_pitch + d] = acc.o[dm][nt][i];
      }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        mm[nt * 8 + 2 * c4 + j] = acc.m[nt][j];
        ml[nt * 8 + 2 * c4 + j] = acc.l[nt][j];
      }
  }
}

// MODE_GRID: CTA (kvh, part, s) covers partition `part` of partition_chunks
//   chunks; a sequence with one partition writes `out`, otherwise the
//   partition's (o, m, l) go to the split-K workspace.  With prefix_lens set,
//   the partitions that the shared pass covers are skipped.
// MODE_CLUSTER: gridDim.y CTAs form a cluster per (kvh, s); CTA `part`
//   takes chunks [part * n / C, (part + 1) * n / C) of the sequence's n chunks
//   and the cluster merges the C results into `out`.
// MODE_SHARED: CTA (kvh, part, z) covers partition `part` of the shared
//   prefix of group z / subgroups for members_per_cta of its sequences
//   (subgroup z % subgroups): it reads the prefix through the group's first
//   table row once and scores every member's queries against it, writing
//   each member's partition row (or `out` for a one-partition sequence).
// KV: the cache element type, T or E4M3.
// APPEND: the cache write of each sequence's new token is fused in.  The
//   warp that holds the chunk of position ctx - 1 (one per sequence and KV
//   head, in the CTA covering the sequence's last chunk) writes the new K/V
//   row into the pools at that position's slot and over the same row of its
//   landed stage, then attends as usual: the result is the one of a separate
//   cache write followed by the decode.  No other CTA reads that slot.
template <typename T, typename KV, int HEAD_DIM, int NT, int WARPS, int STAGES, int MODE, bool APPEND>
__device__ __forceinline__ void decode_cta(const DecodeParams& p) {
  constexpr bool CLUSTER = MODE == MODE_CLUSTER;
  constexpr bool SHARED = MODE == MODE_SHARED;
  constexpr bool LONGEST = MODE == MODE_LONGEST_FIRST;
  static_assert(!(APPEND && SHARED), "the shared pass does not write the cache");
  constexpr bool FP8 = kIsFp8<KV>;
  static_assert(!FP8 || std::is_same<T, __half>::value, "E4M3 caches take float16 queries");
  using Cfg = DecodeCfg<HEAD_DIM, NT, WARPS, STAGES, kElemBytes<KV>>;
  constexpr int KSTEPS = HEAD_DIM / 16;
  constexpr int GMAX = Cfg::GMAX;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // swizzled TMA destinations must be 1024-byte aligned
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + Cfg::BAR_BYTES;

  const int kvh = blockIdx.x;
  const int part = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int H = p.num_heads;

  // The previous kernel on the stream (typically the cache write) may still
  // be running: everything up to here overlapped with its tail.
  grid_dependency_wait();

  // s: the sequence whose table row the CTA reads; ctx: the tokens of that
  // row it covers; queries j < nq belong to sequence s0 + j / G (query_row).
  // Loads that do not depend on the context length go out first, so that
  // their latencies overlap with the one of context_lens[s].
  const int cap = p.max_blocks_per_seq * p.block_size;
  const int partition_tokens = p.partition_chunks * CHUNK;
  int s, s0, ctx, nq = G;
  int lp = 0, ctx_lead = 0;  // the group's prefix length and first sequence's context
  if constexpr (SHARED) {
    const int gi = static_cast<int>(blockIdx.z) / p.subgroups;
    const int lead = gi * p.seqs_per_group;
    s0 = lead + (static_cast<int>(blockIdx.z) - gi * p.subgroups) * p.members_per_cta;
    const int nm = min(min(lead + p.seqs_per_group, p.num_seqs) - s0, p.members_per_cta);
    lp = __ldg(p.prefix_lens + gi);
    ctx_lead = __ldg(p.context_lens + lead);
    s = lead;
    ctx = shared_len(lp, ctx_lead, ctx_lead, cap, partition_tokens);
    nq = nm > 0 ? nm * G : 0;
    if (nq == 0 || ctx == 0) {  // no member here, or the group shares nothing
      allow_dependent_launch();
      return;
    }
  } else {
    s = static_cast<int>(blockIdx.z);
    if constexpr (LONGEST) {
      // rank every context length against the others in shared memory (the
      // ring is not in use yet); the thread whose sequence has rank z names it
      int* lens = reinterpret_cast<int*>(ring);
      int* pick = lens + kLongestFirstMax;
      const int S = p.num_seqs;
      for (int t = threadIdx.x; t < S; t += WARPS * 32) lens[t] = __ldg(p.context_lens + t);
      __syncthreads();
      for (int t = threadIdx.x; t < S; t += WARPS * 32) {
        const int ct = lens[t];
        int rank = 0;
        for (int j = 0; j < S; ++j) {
          const int cj = lens[j];
          rank += (cj > ct) | ((cj == ct) & (j < t));
        }
        if (rank == s) *pick = t;
      }
      __syncthreads();
      s = *pick;
      ctx = lens[s];
      __syncthreads();  // the ring is free again before any copy lands in it
    }
    s0 = s;
    if (!CLUSTER && p.prefix_lens != nullptr) {
      const int gi = s / p.seqs_per_group;
      lp = __ldg(p.prefix_lens + gi);
      ctx_lead = __ldg(p.context_lens + gi * p.seqs_per_group);
    }
    if constexpr (!LONGEST) ctx = __ldg(p.context_lens + s);
  }
  const int cpb_log2 = p.chunks_per_block_log2;
  const int table_chunks = p.max_blocks_per_seq << cpb_log2;
  const bool ctx_bad = ctx < 0 || ctx > cap;
  const int nchunks = ctx_bad ? 0 : (ctx + CHUNK - 1) / CHUNK;
  const int nclu = CLUSTER ? static_cast<int>(gridDim.y) : 1;
  // The split-K chunk range is known before the context length arrives; the
  // cluster split depends on it.
  const int c0 = CLUSTER ? static_cast<int>((static_cast<int64_t>(part) * nchunks) / nclu)
                         : part * p.partition_chunks;
  const int cmax = CLUSTER ? static_cast<int>((static_cast<int64_t>(part + 1) * nchunks) / nclu)
                           : min(c0 + p.partition_chunks, table_chunks);  // chunks the table can hold
  const int first = c0 + warp;
  const int nk_cap = first < cmax ? (cmax - first + WARPS - 1) / WARPS : 0;

  uint32_t qf[KSTEPS][NT][2];
  if constexpr (FP8) {
    load_q_frags_e4m3<HEAD_DIM, NT>(qf, p.q, s0, H, kvh, G, nq, lane);
  } else {
    load_q_frags<HEAD_DIM, NT>(qf, p.q, s0, H, kvh, G, nq, lane);
  }

  // ---- block-table window: lane j holds the physical block of this warp's
  //      chunk (kbase + j); the next window is fetched 32 chunks ahead.  Only
  //      entries inside the table row are read; those past the context are
  //      fetched but never used.
  const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
  auto win_load = [&](int kbase) -> int {
    const int k = kbase + lane;
    if (k >= nk_cap) return 0;
    return __ldg(bt + ((first + k * WARPS) >> cpb_log2));
  };
  int win_cur = win_load(0);
  int win_nxt = win_load(32);

  uint64_t* wbar = bars + warp * STAGES;
  uint8_t* wring = ring + warp * STAGES * Cfg::STAGE_BYTES;
  if (lane == 0) {
    for (int i = 0; i < STAGES; ++i) mbar_init(&wbar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int nparts = CLUSTER ? nclu : (nchunks + p.partition_chunks - 1) / p.partition_chunks;

  if constexpr (MODE == MODE_GRID) {
    // partitions of a shared prefix are written by the shared pass
    if (part * partition_tokens < shared_len(lp, ctx, ctx_lead, cap, partition_tokens)) {
      allow_dependent_launch();
      return;
    }
  }

  if (nchunks == 0) {
    // Empty sequence -> zeros; impossible context length -> NaN.  Written once.
    if (part == 0) {
      const T v = to_elem<T>(ctx_bad ? NAN : 0.f);
      T* o = static_cast<T*>(p.out) + (static_cast<size_t>(s) * H + kvh * G) * HEAD_DIM;
      for (int i = threadIdx.x; i < G * HEAD_DIM; i += WARPS * 32) o[i] = v;
    }
    allow_dependent_launch();
    return;  // in a cluster every CTA takes this exit together
  }
  if (!CLUSTER && part >= nparts) {
    allow_dependent_launch();
    return;
  }
  const bool single = (MODE == MODE_GRID || LONGEST) && nparts == 1;
  const int c1 = CLUSTER ? cmax : min(c0 + p.partition_chunks, nchunks);
  const int nk = first < c1 ? (c1 - first + WARPS - 1) / WARPS : 0;  // <= nk_cap

  // Append: the warp-local index of the chunk holding position ctx - 1 (the
  // sequence's last chunk) if this warp holds it, else -1; its physical block
  // is taken when the chunk is issued (-1 if outside the pool: nothing is
  // written and the result is NaN, as after a skipped cache write).
  int app_k = -1;
  int app_phys = -1;
  if constexpr (APPEND) {
    const int c_last = nchunks - 1;  // nchunks > 0 here
    if (c_last >= first && c_last < c1 && (c_last - first) % WARPS == 0) app_k = (c_last - first) / WARPS;
  }

  // Shared pass: members whose table entries over this partition differ from
  // the first sequence's get NaN (one bit per member of the CTA).
  int* mismatch = reinterpret_cast<int*>(smem + Cfg::BAR_BYTES - sizeof(int));
  if constexpr (SHARED) {
    static_assert(WARPS * STAGES * 8 + sizeof(int) <= Cfg::BAR_BYTES, "barrier area");
    if (threadIdx.x == 0) *mismatch = 0;
    __syncthreads();
    const int blk0 = c0 >> cpb_log2;
    const int nblk = ((c1 - 1) >> cpb_log2) - blk0 + 1;
    const int nm = nq / G;
    const int32_t* lead_row = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq + blk0;
    for (int i = threadIdx.x; i < nm * nblk; i += WARPS * 32) {
      const int mi = i / nblk;
      const int b = i - mi * nblk;
      const int32_t* row = p.block_tables + static_cast<size_t>(s0 + mi) * p.max_blocks_per_seq + blk0;
      if (__ldg(row + b) != __ldg(lead_row + b)) atomicOr(mismatch, 1 << mi);
    }
  }

  // A stage holds CPS of the warp's chunks (its k-th chunk is chunk
  // first + k * WARPS of the range); `issued` and `consumed` count stages.
  constexpr int CPS = Cfg::CPS;
  const int nst = (nk + CPS - 1) / CPS;
  int issued = 0;
  bool bad = false;

  auto issue_next = [&]() {
    const int it = issued;
    const int slot = it % STAGES;
    const int nload = min(CPS, nk - it * CPS);  // >= 1
    uint8_t* dst = wring + slot * Cfg::STAGE_BYTES;
    if (lane == 0) mbar_arrive_expect_tx(&wbar[slot], nload * Cfg::CHUNK_BYTES);
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      const int k = it * CPS + j;
      if (j > 0 && k >= nk) break;  // warp-uniform
      if (k > 0 && (k & 31) == 0) {
        win_cur = win_nxt;
        win_nxt = win_load(k + 32);
      }
      int phys = __shfl_sync(FULL_MASK, win_cur, k & 31);
      const bool in_pool = static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
      if constexpr (APPEND) {
        if (k == app_k) app_phys = in_pool ? phys : -1;
      }
      if (!in_pool) {
        bad = true;  // never read outside the pool; the result becomes NaN
        phys = 0;
      }
      const int ch = first + k * WARPS;
      const int row0 = (ch & ((1 << cpb_log2) - 1)) * CHUNK;
      if (lane == 0) {
        uint8_t* cd = dst + j * Cfg::CHUNK_BYTES;
        const int y = phys * p.block_size + row0;  // pool row of the chunk's first token
#pragma unroll
        for (int b = 0; b < Cfg::DBOX; ++b) {
          tma_load_3d(cd + b * Cfg::BOX_B, &p.tmap_k, b * Cfg::BOX_ELEMS, kvh, y, &wbar[slot]);
          tma_load_3d(cd + Cfg::HALF_BYTES + b * Cfg::BOX_B, &p.tmap_v, b * Cfg::BOX_ELEMS, kvh, y, &wbar[slot]);
        }
      }
    }
    ++issued;
  };

#pragma unroll 1
  for (int i = 0; i < STAGES && i < nst; ++i) issue_next();

  WarpAcc<HEAD_DIM, NT> acc;
  acc.reset();
  const float sl2 = p.scale_log2;

  int consumed = 0;
  bool timed_out = false;
#pragma unroll 1
  for (; consumed < nst; ++consumed) {
    const int it = consumed;
    const int slot = it % STAGES;
    const bool ok = mbar_wait_bounded(&wbar[slot], (it / STAGES) & 1, WAIT_LIMIT_NS);
    if (!__all_sync(FULL_MASK, ok)) {  // a warp-uniform decision
      timed_out = true;
      break;
    }
    const int k0 = it * CPS;
    const int ch = first + k0 * WARPS;
    const int valid = min(CHUNK, ctx - ch * CHUNK);
    const uint32_t stage = smem_addr(wring + slot * Cfg::STAGE_BYTES);
    if constexpr (APPEND) {
      // the stage holding the new token's chunk (the warp's last)
      if (app_k >= 0 && it == app_k / CPS && app_phys >= 0) {
        const int pos = ctx - 1;
        const int64_t prow = static_cast<int64_t>(app_phys) * p.block_size + (pos & (p.block_size - 1));
        append_chunk_row<KV, HEAD_DIM, Cfg::ROW_BYTES, Cfg::BOX_B, Cfg::HALF_BYTES>(
            p, s, kvh, prow, stage + (app_k % CPS) * Cfg::CHUNK_BYTES, static_cast<uint32_t>(pos & (CHUNK - 1)),
            lane);
        __syncwarp();  // the new row is in shared memory before any lane reads the chunk
      }
    }
    if constexpr (FP8) {
      if (CPS == 2 && k0 + 1 < nk) {  // two chunks: the first is full (the second lies further in)
        const int valid2 = min(CHUNK, ctx - (ch + WARPS) * CHUNK);
        attend_pair_e4m3<HEAD_DIM, NT, Cfg::ROW_BYTES>(acc, qf, stage, Cfg::CHUNK_BYTES, Cfg::HALF_BYTES, valid2,
                                                       sl2, lane);
      } else {
        attend_chunk_e4m3<HEAD_DIM, NT, Cfg::ROW_BYTES>(acc, qf, stage, Cfg::HALF_BYTES, valid, sl2, lane);
      }
    } else {
      attend_chunk<T, HEAD_DIM, NT>(acc, qf, stage, Cfg::HALF_BYTES, valid, sl2, lane);
    }

    fence_proxy_async_smem();  // this lane's reads of the slot precede the refill's writes
    __syncwarp();
    if (issued < nst) issue_next();
  }

  if (timed_out) {
    bad = true;
    // let the copies still in flight land before the shared memory is reused
    for (int k = consumed; k < issued; ++k)
      (void)mbar_wait_bounded(&wbar[k % STAGES], (k / STAGES) & 1, WAIT_LIMIT_NS);
  }

  reduce_warp_sums<HEAD_DIM, NT>(acc);

  __syncthreads();  // every warp is done with its ring: reuse it for the merge
  float* mo = reinterpret_cast<float*>(ring);
  float* mm = mo + WARPS * GMAX * Cfg::MO_PITCH;
  float* ml = mm + WARPS * GMAX;
  int* mbad = reinterpret_cast<int*>(ml + WARPS * GMAX);
  store_warp_state<HEAD_DIM, NT, FP8>(acc, mo + warp * GMAX * Cfg::MO_PITCH, mm + warp * GMAX, ml + warp * GMAX,
                                      Cfg::MO_PITCH, lane);
  if (lane == 0) mbad[warp] = bad ? 1 : 0;
  __syncthreads();

  bool any_bad = false;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) any_bad |= mbad[w] != 0;

  for (int idx = threadIdx.x; idx < nq * HEAD_DIM; idx += WARPS * 32) {
    const int head = idx / HEAD_DIM;  // the CTA's query
    const int d = idx - head * HEAD_DIM;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, mm[w * GMAX + head]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {  // only a cluster CTA can have no chunk at all
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float f = ex2(mm[w * GMAX + head] - M);  // warps without chunks: 2^-inf = 0
        L += ml[w * GMAX + head] * f;
        O += mo[(w * GMAX + head) * Cfg::MO_PITCH + d] * f;
      }
    }
    float r = any_bad ? NAN : (L > 0.f ? O / L : 0.f);
    if constexpr (FP8) r *= p.out_scale;  // V codes times v_scale
    const size_t qrow = query_row(s0, head, H, kvh, G);
    if constexpr (SHARED) {
      const int m = s0 + head / G;  // the member sequence
      const int ctx_m = __ldg(p.context_lens + m);
      if (shared_len(lp, ctx_m, ctx_lead, cap, partition_tokens) == 0) continue;  // decoded on its own
      const bool nan = any_bad || ((*mismatch >> (head / G)) & 1);
      if (ctx_m <= partition_tokens) {  // one partition in all: this is the result
        static_cast<T*>(p.out)[qrow * HEAD_DIM + d] = to_elem<T>(nan ? NAN : r);
      } else {
        const size_t row = qrow * p.max_num_partitions + part;
        p.ws_o[row * HEAD_DIM + d] = nan ? NAN : r;
        if (d == 0) {
          p.ws_m[row] = nan ? 0.f : M;
          p.ws_l[row] = nan ? 1.f : L;
        }
      }
    } else if (CLUSTER) {
      // an empty CTA publishes m = -inf, l = 0: weight 0 in the cluster merge
      float* cta = reinterpret_cast<float*>(ring + Cfg::CTA_OFFSET);
      cta[head * HEAD_DIM + d] = r;
      if (d == 0) {
        cta[GMAX * HEAD_DIM + head] = any_bad ? 0.f : M;
        cta[GMAX * HEAD_DIM + GMAX + head] = any_bad ? 1.f : L;
      }
    } else if (single) {
      static_cast<T*>(p.out)[qrow * HEAD_DIM + d] = to_elem<T>(r);
    } else {
      const size_t row = qrow * p.max_num_partitions + part;
      p.ws_o[row * HEAD_DIM + d] = r;
      if (d == 0) {
        p.ws_m[row] = any_bad ? 0.f : M;
        p.ws_l[row] = any_bad ? 1.f : L;
      }
    }
  }

  if constexpr (CLUSTER) {
    // Merge the cluster's CTA results (o_r, m_r, l_r) read from each CTA's
    // shared memory: M = max m_r, w_r = l_r 2^(m_r - M), out = sum w_r o_r / sum w_r.
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every CTA's result is in its shared memory
    float* cta = reinterpret_cast<float*>(ring + Cfg::CTA_OFFSET);
    const int rank = static_cast<int>(cluster.block_rank());
    for (int idx = rank * (WARPS * 32) + threadIdx.x; idx < G * HEAD_DIM; idx += nclu * WARPS * 32) {
      const int head = idx / HEAD_DIM;
      const int d = idx - head * HEAD_DIM;
      float M = -INFINITY;
      for (int r = 0; r < nclu; ++r) {
        const float* peer = cluster.map_shared_rank(cta, r);
        M = fmaxf(M, peer[GMAX * HEAD_DIM + head]);
      }
      float L = 0.f, O = 0.f;
      for (int r = 0; r < nclu; ++r) {
        const float* peer = cluster.map_shared_rank(cta, r);
        const float w = peer[GMAX * HEAD_DIM + GMAX + head] * ex2(peer[GMAX * HEAD_DIM + head] - M);
        L += w;
        O += w * peer[head * HEAD_DIM + d];
      }
      static_cast<T*>(p.out)[(static_cast<size_t>(s) * H + kvh * G + head) * HEAD_DIM + d] = to_elem<T>(O / L);
    }
    cluster.sync();  // no CTA leaves while the others still read its shared memory
  }
  allow_dependent_launch();
}

template <typename T, typename KV, int HEAD_DIM, int NT, int WARPS, int STAGES, int MODE>
__global__ void __launch_bounds__(WARPS * 32) paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  decode_cta<T, KV, HEAD_DIM, NT, WARPS, STAGES, MODE, false>(p);
}

// Resident CTAs per SM that an append kernel is compiled to keep: the count
// its plain twin reaches (set by the twin's registers, or by shared memory
// where that binds first), so that the fused write costs no occupancy.
// Unbounded, the append path would raise the register count past it.
constexpr int append_min_ctas(int elem, int head_dim, int nt, int warps, int stages) {
  if (elem == 1) {  // E4M3: 4 warps x 2 stages of 8 KB (4 KB at d = 64)
    if (head_dim == 64) return nt == 1 ? 6 : 4;
    return 3;
  }
  if (head_dim == 64) return nt == 1 ? 6 : 4;
  if (head_dim == 128) return (nt == 1 && warps == 4 && stages == 1) ? 5 : 3;
  return 6;  // d = 256: 2 warps x 1 stage of 16 KB
}

// The decode with the new tokens' cache write fused in (APPEND above).
template <typename T, typename KV, int HEAD_DIM, int NT, int WARPS, int STAGES, int MODE>
__global__ void __launch_bounds__(WARPS * 32, append_min_ctas(kElemBytes<KV>, HEAD_DIM, NT, WARPS, STAGES))
    paged_append_decode_kernel(const __grid_constant__ DecodeParams p) {
  decode_cta<T, KV, HEAD_DIM, NT, WARPS, STAGES, MODE, true>(p);
}

// ================================================================ reduce
template <int VEC>
struct FVec {
  float v[VEC];
};

// VEC consecutive floats (VEC * 4 bytes aligned) through the read-only path.
template <int VEC>
__device__ __forceinline__ FVec<VEC> ldg_vec(const float* ptr) {
  FVec<VEC> r;
  if constexpr (VEC % 4 == 0) {
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(ptr) + i);
      r.v[4 * i] = t.x;
      r.v[4 * i + 1] = t.y;
      r.v[4 * i + 2] = t.z;
      r.v[4 * i + 3] = t.w;
    }
  } else {
    const float2 t = __ldg(reinterpret_cast<const float2*>(ptr));
    r.v[0] = t.x;
    r.v[1] = t.y;
  }
  return r;
}

// acc[0..VEC) * scale rounded to T and stored with one vector store.
template <typename T, int VEC>
__device__ __forceinline__ void store_vec(T* dst, const float (&acc)[VEC], float scale) {
  uint32_t w[VEC / 2];
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) w[i] = pack2<T>(acc[2 * i] * scale, acc[2 * i + 1] * scale);
  if constexpr (VEC == 8) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (VEC == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = w[0];
  }
}

struct ReduceParams {
  void* out;  // [S][H][d] of T
  const float* ws_o;
  const float* ws_m;
  const float* ws_l;
  const int32_t* context_lens;
  int cap;  // max_blocks_per_seq * block_size
  int num_heads;
  int partition_size;
  int max_num_partitions;
};

// At most PMAX partitions: one warp per (sequence, head), 8 per CTA.  Every
// load is issued at once -- the context length, lane q's (m_q, l_q) and each
// lane's HEAD_DIM / 32 dims of all PMAX partition outputs -- so the kernel
// waits for memory once.  Rows past the sequence's partitions hold stale data
// and are dropped by select, never multiplied by a zero weight.
template <typename T, int HEAD_DIM, int PMAX>
__global__ void __launch_bounds__(256) splitk_reduce_small_kernel(const __grid_constant__ ReduceParams p) {
  constexpr int VEC = HEAD_DIM / 32;
  using VecT = FVec<VEC>;
  grid_dependency_wait();  // the partitions come from the decode kernel just before
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * 8 + warp;
  const int s = blockIdx.y;
  if (h >= p.num_heads) return;
  const size_t row0 = (static_cast<size_t>(s) * p.num_heads + h) * p.max_num_partitions;
  const int ctx = __ldg(p.context_lens + s);
  VecT o[PMAX];
#pragma unroll
  for (int q = 0; q < PMAX; ++q)
    o[q] = q < p.max_num_partitions ? ldg_vec<VEC>(p.ws_o + (row0 + q) * HEAD_DIM + lane * VEC) : VecT{};
  const bool mine = lane < p.max_num_partitions;
  const float m = mine ? __ldg(p.ws_m + row0 + lane) : -INFINITY;
  const float l = mine ? __ldg(p.ws_l + row0 + lane) : 0.f;
  const int nparts = (ctx <= 0 || ctx > p.cap) ? 0 : (ctx + p.partition_size - 1) / p.partition_size;
  if (nparts <= 1) return;  // finished by the decode kernel
  const float mv = lane < nparts ? m : -INFINITY;
  float M = mv;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w = lane < nparts ? l * ex2(m - M) : 0.f;
  float L = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  float acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
#pragma unroll
  for (int q = 0; q < PMAX; ++q) {
    const float wq = __shfl_sync(0xffffffffu, w, q);
    if (q < nparts) {
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += wq * o[q].v[v];
    }
  }
    store_vec<T, VEC>(static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.num_heads + h) * HEAD_DIM + lane * VEC,
                    acc, 1.f / L);
}

// Warps per (sequence, head): WPH warps split the partitions (q = sub, sub +
// WPH, ...); each lane owns HEAD_DIM / 32 consecutive output dims and reads
// them as one vector per partition.  A CTA has 8 warps = 8 / WPH heads, or
// 16 warps for one head when WPH = 16.
template <int WPH>
constexpr int reduce_warps() { return WPH > 8 ? WPH : 8; }

template <typename T, int HEAD_DIM, int WPH>
__global__ void __launch_bounds__(reduce_warps<WPH>() * 32) splitk_reduce_kernel(const __grid_constant__ ReduceParams p) {
  constexpr int VEC = HEAD_DIM / 32;
  constexpr int NW = reduce_warps<WPH>();
  constexpr int HPC = NW / WPH;
  using VecT = FVec<VEC>;
  __shared__ float sm_m[NW], sm_l[NW];
  __shared__ VecT sm_o[NW][32];
  grid_dependency_wait();  // the partitions come from the decode kernel just before
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * HPC + warp / WPH;
  const int sub = warp % WPH;
  const int s = blockIdx.y;
  const int ctx = __ldg(p.context_lens + s);
  const int nparts = (ctx <= 0 || ctx > p.cap) ? 0 : (ctx + p.partition_size - 1) / p.partition_size;
  const bool active = h < p.num_heads && nparts > 1;  // one partition: finished by the decode kernel
  const size_t row0 = (static_cast<size_t>(s) * p.num_heads + (active ? h : 0)) * p.max_num_partitions;
  const int cnt = active ? (nparts - sub + WPH - 1) / WPH : 0;  // this warp's partitions

  // maximum over this warp's partitions
  float Mw = -INFINITY;
  for (int i = lane; i < cnt; i += 32) Mw = fmaxf(Mw, __ldg(p.ws_m + row0 + sub + i * WPH));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, off));

  // weights w_q = l_q 2^(m_q - Mw), broadcast 32 at a time; weighted sum of o_q
  float Lw = 0.f;
  float acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
  for (int base = 0; base < cnt; base += 32) {
    const int i = base + lane;
    float w = 0.f;
    if (i < cnt) {
      const size_t r = row0 + sub + static_cast<size_t>(i) * WPH;
      w = __ldg(p.ws_l + r) * ex2(__ldg(p.ws_m + r) - Mw);
    }
    Lw += w;
    const int n = min(32, cnt - base);
#pragma unroll 8
    for (int j = 0; j < n; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const size_t r = row0 + sub + static_cast<size_t>(base + j) * WPH;
      const VecT o = ldg_vec<VEC>(p.ws_o + r * HEAD_DIM + lane * VEC);
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += wj * o.v[v];
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Lw += __shfl_xor_sync(0xffffffffu, Lw, off);

  if constexpr (WPH > 1) {
    // combine the WPH warps of each head
    if (lane == 0) {
      sm_m[warp] = Mw;
      sm_l[warp] = Lw;
    }
    VecT o;
#pragma unroll
    for (int v = 0; v < VEC; ++v) o.v[v] = acc[v];
    sm_o[warp][lane] = o;
    __syncthreads();
    if (sub != 0 || !active) return;
    const int w0 = warp;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < WPH; ++k) M = fmaxf(M, sm_m[w0 + k]);
    float L = 0.f;
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
#pragma unroll
    for (int k = 0; k < WPH; ++k) {
      const float f = ex2(sm_m[w0 + k] - M);  // a warp without partitions: 2^-inf = 0
      L += sm_l[w0 + k] * f;
      const VecT ok = sm_o[w0 + k][lane];
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += f * ok.v[v];
    }
    Lw = L;
  } else {
    if (!active) return;
  }
  store_vec<T, VEC>(static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.num_heads + h) * HEAD_DIM + lane * VEC,
                    acc, 1.f / Lw);
}

// ================================================================ launchers
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, resolved through the runtime once (the library does
// not link the driver library directly).
inline cudaError_t encode_fn(EncodeTiledFn* out) {
  static std::atomic<EncodeTiledFn> cached{nullptr};
  EncodeTiledFn f = cached.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || ptr == nullptr) return cudaErrorNotSupported;
    f = reinterpret_cast<EncodeTiledFn>(ptr);
    cached.store(f, std::memory_order_release);
  }
  *out = f;
  return cudaSuccess;
}

template <typename KV>
constexpr CUtensorMapDataType tma_dtype() {
  return kIsFp8<KV> ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                    : (std::is_same<KV, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// A KV pool [N][B][Hk][d] of KV elements seen as rows x heads x dims, boxes
// of 16 rows x 1 head x one box row (128 bytes; 64 for 64 one-byte dims),
// swizzled over the box row's width.
template <typename KV, int HEAD_DIM>
cudaError_t encode_pool_map(CUtensorMap* map, const void* pool, int num_kv_heads, int64_t rows) {
  using Cfg = DecodeCfg<HEAD_DIM, 1, 1, 1, kElemBytes<KV>>;
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encode_fn(&enc);
  if (e != cudaSuccess) return e;
  constexpr int ELEM = kElemBytes<KV>;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HEAD_DIM), static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(HEAD_DIM) * ELEM,
                                 static_cast<cuuint64_t>(num_kv_heads) * HEAD_DIM * ELEM};
  const cuuint32_t box[3] = {Cfg::BOX_ELEMS, 1, CHUNK};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = Cfg::ROW_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = enc(map, tma_dtype<KV>(), 3, const_cast<void*>(pool), dims, strides, box, estride,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// encode_pool_map through a per-thread cache of recent encodings.  A map is a
// pure function of (pool address, heads, rows) for a given element type and
// head size (each instantiation has its own cache), so a hit is always the
// map that encoding would produce, even for a pool freed and reallocated at
// the same address.  Decode loops that rotate a few pools skip the encode.
template <typename KV, int HEAD_DIM>
cudaError_t make_pool_map(CUtensorMap* map, const void* pool, int num_kv_heads, int64_t rows) {
  constexpr int kEntries = 16;
  struct Entry {
    CUtensorMap map;
    const void* pool;
    int64_t rows;
    int heads;
  };
  thread_local Entry cache[kEntries];  // zero-initialised: pool == nullptr marks an empty entry
  thread_local int next = 0;
  if (pool != nullptr) {
    for (int i = 0; i < kEntries; ++i) {
      const Entry& e = cache[i];
      if (e.pool == pool && e.rows == rows && e.heads == num_kv_heads) {
        *map = e.map;
        return cudaSuccess;
      }
    }
  }
  const cudaError_t err = encode_pool_map<KV, HEAD_DIM>(map, pool, num_kv_heads, rows);
  if (err == cudaSuccess && pool != nullptr) {
    Entry& e = cache[next];
    e.map = *map;
    e.pool = pool;
    e.rows = rows;
    e.heads = num_kv_heads;
    next = (next + 1) % kEntries;
  }
  return err;
}

template <typename Kernel>
cudaError_t ensure_smem(Kernel k, int bytes, std::atomic<uint64_t>& done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done_mask.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 2
#endif

#ifndef PA_DECODE_FP8_WARPS
#define PA_DECODE_FP8_WARPS 4
#endif
#ifndef PA_DECODE_FP8_STAGES
#define PA_DECODE_FP8_STAGES 2
#endif
// the per-sequence (suffix) pass of the shared-prefix decode, up to d = 128
#ifndef PA_SUFFIX_WARPS
#define PA_SUFFIX_WARPS 2
#endif
#ifndef PA_SUFFIX_STAGES
#define PA_SUFFIX_STAGES 2
#endif

// Launch kinds, each with its CTA shape: the single launch, the split-K
// launch, and the two passes of the shared-prefix decode (the per-sequence
// suffixes, the shared prefix).
enum LaunchKind { KIND_SINGLE = 0, KIND_SPLITK = 1, KIND_SUFFIX = 2, KIND_SHARED = 3 };

// CTA shape per head size: 4 warps x 2 stages (8 KB stages up to d = 128,
// three CTAs per SM).  d = 256 has 16 KB stages and uses 2 warps x 1 stage,
// six CTAs per SM: more CTAs in flight beat deeper per-warp pipelining there
// (59.9 -> 55.0 us on the head-dim-256 workload; 2x2, 3x2, 4x2, 2x3, 4x1,
// 8x1 and 1-warp shapes were slower).  E4M3 stages are 8 KB for every head
// size (two chunks up to d = 128), so E4M3 keeps 4 warps x 2 stages
// throughout; sweeps over 2-8 warps and 1-4 stages found nothing faster.
// KIND_SPLITK: the split-K launch.  Its CTAs each cover one partition (at
// most partition_size tokens), and at d = 128 one stage per warp (six CTAs
// per SM) is faster there: llama3-8b 53.2 -> 52.6 us, long-context 227.0 ->
// 217.9 us, 70B unchanged.  The single launch keeps two stages (with one it
// lost 10-30%).  KIND_SUFFIX: the per-sequence pass of the shared-prefix
// decode, whose CTAs cover suffixes of a partition or less: 2 warps x 2
// stages (six CTAs per SM) for both element types (shared-prefix batch:
// E4M3 144.0 -> 124.6 us, fp16 179.7 -> 178.5 us; 2x1, 2x3, 3x2, 1x4 and
// the split-K shapes were slower).  KIND_SHARED, the shared pass, keeps the
// single launch's shape (4x1, 2x2 and 8x1 were slower).
template <int HEAD_DIM, int ELEM = 2, int KIND = KIND_SINGLE>
struct DecodeShape {
  static constexpr bool FP8 = ELEM == 1;
  static constexpr bool PARTS = KIND == KIND_SPLITK || KIND == KIND_SUFFIX;
  static constexpr bool SUFFIX = KIND == KIND_SUFFIX && HEAD_DIM <= 128;
  static constexpr int WARPS = SUFFIX ? PA_SUFFIX_WARPS
                               : FP8  ? PA_DECODE_FP8_WARPS
                                      : (HEAD_DIM > 128 ? 2 : PA_DECODE_WARPS);
  static constexpr int STAGES = SUFFIX ? PA_SUFFIX_STAGES
                                : FP8  ? (HEAD_DIM > 128 ? 2 : PA_DECODE_FP8_STAGES)
                                       : (HEAD_DIM > 128 || (PARTS && HEAD_DIM == 128) ? 1 : PA_DECODE_STAGES);
};

template <typename T, typename KV, int HEAD_DIM>
cudaError_t fill_decode_params(const DecodeArgs& a, DecodeParams* pp) {
  DecodeParams& p = *pp;
  const int64_t pool_rows = static_cast<int64_t>(a.num_blocks) * a.block_size;
  cudaError_t e = make_pool_map<KV, HEAD_DIM>(&p.tmap_k, a.k_cache, a.num_kv_heads, pool_rows);
  if (e != cudaSuccess) return e;
  e = make_pool_map<KV, HEAD_DIM>(&p.tmap_v, a.v_cache, a.num_kv_heads, pool_rows);
  if (e != cudaSuccess) return e;
  p.out = a.out;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  const size_t rows = ws_rows(a.num_seqs, a.num_heads, a.max_num_partitions);
  p.ws_o = a.ws;
  p.ws_m = a.ws ? a.ws + rows * HEAD_DIM : nullptr;
  p.ws_l = a.ws ? a.ws + rows * HEAD_DIM + rows : nullptr;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.chunks_per_block_log2 = __builtin_ctz(static_cast<unsigned>(a.block_size / CHUNK));
  p.num_blocks = a.num_blocks;
  p.partition_chunks = a.partition_size / CHUNK;
  p.max_num_partitions = a.max_num_partitions;
  const bool fp8 = kIsFp8<KV>;
  p.scale_log2 = a.scale * (fp8 ? a.k_scale : 1.f) * 1.4426950408889634f;
  p.out_scale = fp8 ? a.v_scale : 1.f;
  p.prefix_lens = a.prefix_lens;
  p.seqs_per_group = a.seqs_per_group > 0 ? a.seqs_per_group : 1;
  p.members_per_cta = 1;
  p.subgroups = 1;
  p.num_seqs = a.num_seqs;
  p.new_k = a.new_key;
  p.new_v = a.new_value;
  p.k_pool = const_cast<void*>(a.k_cache);  // written only by the append path
  p.v_pool = const_cast<void*>(a.v_cache);
  p.k_scale = fp8 ? a.k_scale : 1.f;
  p.v_scale = fp8 ? a.v_scale : 1.f;
  return cudaSuccess;
}

// Members of a group whose queries one shared-pass CTA holds: as many whole
// query groups as fit in 8 * NT query rows, at most the group size.
template <int NT>
int members_per_cta(const DecodeArgs& a) {
  const int G = a.num_heads / a.num_kv_heads;
  return std::max(1, std::min(a.seqs_per_group, 8 * NT / G));
}

template <typename T, typename KV, int HEAD_DIM, int NT, int MODE, int KIND = KIND_SINGLE, bool APPEND = false>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  constexpr bool CLUSTER = MODE == MODE_CLUSTER;
  constexpr int ELEM = kElemBytes<KV>;
  constexpr int WARPS = DecodeShape<HEAD_DIM, ELEM, KIND>::WARPS;
  constexpr int STAGES = DecodeShape<HEAD_DIM, ELEM, KIND>::STAGES;
  using Cfg = DecodeCfg<HEAD_DIM, NT, WARPS, STAGES, ELEM>;
  auto kern = [] {
    if constexpr (APPEND) {
      return paged_append_decode_kernel<T, KV, HEAD_DIM, NT, WARPS, STAGES, MODE>;
    } else {
      return paged_decode_kernel<T, KV, HEAD_DIM, NT, WARPS, STAGES, MODE>;
    }
  }();
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_smem(kern, Cfg::SMEM_BYTES, smem_set);
  if (e != cudaSuccess) return e;
  DecodeParams p;
  e = fill_decode_params<T, KV, HEAD_DIM>(a, &p);
  if (e != cudaSuccess) return e;
  unsigned gz = static_cast<unsigned>(a.num_seqs);
  if constexpr (MODE == MODE_SHARED) {
    const int groups = (a.num_seqs + p.seqs_per_group - 1) / p.seqs_per_group;
    p.members_per_cta = members_per_cta<NT>(a);
    p.subgroups = (std::min(a.seqs_per_group, a.num_seqs) + p.members_per_cta - 1) / p.members_per_cta;
    gz = static_cast<unsigned>(groups) * static_cast<unsigned>(p.subgroups);
  }
  dim3 grid(a.num_kv_heads, CLUSTER ? a.cluster_size : a.max_num_partitions, gz);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (CLUSTER) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = a.cluster_size;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Resident decode CTAs the device holds at once (SMs x CTAs per SM), cached
// per device.
template <typename T, typename KV, int HEAD_DIM, int NT>
cudaError_t decode_slots(int* slots) {
  constexpr int ELEM = kElemBytes<KV>;
  constexpr int WARPS = DecodeShape<HEAD_DIM, ELEM>::WARPS;
  constexpr int STAGES = DecodeShape<HEAD_DIM, ELEM>::STAGES;
  using Cfg = DecodeCfg<HEAD_DIM, NT, WARPS, STAGES, ELEM>;
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_acquire);
    if (c > 0) {
      *slots = c;
      return cudaSuccess;
    }
  }
  auto kern = paged_decode_kernel<T, KV, HEAD_DIM, NT, WARPS, STAGES, MODE_GRID>;
  static std::atomic<uint64_t> smem_set{0};
  e = ensure_smem(kern, Cfg::SMEM_BYTES, smem_set);
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, WARPS * 32, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int v = sms * (per_sm > 0 ? per_sm : 1);
  if (dev < 64) cache[dev].store(v, std::memory_order_release);
  *slots = v;
  return cudaSuccess;
}

// Single-launch decode: one CTA per (sequence, KV head) when those fill the
// resident slots; otherwise a cluster of up to 8 CTAs per pair, each with at
// least 512 tokens of capacity.  Split-K (a workspace given): the plain grid.
template <typename T, typename KV, int HEAD_DIM, int NT, bool APPEND = false>
cudaError_t launch_decode_auto(const DecodeArgs& a, cudaStream_t stream) {
  if (a.cluster_size >= 0) {
    if (a.cluster_size > 0) return launch_decode_t<T, KV, HEAD_DIM, NT, MODE_CLUSTER, KIND_SINGLE, APPEND>(a, stream);
    return a.ws != nullptr ? launch_decode_t<T, KV, HEAD_DIM, NT, MODE_GRID, KIND_SPLITK, APPEND>(a, stream)
                           : launch_decode_t<T, KV, HEAD_DIM, NT, MODE_GRID, KIND_SINGLE, APPEND>(a, stream);
  }
  int slots = 0;
  cudaError_t e = decode_slots<T, KV, HEAD_DIM, NT>(&slots);
  if (e != cudaSuccess) return e;
  const int64_t pairs = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  int64_t k = pairs > 0 ? slots / pairs : 1;
  const int64_t cap = static_cast<int64_t>(a.max_blocks_per_seq) * a.block_size;
  k = std::min<int64_t>(k, (cap + 511) / 512);
  DecodeArgs b = a;
  b.cluster_size = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(8, k)));
  if (b.cluster_size == 1) {
    b.cluster_size = 0;
    // A second wave of CTAs, but at most one: the longest sequences go in the
    // first.  Over more waves the block scheduler balances by itself, and the
    // ranking would scatter sequences that sit side by side in the batch and
    // share blocks (samples of one prompt), whose reads L2 serves when their
    // CTAs run together.
    if (pairs > slots && pairs <= 2 * static_cast<int64_t>(slots) && a.num_seqs <= kLongestFirstMax &&
        a.prefix_lens == nullptr)
      return launch_decode_t<T, KV, HEAD_DIM, NT, MODE_LONGEST_FIRST, KIND_SINGLE, APPEND>(b, stream);
    return launch_decode_t<T, KV, HEAD_DIM, NT, MODE_GRID, KIND_SINGLE, APPEND>(b, stream);
  }
  return launch_decode_t<T, KV, HEAD_DIM, NT, MODE_CLUSTER, KIND_SINGLE, APPEND>(b, stream);
}

template <typename T, int HEAD_DIM>
cudaError_t launch_reduce_t(const ReduceArgs& a, cudaStream_t stream) {
  ReduceParams p;
  const size_t rows = ws_rows(a.num_seqs, a.num_heads, a.max_num_partitions);
  p.out = a.out;
  p.ws_o = a.ws;
  p.ws_m = a.ws + rows * HEAD_DIM;
  p.ws_l = a.ws + rows * HEAD_DIM + rows;
  p.context_lens = a.context_lens;
  p.cap = a.max_blocks_per_seq * a.block_size;
  p.num_heads = a.num_heads;
  p.partition_size = a.partition_size;
  p.max_num_partitions = a.max_num_partitions;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.max_num_partitions <= 8) {  // one warp per (sequence, head), one memory round trip
    cfg.gridDim = dim3((a.num_heads + 7) / 8, a.num_seqs);
    e = cudaLaunchKernelEx(&cfg, splitk_reduce_small_kernel<T, HEAD_DIM, 8>, p);
  } else if (a.max_num_partitions <= 32) {  // one warp per (sequence, head)
    cfg.gridDim = dim3((a.num_heads + 7) / 8, a.num_seqs);
    e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<T, HEAD_DIM, 1>, p);
  } else if (a.max_num_partitions <= 64) {  // four warps per (sequence, head)
    cfg.gridDim = dim3((a.num_heads + 1) / 2, a.num_seqs);
    e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<T, HEAD_DIM, 4>, p);
  } else if (a.max_num_partitions <= 128) {  // eight warps per (sequence, head): fewer serial
                                             // round trips per warp
    cfg.gridDim = dim3(a.num_heads, a.num_seqs);
    e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<T, HEAD_DIM, 8>, p);
  } else {  // sixteen warps per (sequence, head), one head per CTA (long context, 256
            // partitions: step 216.5 us with four warps, 209.5 with eight, 207.5 with sixteen)
    cfg.gridDim = dim3(a.num_heads, a.num_seqs);
    cfg.blockDim = dim3(16 * 32);
    e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<T, HEAD_DIM, 16>, p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Entry points used by the per-dtype translation units (KV = T for 16-bit
// caches, E4M3 for one-byte caches).
template <typename T, typename KV, bool APPEND>
cudaError_t launch_decode_typed_as(const DecodeArgs& a, cudaStream_t stream) {
  const bool two = a.num_heads / a.num_kv_heads > 8;
  switch (a.head_dim) {
    case 64:
      return two ? launch_decode_auto<T, KV, 64, 2, APPEND>(a, stream)
                 : launch_decode_auto<T, KV, 64, 1, APPEND>(a, stream);
    case 128:
      return two ? launch_decode_auto<T, KV, 128, 2, APPEND>(a, stream)
                 : launch_decode_auto<T, KV, 128, 1, APPEND>(a, stream);
    case 256: return two ? cudaErrorInvalidValue : launch_decode_auto<T, KV, 256, 1, APPEND>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The append variant (the new tokens' cache write fused in) when the
// arguments carry new K/V rows.
template <typename T, typename KV = T>
cudaError_t launch_decode_typed(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  return a.new_key != nullptr ? launch_decode_typed_as<T, KV, true>(a, stream)
                              : launch_decode_typed_as<T, KV, false>(a, stream);
}

// Shared-prefix split-K: the shared pass (query tiles of NTS x 8 rows: the
// members of a group times G), then the per-sequence pass, which skips the
// partitions the shared pass wrote.  That pass is the split-K kernel and takes
// its CTA shape (at d = 128, one stage per warp and five CTAs per SM): its
// CTAs cover a sequence's private suffix, often a partition or less, and more
// of them in flight overlap more of their prologues (shared-prefix fp16:
// 187.8 -> 179.7 us per step).
template <typename T, typename KV, int HEAD_DIM, int NTS, int NT>
cudaError_t launch_prefix_t(const DecodeArgs& a, cudaStream_t stream) {
  cudaError_t e = launch_decode_t<T, KV, HEAD_DIM, NTS, MODE_SHARED, KIND_SHARED>(a, stream);
  if (e != cudaSuccess) return e;
  return launch_decode_t<T, KV, HEAD_DIM, NT, MODE_GRID, KIND_SUFFIX>(a, stream);
}

template <typename T, typename KV = T>
cudaError_t launch_decode_prefix_typed(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int G = a.num_heads / a.num_kv_heads;
  const bool two = G > 8;
  // one query tile when a whole group's queries fit in 8 rows, else two
  const bool two_s = std::min(a.seqs_per_group, 16 / G) * G > 8;
  switch (a.head_dim) {
    case 64:
      if (two) return launch_prefix_t<T, KV, 64, 2, 2>(a, stream);
      return two_s ? launch_prefix_t<T, KV, 64, 2, 1>(a, stream) : launch_prefix_t<T, KV, 64, 1, 1>(a, stream);
    case 128:
      if (two) return launch_prefix_t<T, KV, 128, 2, 2>(a, stream);
      return two_s ? launch_prefix_t<T, KV, 128, 2, 1>(a, stream) : launch_prefix_t<T, KV, 128, 1, 1>(a, stream);
    case 256: return two ? cudaErrorInvalidValue : launch_prefix_t<T, KV, 256, 1, 1>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_splitk_reduce_typed(const ReduceArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  switch (a.head_dim) {
    case 64: return launch_reduce_t<T, 64>(a, stream);
    case 128: return launch_reduce_t<T, 128>(a, stream);
    case 256: return launch_reduce_t<T, 256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

}  // namespace pa
