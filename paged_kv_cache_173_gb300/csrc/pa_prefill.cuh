// pa_prefill.cuh -- paged prefill attention (whole prompts and chunks of
// them) over the K/V pools, templated on the element type T (__half or
// __nv_bfloat16) and the head size.
//
//  paged_prefill_kernel   one CTA per (query tile, KV head, sequence).  A tile
//                         is 64 query rows: 64 / G consecutive new tokens of
//                         the sequence times the G query heads of the KV
//                         head, so that every K/V byte a CTA loads serves G
//                         heads.  Four warps own 16 rows each.  The CTA walks
//                         the keys from position 0 up to its last row's
//                         position in stages of 64 keys, loaded by TMA through
//                         the block table (one lookup per 16 tokens); S = Q K^T
//                         and O += P V run on m16n8k16 MMAs, with the online
//                         softmax in float32 between them.
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

constexpr int PF_ROWS = 64;   // query rows per CTA
constexpr int PF_KEYS = 64;   // keys per stage
constexpr int PF_WARPS = 4;
constexpr int PF_STAGES = 2;

struct PrefillParams {
  CUtensorMap tmap_k;  // pools as [N*B rows][Hk][d], 16 x 1 x 64 boxes, 128-byte swizzle
  CUtensorMap tmap_v;
  void* out;       // [rows][H][d] of T
  const void* q;   // [rows][H][d] of T
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;  // [S + 1]
  int max_blocks_per_seq;
  int num_heads;
  int group;
  int block_size;
  int num_blocks;
  int tiles;        // query tiles per sequence (grid x)
  int tile_tokens;  // PF_ROWS / group
  float scale_log2;
};

template <int HEAD_DIM>
struct PrefillCfg {
  static constexpr int DBOX = HEAD_DIM / BOX_DIMS;   // 64-dim boxes per row
  static constexpr int SUB = PF_KEYS / CHUNK;        // 16-token boxes per stage
  static constexpr int HALF_BYTES = DBOX * SUB * BOX_BYTES;  // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * HALF_BYTES;
  static constexpr int SMEM_BYTES = 1024 + 1024 + PF_STAGES * STAGE_BYTES;
};

// Byte offset, within a K (or V) stage, of 16-byte unit u (dims 8u .. 8u+7)
// of key t: box (u / 8, t / 16), row t % 16, 128-byte swizzle.
template <int HEAD_DIM>
__device__ __forceinline__ uint32_t pf_offset(uint32_t t, uint32_t u) {
  using Cfg = PrefillCfg<HEAD_DIM>;
  const uint32_t row = t & 15u;
  return ((u >> 3) * Cfg::SUB + (t >> 4)) * BOX_BYTES + row * 128u + (((u & 7u) ^ (row & 7u)) << 4);
}

template <typename T, int HEAD_DIM>
__global__ void __launch_bounds__(PF_WARPS * 32)
paged_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using Cfg = PrefillCfg<HEAD_DIM>;
  constexpr int KSTEPS = HEAD_DIM / 16;  // k-steps of S = Q K^T
  constexpr int DT = HEAD_DIM / 8;       // n-tiles of O
  constexpr int NT = PF_KEYS / 8;        // n-tiles of S
  constexpr bool kBf16 = !std::is_same<T, __half>::value;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + 1024;

  const int tile = p.tiles - 1 - static_cast<int>(blockIdx.x);  // the longest tiles start first
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int c4 = lane & 3;
  const int G = p.group;
  const int H = p.num_heads;

  grid_dependency_wait();  // the cache write before this launch has finished

  const int q0 = __ldg(p.query_start_loc + s);
  const int qlen = __ldg(p.query_start_loc + s + 1) - q0;
  const int ctx = __ldg(p.context_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  const int t0 = tile * p.tile_tokens;  // first token of the tile
  if (t0 >= qlen) {
    allow_dependent_launch();
    return;
  }
  const int t1 = min(qlen, t0 + p.tile_tokens);
  const bool ctx_bad = ctx < qlen || ctx > cap;
  const int base = ctx - qlen;          // position of the sequence's first new token
  const int kend = ctx_bad ? 0 : base + t1;  // keys 0 .. kend - 1 are read
  const int nst = (kend + PF_KEYS - 1) / PF_KEYS;

  // This thread's rows: r = 16 * warp + g (+ 8); token t0 + r / G, head r % G.
  int pos[2];
  size_t qrow[2];
  bool rv[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = 16 * warp + g + 8 * i;
    const int t = t0 + r / G;
    rv[i] = t < t1;
    pos[i] = rv[i] ? base + t : -1;
    qrow[i] = static_cast<size_t>(q0 + (rv[i] ? t : t0)) * H + kvh * G + r % G;
  }

  // Q as the A operand: a0 (row g, dims 2c..), a1 (row g+8), a2/a3 the same at dims + 8.
  uint32_t qa[KSTEPS][4];
  {
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) + qrow[0] * HEAD_DIM);
    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) + qrow[1] * HEAD_DIM);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      qa[ks][0] = __ldg(r0 + ks * 8 + c4);
      qa[ks][1] = __ldg(r1 + ks * 8 + c4);
      qa[ks][2] = __ldg(r0 + ks * 8 + c4 + 4);
      qa[ks][3] = __ldg(r1 + ks * 8 + c4 + 4);
    }
  }

  const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
  if (threadIdx.x == 0) {
    for (int i = 0; i < PF_STAGES; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // One thread fills stage `st` with keys [st * 64, st * 64 + 64) below kend.
  bool bad = false;
  auto issue = [&](int st) {
    const int slot = st % PF_STAGES;
    uint8_t* kd = ring + slot * Cfg::STAGE_BYTES;
    const int nsub = min(Cfg::SUB, (kend - st * PF_KEYS + CHUNK - 1) / CHUNK);
    mbar_arrive_expect_tx(&bars[slot], nsub * 2 * Cfg::DBOX * BOX_BYTES);
    for (int j = 0; j < nsub; ++j) {
      const int key0 = st * PF_KEYS + j * CHUNK;
      int phys = __ldg(bt + key0 / p.block_size);
      if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
        bad = true;  // never read outside the pool; the tile's outputs become NaN
        phys = 0;
      }
      const int y = phys * p.block_size + key0 % p.block_size;
#pragma unroll
      for (int db = 0; db < Cfg::DBOX; ++db) {
        tma_load_3d(kd + (db * Cfg::SUB + j) * BOX_BYTES, &p.tmap_k, db * BOX_DIMS, kvh, y, &bars[slot]);
        tma_load_3d(kd + Cfg::HALF_BYTES + (db * Cfg::SUB + j) * BOX_BYTES, &p.tmap_v, db * BOX_DIMS, kvh, y,
                    &bars[slot]);
      }
    }
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < PF_STAGES && i < nst; ++i) issue(i);

  float o[DT][4];
#pragma unroll
  for (int n = 0; n < DT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
  float m[2] = {-INFINITY, -INFINITY};
  float l[2] = {0.f, 0.f};
  const float sl2 = p.scale_log2;

  // ldmatrix lane roles: matrix lane / 8 of the four; row (lane % 8)
  const uint32_t lrow = lane & 7;
  const uint32_t lmat = lane >> 3;
  bool timed_out = false;
  int consumed = 0;
#pragma unroll 1
  for (; consumed < nst; ++consumed) {
    const int st = consumed;
    const int slot = st % PF_STAGES;
    const bool ok = mbar_wait_bounded(&bars[slot], (st / PF_STAGES) & 1, WAIT_LIMIT_NS);
    if (!__syncthreads_and(ok)) {  // a CTA-uniform decision
      timed_out = true;
      break;
    }
    const uint32_t kb = smem_addr(ring + slot * Cfg::STAGE_BYTES);
    const uint32_t vb = kb + Cfg::HALF_BYTES;
    const int k0 = st * PF_KEYS;

    // S[16 rows][64 keys] = Q K^T.  ldmatrix.x4 of K: matrices (keys 16j+0-7, dims 16ks+0-7),
    // (keys 16j+0-7, dims +8), (keys 16j+8-15, dims +0), (keys 16j+8-15, dims +8) give the
    // B fragments of n-tiles 2j and 2j+1 at k-step ks.
    float sc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[n][i] = 0.f;
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      const uint32_t key = 16 * j + lrow + ((lmat >> 1) << 3);
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        uint32_t r[4];
        ldsm_x4(r, kb + pf_offset<HEAD_DIM>(key, 2 * ks + (lmat & 1)));
        mma_16816<T>(sc[2 * j], qa[ks], r[0], r[1]);
        mma_16816<T>(sc[2 * j + 1], qa[ks], r[2], r[3]);
      }
    }

    // online softmax per row (base 2): key k is visible to a row at position
    // pos iff k <= pos (pos < kend, so every visible key was loaded)
    const bool diag = k0 + PF_KEYS - 1 > base + t0;  // some key here lies past some row
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = k0 + 8 * n + 2 * c4 + (i & 1);
        const int ri = i >> 1;
        float x = sc[n][i] * sl2;
        if (diag && key > pos[ri]) x = -INFINITY;
        sc[n][i] = x;
        mx[ri] = fmaxf(mx[ri], x);
      }
    float cr[2], mb[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(FULL_MASK, mx[ri], 1));
      mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(FULL_MASK, mx[ri], 2));
      const float mn = fmaxf(m[ri], mx[ri]);
      mb[ri] = mn == -INFINITY ? 0.f : mn;  // a row that has seen no key yet
      cr[ri] = ex2(m[ri] - mb[ri]);
      m[ri] = mn;
    }
    // P as the A operand of P V: n-tiles 2j, 2j+1 of S are k-step j (keys 16j..16j+15).
    // fp16: the sums add the rounded weights that multiply V.  bf16 keeps 8
    // significant bits, so P also goes in as its rounded residual (pr) and
    // the sums add P itself.
    uint32_t pa[NT / 2][4];
    uint32_t pr[kBf16 ? NT / 2 : 1][4];
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float* c = sc[2 * j + h];
        const float p0 = ex2(c[0] - mb[0]), p1 = ex2(c[1] - mb[0]);  // row g
        const float p2 = ex2(c[2] - mb[1]), p3 = ex2(c[3] - mb[1]);  // row g + 8
        const uint32_t lo = pack2<T>(p0, p1);
        const uint32_t hi = pack2<T>(p2, p3);
        const float2 flo = unpack2<T>(lo);
        const float2 fhi = unpack2<T>(hi);
        if constexpr (kBf16) {
          pr[j][2 * h] = pack2<T>(p0 - flo.x, p1 - flo.y);
          pr[j][2 * h + 1] = pack2<T>(p2 - fhi.x, p3 - fhi.y);
          ps[0] += p0 + p1;
          ps[1] += p2 + p3;
        } else {
          ps[0] += flo.x + flo.y;
          ps[1] += fhi.x + fhi.y;
        }
        pa[j][2 * h] = lo;
        pa[j][2 * h + 1] = hi;
      }
    }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) l[ri] = l[ri] * cr[ri] + ps[ri];
#pragma unroll
    for (int n = 0; n < DT; ++n) {
      o[n][0] *= cr[0];
      o[n][1] *= cr[0];
      o[n][2] *= cr[1];
      o[n][3] *= cr[1];
    }

    // O += P V.  ldmatrix.x4.trans of V: matrices (keys 16j+0-7, dims 16d+0-7), (keys +8, dims
    // +0), (keys +0, dims +8), (keys +8, dims +8) give the B fragments of dim n-tiles 2d, 2d+1
    // at k-step j.  Keys at or past kend hold stale data: zeroed by select.
    const bool tail = k0 + PF_KEYS > kend;
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      const uint32_t key = 16 * j + lrow + ((lmat & 1) << 3);
      uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
      if (tail) {
        const int kk = k0 + 16 * j + 2 * c4;
        mlo = (kk < kend ? 0x0000ffffu : 0u) | (kk + 1 < kend ? 0xffff0000u : 0u);
        mhi = (kk + 8 < kend ? 0x0000ffffu : 0u) | (kk + 9 < kend ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int dd = 0; dd < DT / 2; ++dd) {
        uint32_t r[4];
        ldsm_x4_trans(r, vb + pf_offset<HEAD_DIM>(key, 2 * dd + (lmat >> 1)));
        mma_16816<T>(o[2 * dd], pa[j], r[0] & mlo, r[1] & mhi);
        mma_16816<T>(o[2 * dd + 1], pa[j], r[2] & mlo, r[3] & mhi);
        if constexpr (kBf16) {
          mma_16816<T>(o[2 * dd], pr[j], r[0] & mlo, r[1] & mhi);
          mma_16816<T>(o[2 * dd + 1], pr[j], r[2] & mlo, r[3] & mhi);
        }
      }
    }

    fence_proxy_async_smem();
    __syncthreads();  // every warp is done with this stage
    if (threadIdx.x == 0 && st + PF_STAGES < nst) issue(st + PF_STAGES);
  }

  if (timed_out) {
    bad = true;
    if (threadIdx.x == 0)
      for (int st = consumed; st < min(nst, consumed + PF_STAGES); ++st)
        (void)mbar_wait_bounded(&bars[st % PF_STAGES], (st / PF_STAGES) & 1, WAIT_LIMIT_NS);
  }
  bad = __syncthreads_or(bad) != 0;

  // normalise and store: row sums over the quad, then out = O / l
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    l[ri] += __shfl_xor_sync(FULL_MASK, l[ri], 1);
    l[ri] += __shfl_xor_sync(FULL_MASK, l[ri], 2);
  }
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    if (!rv[ri]) continue;
    const float inv = (bad || ctx_bad) ? NAN : 1.f / l[ri];
    T* dst = static_cast<T*>(p.out) + qrow[ri] * HEAD_DIM;
#pragma unroll
    for (int n = 0; n < DT; ++n)
      *reinterpret_cast<uint32_t*>(dst + 8 * n + 2 * c4) = pack2<T>(o[n][2 * ri] * inv, o[n][2 * ri + 1] * inv);
  }
  allow_dependent_launch();
}

template <typename T, int HEAD_DIM>
cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  using Cfg = PrefillCfg<HEAD_DIM>;
  auto kern = paged_prefill_kernel<T, HEAD_DIM>;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_smem(kern, Cfg::SMEM_BYTES, smem_set);
  if (e != cudaSuccess) return e;
  PrefillParams p;
  const int64_t pool_rows = static_cast<int64_t>(a.num_blocks) * a.block_size;
  e = make_pool_map<T, HEAD_DIM>(&p.tmap_k, a.k_cache, a.num_kv_heads, pool_rows);
  if (e != cudaSuccess) return e;
  e = make_pool_map<T, HEAD_DIM>(&p.tmap_v, a.v_cache, a.num_kv_heads, pool_rows);
  if (e != cudaSuccess) return e;
  p.out = a.out;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.query_start_loc = a.query_start_loc;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_heads = a.num_heads;
  p.group = a.num_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.tile_tokens = PF_ROWS / p.group;
  p.tiles = (a.max_query_len + p.tile_tokens - 1) / p.tile_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (p.tiles == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.tiles, a.num_kv_heads, a.num_seqs);
  cfg.blockDim = dim3(PF_WARPS * 32);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
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
    case 64: return a.use_mma_sync ? launch_prefill_t<T, 64>(a, stream) : launch_prefill_tc_t<T, 64>(a, stream);
    case 128: return a.use_mma_sync ? launch_prefill_t<T, 128>(a, stream) : launch_prefill_tc_t<T, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

}  // namespace pa
