// pa_prefill_tc.cuh -- paged prefill on the tcgen05 tensor cores: S = Q K^T and
// O += P V accumulate in tensor memory (TMEM); the softmax runs on one thread
// per query row between them.
//
//  paged_prefill_tc_kernel  one CTA per (pair of query tiles, KV head,
//                           sequence), one CTA per SM.  A tile is 128 query
//                           rows: 128 / G new tokens of the sequence times the
//                           G query heads of the KV head, loaded by TMA as one
//                           box per 64 dims.  The two tiles of a CTA are
//                           consecutive and share every K and V stage, so the
//                           K/V bytes an SM copies per MMA flop are half of
//                           what one tile per CTA would copy.
//
//  Warps 0-3 run the softmax of tile 0 and warps 4-7 that of tile 1, one
//  thread per query row: they read the row's scores from TMEM, apply the
//  causal mask and the online softmax, and write P back over the scores in
//  TMEM, where the P V MMA reads it as its A operand (P never passes through
//  shared memory, whose bandwidth the Q K^T operands already use).  Warp 8
//  issues the MMAs (one lane).  Warp 9 streams K blocks of 128 keys into a
//  ring of K stages and warp 10 streams V into a ring of its own, each through
//  the block table, read one block ahead; a K stage is free again once both
//  tiles' Q K^T of it are done, a V stage once both P V are.  Warp 10 also
//  zeroes the V rows past the last key of the stream, so that P V never meets
//  stale shared memory (0 x NaN).
//
// TMEM (512 columns, the whole SM): tile u owns columns [256 u, 256 u + 256):
// S of the current block in [0, 128), O in [128, 128 + d).  P is written over
// S as the softmax consumes it, one half of the keys at a time: the P of keys
// [64 h, 64 h + 64) in columns [64 h, 64 h + 32) (bf16: its residual in the
// next 32).  The tensor core runs one CTA's MMAs in issue order, so a tile's
// next Q K^T, issued after its P V, overwrites S only after P V has read P;
// the overlap comes from the two tiles: while one tile's softmax runs, the
// tensor core runs the other tile's P V and Q K^T.  The running maximum used
// for the exponent moves only when a row's maximum grows by more than 2^8
// (then O and l of that row are rescaled in place), so P stays within
// [0, 256] and the rescale is rare.
//
// The method: each new token attends to the positions up to its own
// ("in-depth reading", section 5.1, item 5; "vAttention", paged prefill;
// online softmax of "vLLM PagedAttention source walk-through", section 3.4).
#pragma once

#include "pa_decode.cuh"

namespace pa {

namespace {

constexpr int TC_ROWS = 128;   // query rows per tile (the MMA's M)
constexpr int TC_KEYS = 128;   // keys per stage (the Q K^T MMA's N)
constexpr int TC_HALF = 64;    // keys the softmax holds in registers at a time
constexpr int TC_TILES = 2;    // query tiles per CTA
constexpr float TC_RESCALE_LOG2 = 8.f;  // rescale O when a row maximum grows by more than 2^8

struct PrefillTcParams {
  CUtensorMap tmap_q;  // q as [rows][H][d]: box of 64 dims x G heads x 128 / G rows, 128-byte swizzle
  CUtensorMap tmap_k;  // pools as [N*B rows][Hk][d], 16 x 1 x 64 boxes, 128-byte swizzle
  CUtensorMap tmap_v;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int max_blocks_per_seq;
  int num_heads;
  int group;
  int block_size;
  int num_blocks;
  int pairs;        // CTAs along x: ceil(query tiles / 2)
  int tile_tokens;  // TC_ROWS / group
  float scale_log2;
};

#ifndef PA_TC_MAX_STAGES
#define PA_TC_MAX_STAGES 6
#endif

// Shared memory of one CTA: Q of both tiles, the K and V rings, the barriers.
// The rings take what is left of the 227 KB, up to PA_TC_MAX_STAGES each.
template <typename T, int HEAD_DIM>
struct TcCfg {
  static constexpr bool BF16 = !std::is_same<T, __half>::value;
  static constexpr int SOFT = TC_TILES * TC_ROWS;  // softmax threads
  static constexpr int MMA_WARP = SOFT / 32;
  static constexpr int KLOAD_WARP = MMA_WARP + 1;
  static constexpr int VLOAD_WARP = MMA_WARP + 2;
  static constexpr int THREADS = SOFT + 96;
  static constexpr int DBOX = HEAD_DIM / BOX_DIMS;       // 64-dim atoms per row
  static constexpr int QATOM = TC_ROWS * 128;            // 128 rows x 128 B
  static constexpr int QBYTES = DBOX * QATOM;            // Q of one tile
  static constexpr int KATOM = TC_KEYS * 128;            // 128 keys x 128 B
  static constexpr int KBYTES = DBOX * KATOM;            // K (or V) of one block
  static constexpr int SMEM_MAX = 227 * 1024;
  static constexpr int RESERVE = 1024 + 512;             // base alignment slack, barriers
  static constexpr int FIXED = TC_TILES * QBYTES;
  static constexpr int STAGES_FIT = (SMEM_MAX - RESERVE - FIXED) / KBYTES;
  static constexpr int KSTAGES = STAGES_FIT / 2 < PA_TC_MAX_STAGES ? STAGES_FIT / 2 : PA_TC_MAX_STAGES;
  static constexpr int VSTAGES = STAGES_FIT - KSTAGES < PA_TC_MAX_STAGES ? STAGES_FIT - KSTAGES : PA_TC_MAX_STAGES;
  static_assert(KSTAGES >= 2 && VSTAGES >= 1, "the rings do not fit");
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = TC_TILES * QBYTES;
  static constexpr int V_OFF = K_OFF + KSTAGES * KBYTES;
  static constexpr int BAR_OFF = V_OFF + VSTAGES * KBYTES;
  static constexpr int NBARS = 2 * KSTAGES + 2 * VSTAGES + 3 * TC_TILES + 3;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBARS;  // TMEM base address, then two flags
  static constexpr int LAYOUT_BYTES = SLOT_OFF + 16;
  static constexpr int SMEM_BYTES = LAYOUT_BYTES + 1024;  // + slack to align the base to 1024
  static_assert(SMEM_BYTES <= SMEM_MAX, "shared memory");
  static constexpr uint32_t TMEM_COLS = 512;  // per tile: S / P (128), O (<= 128)
  static constexpr uint32_t ID_S = umma_idesc_f16(TC_ROWS, TC_KEYS, BF16, false);
  static constexpr uint32_t ID_PV = umma_idesc_f16(TC_ROWS, HEAD_DIM, BF16, true);
};

// The waits on the prefill pipeline's critical path.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_bounded(bar, parity, WAIT_LIMIT_NS);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <typename T, int HEAD_DIM>
__global__ void __launch_bounds__(TcCfg<T, HEAD_DIM>::THREADS, 1)
paged_prefill_tc_kernel(const __grid_constant__ PrefillTcParams p) {
  using C = TcCfg<T, HEAD_DIM>;
  constexpr bool BF16 = C::BF16;
  constexpr int DO = HEAD_DIM;  // O columns
  constexpr int KS = C::KSTAGES;
  constexpr int VS = C::VSTAGES;
  constexpr int NSUB = TC_KEYS / CHUNK;  // 16-key boxes per block

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* kfull = bars;                  // [KS] K of a block landed
  uint64_t* kempty = kfull + KS;           // [KS] that block's Q K^T (both tiles) is done
  uint64_t* vfull = kempty + KS;           // [VS] V of a block landed
  uint64_t* vempty = vfull + VS;           // [VS] that block's P V (both tiles) is done
  uint64_t* sfull = vempty + VS;           // [tile] S of the tile's next block is in TMEM
  uint64_t* pfull = sfull + TC_TILES;      // [tile] P of that block is written (128 arrivals)
  uint64_t* pvdone = pfull + TC_TILES;     // [tile] the tile's P V of that block has completed
  uint64_t* qbar = pvdone + TC_TILES;      // Q of both tiles landed
  uint64_t* drain = qbar + 1;              // every MMA issued has completed
  uint64_t* vready = drain + 1;            // the stream's last V stage landed and its tail is zeroed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::SLOT_OFF);
  volatile int* flags = reinterpret_cast<volatile int*>(sm + C::SLOT_OFF + 4);  // [0] bad block, [1] timeout

  const int pair = p.pairs - 1 - static_cast<int>(blockIdx.x);  // the longest pairs start first
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int H = p.num_heads;
  const int tt = p.tile_tokens;

  grid_dependency_wait();  // the cache write before this launch has finished

  const int q0 = __ldg(p.query_start_loc + s);
  const int qlen = __ldg(p.query_start_loc + s + 1) - q0;
  const int ctx = __ldg(p.context_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  const int ta = 2 * pair * tt;  // first new token of tile 0
  if (ta >= qlen) {
    allow_dependent_launch();
    return;
  }
  const int ntiles = ta + tt < qlen ? 2 : 1;
  const bool ctx_bad = ctx < qlen || ctx > cap;
  const int base = ctx - qlen;
  // tile u holds the new tokens [ta + u tt, tile_end(u)) and reads the keys [0, base + tile_end(u))
  auto tile_end = [&](int u) { return min(qlen, ta + (u + 1) * tt); };
  auto tile_blocks = [&](int u) { return ctx_bad ? 0 : (base + tile_end(u) + TC_KEYS - 1) / TC_KEYS; };
  const int kend = ctx_bad ? 0 : base + tile_end(ntiles - 1);  // the K/V stream's last key + 1
  const int nblk = tile_blocks(ntiles - 1);

  // The K load lane sets up the barriers and starts the Q copy at once, so that the
  // copy overlaps the TMEM allocation and the barrier below.
  if (warp == C::KLOAD_WARP && lane == 0) {
    for (int i = 0; i < KS; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < TC_TILES; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], TC_ROWS);
      mbar_init(&pvdone[i], 1);
    }
    mbar_init(qbar, 1);
    mbar_init(drain, 1);
    mbar_init(vready, 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
    if (nblk > 0) {
      mbar_arrive_expect_tx(qbar, ntiles * C::QBYTES);
      for (int u = 0; u < ntiles; ++u)
        for (int db = 0; db < C::DBOX; ++db)
          tma_load_3d(sm + C::Q_OFF + u * C::QBYTES + db * C::QATOM, &p.tmap_q, db * BOX_DIMS, kvh * G,
                      q0 + ta + u * tt, qbar);
    }
  }
  if (warp == 0) tmem_alloc(tslot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == C::KLOAD_WARP || warp == C::VLOAD_WARP) {
    // ------------------------------------------------ loads: warp 9 Q and K, warp 10 V
    const bool is_v = warp == C::VLOAD_WARP;
    const int ns = is_v ? VS : KS;
    uint64_t* fullb = is_v ? vfull : kfull;
    uint64_t* emptyb = is_v ? vempty : kempty;
    const CUtensorMap* map = is_v ? &p.tmap_v : &p.tmap_k;
    uint8_t* ring = sm + (is_v ? C::V_OFF : C::K_OFF);
    int loaded = 0;
    if (lane == 0 && nblk > 0) {
      const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
      // table entry of each box of block j, read a block ahead (the index is clamped to the
      // stream's last key, so that the loads need no select that would wait for them)
      int ph[NSUB];
      auto fetch = [&](int j) {
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) ph[sub] = __ldg(bt + min(j * TC_KEYS + sub * CHUNK, kend - 1) / p.block_size);
      };
      fetch(0);
      for (int j = 0; j < nblk; ++j) {
        const int slot = j % ns;
        if (j >= ns && !tc_wait(&emptyb[slot], ((j / ns) - 1) & 1)) {
          flags[1] = 1;
          break;
        }
        const int nsub = min(NSUB, (kend - j * TC_KEYS + CHUNK - 1) / CHUNK);
        uint8_t* dst = ring + slot * C::KBYTES;
        mbar_arrive_expect_tx(&fullb[slot], nsub * C::DBOX * BOX_BYTES);
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
          if (sub >= nsub) break;
          int phys = ph[sub];
          if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
            flags[0] = 1;  // never read outside the pool; the tiles' outputs become NaN
            phys = 0;
          }
          const int y = phys * p.block_size + (j * TC_KEYS + sub * CHUNK) % p.block_size;
#pragma unroll
          for (int db = 0; db < C::DBOX; ++db)
            tma_load_3d(dst + db * C::KATOM + sub * BOX_BYTES, map, db * BOX_DIMS, kvh, y, &fullb[slot]);
        }
        loaded = j + 1;
        if (loaded < nblk) fetch(loaded);
      }
    }
    if (is_v && nblk > 0) {
      // The keys of the last block past kend hold stale shared memory (or pool rows past the
      // context): zero those V rows once they have landed, before any P V reads them.
      loaded = __shfl_sync(FULL_MASK, loaded, 0);
      if (loaded == nblk) {
        const int j = nblk - 1;
        const int vslot = j % VS;
        const bool ok = __all_sync(FULL_MASK, tc_wait(&vfull[vslot], (j / VS) & 1));
        if (!ok) {
          if (lane == 0) flags[1] = 1;
        } else if (kend < nblk * TC_KEYS) {
          uint8_t* vd = ring + vslot * C::KBYTES;
          const int key_lo = kend - j * TC_KEYS;
          const int units = (TC_KEYS - key_lo) * 8;  // 16-byte units per atom
          for (int i = lane; i < units * C::DBOX; i += 32) {
            const int db = i / units;
            const int rem = i - db * units;
            *reinterpret_cast<uint4*>(vd + db * C::KATOM + (key_lo + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // the zeroed rows become visible to the tensor core
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(vready);
      }
    }
    // the copies in flight land before the shared memory is released
    if (lane == 0)
      for (int j = max(0, loaded - ns); j < loaded; ++j) (void)tc_wait(&fullb[j % ns], (j / ns) & 1);
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------ MMA issue (lane 0)
    // Per block j and tile u: P V(j) once the tile's P(j) is written, then at once the
    // tile's Q K^T(j + 1) into the same columns (issue order keeps them apart), so that
    // the tile's next softmax can start while the other tile's MMAs run.
    if (lane == 0 && nblk > 0) {
      const uint32_t sQ = smem_addr(sm + C::Q_OFF);
      int nbt[TC_TILES];
      for (int u = 0; u < TC_TILES; ++u) nbt[u] = u < ntiles ? tile_blocks(u) : 0;
      int k_seen = -1;  // the last block whose K stage this thread has waited for
      auto wait_k = [&](int j) -> bool {
        if (j <= k_seen) return true;
        if (!tc_wait(&kfull[j % KS], (j / KS) & 1)) return false;
        k_seen = j;
        tc_fence_after_sync();
        return true;
      };
      // The shared-memory descriptors are built once and moved by byte offsets per MMA: the
      // issue of one thread is the MMAs' limit, and rebuilding a descriptor is a dependent
      // chain of integer operations per instruction.
      const uint64_t dq = umma_desc_sw128(sQ, 16, 1024);                                 // Q, K-major
      const uint64_t dk = umma_desc_sw128(smem_addr(sm + C::K_OFF), 16, 1024);           // K, K-major
      const uint64_t dv = umma_desc_sw128(smem_addr(sm + C::V_OFF), C::KATOM, 1024);     // V, MN-major
      auto qk = [&](int u, int j) {
        const uint64_t qu = umma_desc_add(dq, u * C::QBYTES);
        const uint64_t kj = umma_desc_add(dk, (j % KS) * C::KBYTES);
#pragma unroll
        for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::QATOM + ((ks & 3) << 5);  // 16 dims = 32 bytes along a row
          const uint32_t koff = (ks >> 2) * C::KATOM + ((ks & 3) << 5);
          umma_f16(tmem + 256 * u, umma_desc_add(qu, off), umma_desc_add(kj, koff), C::ID_S, ks > 0);
        }
        umma_commit(&sfull[u]);
      };
      bool ok = tc_wait(qbar, 0) && wait_k(0);
      if (ok) {
        for (int u = 0; u < ntiles; ++u) qk(u, 0);
        umma_commit(&kempty[0]);  // the K stage is free once these Q K^T are done
      }
      for (int j = 0; ok && j < nblk; ++j) {
        const int vslot = j % VS;
        bool have_v = false;
        for (int u = 0; u < ntiles; ++u) {
          if (j >= nbt[u]) continue;
          if (!tc_wait(&pfull[u], j & 1)) {
            ok = false;
            break;
          }
          if (!have_v) {  // the last block's V also has its tail zeroed
            if (!(j == nblk - 1 ? tc_wait(vready, 0) : tc_wait(&vfull[vslot], (j / VS) & 1))) {
              ok = false;
              break;
            }
            have_v = true;
          }
          tc_fence_after_sync();
          const uint64_t vj = umma_desc_add(dv, vslot * C::KBYTES);
          const uint32_t tP = tmem + 256 * u;
          const uint32_t tO = tP + 128;
#pragma unroll
          for (int kk = 0; kk < TC_KEYS / 16; ++kk) {  // 16 keys = 8 columns of P
            const uint32_t pcol = 64 * (kk >> 2) + 8 * (kk & 3);
            const uint64_t bdesc = umma_desc_add(vj, kk * 2048);
            umma_f16_ts(tO, tP + pcol, bdesc, C::ID_PV, j > 0 || kk > 0);
            if constexpr (BF16) umma_f16_ts(tO, tP + pcol + 32, bdesc, C::ID_PV, true);
          }
          umma_commit(&pvdone[u]);
          if (j + 1 < nbt[u]) {
            if (!wait_k(j + 1)) {
              ok = false;
              break;
            }
            qk(u, j + 1);
          }
        }
        if (!ok) break;
        umma_commit(&vempty[vslot]);
        if (j + 1 < nblk) umma_commit(&kempty[(j + 1) % KS]);
      }
      if (!ok) flags[1] = 1;
      umma_commit(drain);  // every MMA finishes before the TMEM is released
      if (!tc_wait(drain, 0)) flags[1] = 1;
    }
  } else {
    // ------------------------------------------------ softmax: warps 4 u .. 4 u + 3 run tile u
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 of the tile's columns: row r of tile u
    const int u = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const bool tile_on = u < ntiles;
    const int t0 = ta + u * tt;
    const int t = t0 + r / G;
    const bool rv = tile_on && t < tile_end(u);
    const int pos = rv ? base + t : -1;
    const int nb = tile_on ? tile_blocks(u) : 0;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + 256 * u + lane_off;
    const uint32_t tO = tS + 128;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // log2 units
    // After a wait gives up (ok false, warp-uniform) a warp skips its remaining
    // waits and the tile's results become NaN.
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(FULL_MASK, tc_wait(bar, parity));
    };
    float x[TC_HALF];  // raw scores of one half of the block's keys; masked ones become -inf
    // half h of block j into x, masked
    auto load_half = [&](int j, int h) {
      uint32_t v[TC_HALF / 16][16];
#pragma unroll
      for (int c = 0; c < TC_HALF / 16; ++c) tmem_ld16(tS + TC_HALF * h + 16 * c, v[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < TC_HALF; ++c) x[c] = __uint_as_float(v[c >> 4][c & 15]);
      const int k0 = j * TC_KEYS + TC_HALF * h;
      if (k0 + TC_HALF - 1 > base + t0) {  // a key here may lie past some row of the tile
#pragma unroll
        for (int c = 0; c < TC_HALF; ++c)
          if (k0 + c > pos) x[c] = -INFINITY;
      }
    };
    auto half_max = [&]() {
      float mq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mq[i] = x[i];
#pragma unroll
      for (int c = 4; c < TC_HALF; ++c) mq[c & 3] = fmaxf(mq[c & 3], x[c]);
      return fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
    };
    // the weights of the half in x, written as P over the half's first 32 columns (bf16:
    // the residual over the next 32); returns their float32 sum
    auto half_weights = [&](int h, float nbias) {
      uint32_t w[TC_HALF / 2], wr[BF16 ? TC_HALF / 2 : 1];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < TC_HALF / 2; ++i) {
        const float p0 = ex2(fmaf(x[2 * i], sl2, nbias));
        const float p1 = ex2(fmaf(x[2 * i + 1], sl2, nbias));
        ls[i & 3] += p0 + p1;
        w[i] = pack2<T>(p0, p1);
        if constexpr (BF16) {
          const float2 f2 = unpack2<T>(w[i]);
          wr[i] = pack2<T>(p0 - f2.x, p1 - f2.y);
        }
      }
      tmem_st16(tS + TC_HALF * h, w);
      tmem_st16(tS + TC_HALF * h + 16, w + 16);
      if constexpr (BF16) {
        tmem_st16(tS + TC_HALF * h + 32, wr);
        tmem_st16(tS + TC_HALF * h + 48, wr + 16);
      }
      return (ls[0] + ls[1]) + (ls[2] + ls[3]);
    };
    for (int j = 0; j < nb; ++j) {
      // S of block j is in TMEM; the tile's P V of block j - 1 has completed with it (the
      // tensor core finished every MMA issued before this Q K^T), so O may be read.
      wait(&sfull[u], j & 1);
      tc_fence_after_sync();
      load_half(j, 0);
      float mx = half_max();
      load_half(j, 1);  // half 1 stays in x for its weights
      mx = fmaxf(mx, half_max());
      const float m_new = fmaxf(m_used, mx * sl2);
      // The exponent's offset moves at the first block and when the row maximum has grown
      // by more than 2^8; O and l then scale by f.
      const bool need = j > 0 && m_new > m_used + TC_RESCALE_LOG2;
      const float f = need ? ex2(m_used - m_new) : 1.f;
      if (j == 0 || need) m_used = m_new;
      const float nbias = m_used == -INFINITY ? 0.f : -m_used;  // a row that has seen no key yet
      if (__any_sync(FULL_MASK, need)) {
#pragma unroll 1
        for (int c = 0; c < DO; c += 16) {
          uint32_t o16[16];
          tmem_ld16(tO + c, o16);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] = __float_as_uint(__uint_as_float(o16[i]) * f);
          tmem_st16(tO + c, o16);
        }
      }
      // half 1 first (its scores are in x; its P goes over columns already read), then half 0
      float lsum = half_weights(1, nbias);
      load_half(j, 0);
      lsum += half_weights(0, nbias);
      l = l * f + lsum;
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(&pfull[u]);
    }
    // ------------------------------------------------ O / l, stored after the barrier below
    float o[DO];
    if (nb > 0) wait(&pvdone[u], (nb - 1) & 1);
    const bool have = ok && nb > 0;
    if (have) {
      tc_fence_after_sync();
#pragma unroll
      for (int c = 0; c < DO; c += 16) {
        uint32_t w16[16];
        tmem_ld16(tO + c, w16);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o[c + i] = __uint_as_float(w16[i]);
      }
    }
    if (!ok) flags[1] = 1;
    tc_fence_before_sync();
    __syncthreads();  // the other warps' flags are visible past this point
    if (rv) {
      const float inv = (!have || ctx_bad || flags[0] || flags[1]) ? NAN : 1.f / l;
      T* dst = static_cast<T*>(p.out) + (static_cast<size_t>(q0 + t) * H + kvh * G + r % G) * HEAD_DIM;
#pragma unroll
      for (int c = 0; c < DO; c += 8) {
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w4[i] = have ? pack2<T>(o[c + 2 * i] * inv, o[c + 2 * i + 1] * inv) : pack2<T>(NAN, NAN);
        *reinterpret_cast<uint4*>(dst + c) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
    allow_dependent_launch();
    return;
  }
  // the MMA and load warps meet the softmax warps at their two barriers
  tc_fence_before_sync();
  __syncthreads();
  __syncthreads();
  allow_dependent_launch();
}

}  // namespace

}  // namespace pa
