// pa_prefill_tc.cuh -- paged prefill on the tcgen05 tensor cores: S = Q K^T and
// O += P V accumulate in tensor memory (TMEM); the softmax runs on one thread
// per query row between them.
//
//  paged_prefill_tc_kernel  one CTA per (query tile, KV head, sequence).  A
//                           tile is 128 query rows: 128 / G new tokens of the
//                           sequence times the G query heads of the KV head,
//                           loaded by TMA as one box per 64 dims.  The last
//                           warp loads: lane 0 streams K blocks of 64 keys
//                           through the block table into a ring of K stages,
//                           lane 1 streams V into a ring of its own, so that a
//                           K stage is refilled as soon as its Q K^T is done,
//                           long before that block's P V.  One lane of the
//                           warp before it issues the MMAs.  The softmax warps
//                           (one or two threads per query row) read the row's
//                           scores from TMEM, apply the causal mask and the
//                           online softmax, and write P to shared memory for
//                           the P V MMA.  fp16 at d = 128 runs two CTAs per SM:
//                           one CTA's softmax overlaps the other's MMAs.
//
// The method is the one of paged_prefill_kernel (pa_prefill.cuh): each new
// token attends to the positions up to its own ("in-depth reading", section
// 5.1, item 5; "vAttention", paged prefill; online softmax of "vLLM
// PagedAttention source walk-through", section 3.4).
#pragma once

#include "pa_decode.cuh"

namespace pa {

namespace {

constexpr int TC_ROWS = 128;   // query rows per CTA (the MMA's M)
constexpr int TC_KEYS = 64;    // keys per stage (the Q K^T MMA's N)
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
  int tiles;
  int tile_tokens;  // TC_ROWS / group
  float scale_log2;
};

#ifndef PA_TC16_SPLIT
#define PA_TC16_SPLIT 1
#endif
#ifndef PA_TC16_KSTAGES
#define PA_TC16_KSTAGES 2
#endif
#ifndef PA_TC16_VSTAGES
#define PA_TC16_VSTAGES 2
#endif
#ifndef PA_TC16_PBUFS
#define PA_TC16_PBUFS 1
#endif
#ifndef PA_TC16_CTAS
#define PA_TC16_CTAS 2
#endif

// Shape of one CTA:
//   SPLIT    softmax threads per query row (1: warps 0-3; 2: warps w and w + 4
//            share TMEM lanes 32 (w % 4) .. + 31 and take half the keys each)
//   KSTAGES  K stages in flight: a K stage is free again once its Q K^T is done
//   VSTAGES  V stages in flight: free once the block's P V is done
//   PBUFS    P buffers (2: block j + 1's softmax writes P while block j's P V runs)
//   CTAS     CTAs per SM the shape is sized for (shared memory, TMEM,
//            registers): two CTAs interleave one's softmax with the other's MMAs
// fp16 at d = 128 runs two CTAs per SM; its layout fills the shared memory
// only when the dynamic base is 1024-byte aligned (NOSLACK), which the kernel
// checks before it touches TMA or TMEM.
template <typename T, int HEAD_DIM>
struct TcShape {
  static constexpr bool F16 = std::is_same<T, __half>::value;
  static constexpr bool TUNED = F16 && HEAD_DIM == 128;
  static constexpr int SPLIT = TUNED ? PA_TC16_SPLIT : (F16 ? 1 : (HEAD_DIM == 128 ? 2 : 1));
  static constexpr int KSTAGES = TUNED ? PA_TC16_KSTAGES : 3;
  static constexpr int VSTAGES = TUNED ? PA_TC16_VSTAGES : 3;
  static constexpr int PBUFS = TUNED ? PA_TC16_PBUFS : 2;
  static constexpr int CTAS = TUNED ? PA_TC16_CTAS : (F16 ? 2 : 1);
};

template <typename T, int HEAD_DIM>
struct TcCfg {
  using Shape = TcShape<T, HEAD_DIM>;
  static constexpr int SPLIT = Shape::SPLIT;
  static constexpr int KSTAGES = Shape::KSTAGES;
  static constexpr int VSTAGES = Shape::VSTAGES;
  static constexpr int PBUFS = Shape::PBUFS;
  static constexpr int CTAS = Shape::CTAS;
  static constexpr int SOFT = 128 * SPLIT;               // softmax threads
  static constexpr int THREADS = SOFT + 64;              // + the MMA warp and the load warp
  static constexpr int MMA_WARP = SOFT / 32;
  static constexpr int LOAD_WARP = SOFT / 32 + 1;
  static constexpr int DBOX = HEAD_DIM / BOX_DIMS;       // 64-dim atoms per row
  static constexpr int QATOM = TC_ROWS * 128;            // 128 rows x 128 B
  static constexpr int KATOM = TC_KEYS * 128;            // 64 keys x 128 B
  static constexpr int KBYTES = DBOX * KATOM;            // K (or V) of one block
  static constexpr int PBYTES = TC_ROWS * TC_KEYS * 2;   // one P tile: 128 rows x 64 keys
  static constexpr int NP = std::is_same<T, __half>::value ? 1 : 2;  // bf16: P and its residual
  static constexpr int PBUF = NP * PBYTES;               // one P buffer
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = DBOX * QATOM;
  static constexpr int V_OFF = K_OFF + KSTAGES * KBYTES;
  static constexpr int P_OFF = V_OFF + VSTAGES * KBYTES;
  // SPLIT 2: [2 blocks][2 halves][128 rows] row maxima, then [2 halves][128 rows] row sums
  static constexpr int XCH_OFF = P_OFF + PBUFS * PBUF;
  static constexpr int BAR_OFF = XCH_OFF + (SPLIT == 2 ? 3 * 2 * TC_ROWS * 4 : 0);
  static constexpr int NBARS = 2 * KSTAGES + 2 * VSTAGES + 8;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBARS;     // TMEM base address, then two flags
  static constexpr int LAYOUT_BYTES = SLOT_OFF + 16;
  // the shared memory of one SM (228 KB) holds CTAS CTAs, each with 1 KB reserved
  static constexpr bool NOSLACK = CTAS * (LAYOUT_BYTES + 1024 + 1024) > 228 * 1024;
  static constexpr int SMEM_BYTES = LAYOUT_BYTES + (NOSLACK ? 0 : 1024);
  static_assert(CTAS * (SMEM_BYTES + 1024) <= 228 * 1024, "CTAS CTAs do not fit in one SM");
  static constexpr uint32_t TMEM_COLS = 256;  // S0, S1 (64 each), O (<= 128)
  static_assert(CTAS * TMEM_COLS <= 512, "tensor memory");
  static constexpr uint32_t ID_S = umma_idesc_f16(TC_ROWS, TC_KEYS, !std::is_same<T, __half>::value, false);
  static constexpr uint32_t ID_PV = umma_idesc_f16(TC_ROWS, HEAD_DIM, !std::is_same<T, __half>::value, true);
};

#ifndef PA_TC_WAIT
#define PA_TC_WAIT 0
#endif
// The waits on the prefill pipeline's critical path.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) {
#if PA_TC_WAIT == 0
  return mbar_wait_bounded(bar, parity, WAIT_LIMIT_NS);
#elif PA_TC_WAIT == 1
  return mbar_wait_try(bar, parity, WAIT_LIMIT_NS);
#else
  return mbar_wait_spin(bar, parity, WAIT_LIMIT_NS);
#endif
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <typename T, int HEAD_DIM>
__global__ void __launch_bounds__(TcCfg<T, HEAD_DIM>::THREADS, TcCfg<T, HEAD_DIM>::CTAS)
paged_prefill_tc_kernel(const __grid_constant__ PrefillTcParams p) {
  using C = TcCfg<T, HEAD_DIM>;
  constexpr bool BF16 = !std::is_same<T, __half>::value;
  constexpr int DO = HEAD_DIM;  // O columns
  constexpr int KS = C::KSTAGES;
  constexpr int VS = C::VSTAGES;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const bool misaligned = C::NOSLACK && (smem_addr(smem_raw) & 1023u) != 0;
  uint8_t* sm = smem_raw + (C::NOSLACK ? 0u : ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* kfull = bars;             // [KS] K of a block landed
  uint64_t* kempty = kfull + KS;      // [KS] that block's Q K^T is done
  uint64_t* vfull = kempty + KS;      // [VS] V of a block landed
  uint64_t* vempty = vfull + VS;      // [VS] that block's P V is done
  uint64_t* sfull = vempty + VS;      // [2] S of block j is in TMEM buffer j % 2
  uint64_t* pfull = sfull + 2;        // [2] P of block j is written (C::SOFT arrivals)
  uint64_t* pvdone = pfull + 2;       // [2] P V of block j has completed
  uint64_t* qbar = pvdone + 2;        // Q landed
  uint64_t* drain = qbar + 1;         // every MMA issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::SLOT_OFF);
  volatile int* flags = reinterpret_cast<volatile int*>(sm + C::SLOT_OFF + 4);  // [0] bad block, [1] timeout

  const int tile = p.tiles - 1 - static_cast<int>(blockIdx.x);  // the longest tiles start first
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int H = p.num_heads;

  grid_dependency_wait();  // the cache write before this launch has finished

  const int q0 = __ldg(p.query_start_loc + s);
  const int qlen = __ldg(p.query_start_loc + s + 1) - q0;
  const int ctx = __ldg(p.context_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  const int t0 = tile * p.tile_tokens;
  if (t0 >= qlen) {
    allow_dependent_launch();
    return;
  }
  const int t1 = min(qlen, t0 + p.tile_tokens);
  if (misaligned) {  // the layout needs an aligned base: refuse, with NaN rows
    for (int i = threadIdx.x; i < (t1 - t0) * G * DO; i += blockDim.x) {
      const int row = i / DO;
      static_cast<T*>(p.out)[(static_cast<size_t>(q0 + t0 + row / G) * H + kvh * G + row % G) * DO + i % DO] =
          to_elem<T>(NAN);
    }
    allow_dependent_launch();
    return;
  }
  const bool ctx_bad = ctx < qlen || ctx > cap;
  const int base = ctx - qlen;
  const int kend = ctx_bad ? 0 : base + t1;
  const int nblk = (kend + TC_KEYS - 1) / TC_KEYS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < KS; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], C::SOFT);
      mbar_init(&pvdone[i], 1);
    }
    mbar_init(qbar, 1);
    mbar_init(drain, 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tO = tmem + 128;
  const uint32_t sQ = smem_addr(sm + C::Q_OFF);

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------ loads: lane 0 streams K (and Q), lane 1 V
    if (lane < 2 && nblk > 0) {
      const bool is_v = lane == 1;
      const int ns = is_v ? VS : KS;
      uint64_t* fullb = is_v ? vfull : kfull;
      uint64_t* emptyb = is_v ? vempty : kempty;
      const CUtensorMap* map = is_v ? &p.tmap_v : &p.tmap_k;
      uint8_t* ring = sm + (is_v ? C::V_OFF : C::K_OFF);
      const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
      if (!is_v) {
        mbar_arrive_expect_tx(qbar, C::DBOX * C::QATOM);
        for (int db = 0; db < C::DBOX; ++db)
          tma_load_3d(sm + C::Q_OFF + db * C::QATOM, &p.tmap_q, db * BOX_DIMS, kvh * G, q0 + t0, qbar);
      }
      int loaded = 0;
      for (int j = 0; j < nblk; ++j) {
        const int slot = j % ns;
        if (j >= ns && !tc_wait(&emptyb[slot], ((j / ns) - 1) & 1)) {
          flags[1] = 1;
          break;
        }
        const int nsub = min(TC_KEYS / CHUNK, (kend - j * TC_KEYS + CHUNK - 1) / CHUNK);
        uint8_t* dst = ring + slot * C::KBYTES;
        mbar_arrive_expect_tx(&fullb[slot], nsub * C::DBOX * BOX_BYTES);
        for (int sub = 0; sub < nsub; ++sub) {
          const int key0 = j * TC_KEYS + sub * CHUNK;
          int phys = __ldg(bt + key0 / p.block_size);
          if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
            flags[0] = 1;  // never read outside the pool; the tile's outputs become NaN
            phys = 0;
          }
          const int y = phys * p.block_size + key0 % p.block_size;
#pragma unroll
          for (int db = 0; db < C::DBOX; ++db)
            tma_load_3d(dst + db * C::KATOM + sub * BOX_BYTES, map, db * BOX_DIMS, kvh, y, &fullb[slot]);
        }
        loaded = j + 1;
      }
      // the copies of the last stages land before the shared memory is released
      for (int j = max(0, loaded - ns); j < loaded; ++j) (void)tc_wait(&fullb[j % ns], (j / ns) & 1);
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------ MMA issue (lane 0)
    if (lane == 0 && nblk > 0) {
      bool ok = tc_wait(qbar, 0);
      auto issue_qk = [&](int j) -> bool {
        const int slot = j % KS;
        if (!tc_wait(&kfull[slot], (j / KS) & 1)) return false;
        tc_fence_after_sync();
        const uint32_t kb = smem_addr(sm + C::K_OFF + slot * C::KBYTES);
#pragma unroll
        for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
          const uint32_t off = (ks & 3) << 5;  // 16 dims = 32 bytes along the swizzled row
          umma_f16(tmem + 64 * (j & 1), umma_desc_sw128(sQ + (ks >> 2) * C::QATOM + off, 16, 1024),
                   umma_desc_sw128(kb + (ks >> 2) * C::KATOM + off, 16, 1024), C::ID_S, ks > 0);
        }
        umma_commit(&sfull[j & 1]);
        umma_commit(&kempty[slot]);  // the K stage is free once this Q K^T is done
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && nblk > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < nblk; ++j) {
        const int b = j & 1;
        const int vslot = j % VS;
        if (!tc_wait(&pfull[b], (j >> 1) & 1) || !tc_wait(&vfull[vslot], (j / VS) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t vb = smem_addr(sm + C::V_OFF + vslot * C::KBYTES);
        const uint32_t pb = smem_addr(sm + C::P_OFF + (j % C::PBUFS) * C::PBUF);
#pragma unroll
        for (int kk = 0; kk < TC_KEYS / 16; ++kk) {
          const uint64_t bdesc = umma_desc_sw128(vb + kk * 2048, C::KATOM, 1024);
          umma_f16(tO, umma_desc_sw128(pb + (kk << 5), 16, 1024), bdesc, C::ID_PV, j > 0 || kk > 0);
          if constexpr (BF16)
            umma_f16(tO, umma_desc_sw128(pb + C::PBYTES + (kk << 5), 16, 1024), bdesc, C::ID_PV, true);
        }
        umma_commit(&pvdone[b]);
        umma_commit(&vempty[vslot]);
        if (j + 2 < nblk && !issue_qk(j + 2)) ok = false;
      }
      if (!ok) flags[1] = 1;
      umma_commit(drain);  // every MMA finishes before the TMEM is released
      if (!tc_wait(drain, 0)) flags[1] = 1;
    }
  } else {
    // ------------------------------------------------ softmax: SPLIT threads per query row
    // warp w reads TMEM lanes 32 (w % 4) .. + 31: row r; half h = w / 4 (SPLIT 2) takes keys
    // [32 h, 32 h + 32) of every block and O columns [h DO / 2, (h + 1) DO / 2)
    constexpr int HK = TC_KEYS / C::SPLIT;  // keys of a block this thread scores
    constexpr int HO = DO / C::SPLIT;       // O columns this thread owns
    const int h = C::SPLIT == 2 ? warp >> 2 : 0;
    const int r = 32 * (warp & 3) + lane;
    const int t = t0 + r / G;
    const bool rv = t < t1;
    const int pos = rv ? base + t : -1;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    float* xch = reinterpret_cast<float*>(sm + C::XCH_OFF);  // [block % 2][half][row]
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // log2 units; l over this thread's keys
    // Every softmax thread runs every block, so that all of them meet at the
    // named barrier each time; after a wait gives up (ok false, warp-uniform)
    // a warp skips its remaining waits and its results become NaN.
    bool ok = true;
    auto softmax_sync = []() { asm volatile("bar.sync 1, %0;" ::"n"(C::SOFT) : "memory"); };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(FULL_MASK, tc_wait(bar, parity));
    };
    for (int j = 0; j < nblk; ++j) {
      const int b = j & 1;
      wait(&sfull[b], (j >> 1) & 1);
      tc_fence_after_sync();
      uint32_t v[HK / 16][16];
#pragma unroll
      for (int c = 0; c < HK / 16; ++c) tmem_ld16(tmem + 64 * b + HK * h + lane_off + 16 * c, v[c]);
      tmem_wait_ld();
      float x[HK];  // raw scores of keys k0 + c; masked ones become -inf
#pragma unroll
      for (int c = 0; c < HK; ++c) x[c] = __uint_as_float(v[c >> 4][c & 15]);
      const int k0 = j * TC_KEYS + HK * h;
      if (k0 + HK - 1 > base + t0) {  // a key here may lie past some row of the tile
#pragma unroll
        for (int c = 0; c < HK; ++c)
          if (k0 + c > pos) x[c] = -INFINITY;
      }
      float mq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mq[i] = x[i];
#pragma unroll
      for (int c = 4; c < HK; ++c) mq[c & 3] = fmaxf(mq[c & 3], x[c]);
      float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      if constexpr (C::SPLIT == 2) {
        xch[(b * 2 + h) * TC_ROWS + r] = mx;
        softmax_sync();  // both halves of every row have published their maxima
        mx = fmaxf(mx, xch[(b * 2 + (h ^ 1)) * TC_ROWS + r]);
      }
      const float m_new = fmaxf(m_used, mx * sl2);
      // the P buffer of block j is free once the P V of block j - PBUFS is done
      if (j >= C::PBUFS) {
        const int jj = j - C::PBUFS;
        wait(&pvdone[jj & 1], (jj >> 1) & 1);
      }
      if (j == 0) {
        m_used = m_new;
      } else {
        const bool need = m_new > m_used + TC_RESCALE_LOG2;  // the same for every thread of a row
        if (__any_sync(FULL_MASK, need)) {
          // O must hold the P V of block j - 1 before this warp rescales its rows
          wait(&pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1);
          tc_fence_after_sync();
          const float f = need ? ex2(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < HO; c += 16) {
            uint32_t w[16];
            tmem_ld16(tO + HO * h + lane_off + c, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * f);
            tmem_st16(tO + HO * h + lane_off + c, w);
          }
          tmem_wait_st();
          l *= f;
          if (need) m_used = m_new;
        }
      }
      const float nb = m_used == -INFINITY ? 0.f : -m_used;  // a row that has seen no key yet
      // this thread's keys of the P row (128-byte-swizzled K-major); the sums add the float32 weights
      uint8_t* prow = sm + C::P_OFF + (j % C::PBUFS) * C::PBUF + r * 128;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < HK / 8; ++u) {
        uint32_t w[4], wr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float p0 = ex2(fmaf(x[8 * u + 2 * i], sl2, nb));
          const float p1 = ex2(fmaf(x[8 * u + 2 * i + 1], sl2, nb));
          ls[i] += p0 + p1;
          w[i] = pack2<T>(p0, p1);
          if constexpr (BF16) {
            const float2 f2 = unpack2<T>(w[i]);
            wr[i] = pack2<T>(p0 - f2.x, p1 - f2.y);
          }
        }
        const int pu = (((HK / 8) * h + u) ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(prow + pu) = make_uint4(w[0], w[1], w[2], w[3]);
        if constexpr (BF16) *reinterpret_cast<uint4*>(prow + C::PBYTES + pu) = make_uint4(wr[0], wr[1], wr[2], wr[3]);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // keys at or past kend in the last block hold stale data: zero those V rows
      if (j == nblk - 1 && kend < (j + 1) * TC_KEYS) {
        const int vslot = j % VS;
        wait(&vfull[vslot], (j / VS) & 1);
        uint8_t* vd = sm + C::V_OFF + vslot * C::KBYTES;
        const int key_lo = kend - j * TC_KEYS;
        const int units = (TC_KEYS - key_lo) * 8;  // 16-byte units per atom
        for (int i = threadIdx.x; i < units * C::DBOX; i += C::SOFT) {
          const int db = i / units;
          const int rem = i - db * units;
          *reinterpret_cast<uint4*>(vd + db * C::KATOM + (key_lo + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();  // P (and the zeroed rows) become visible to the tensor core
      tc_fence_before_sync();
      mbar_arrive(&pfull[b]);
    }
    // ------------------------------------------------ O / l, stored after the barrier below
    float o[HO];
    if (nblk > 0) wait(&pvdone[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1);
    const bool have = ok && nblk > 0;
    if (have) {
      tc_fence_after_sync();
#pragma unroll
      for (int c = 0; c < HO; c += 16) {
        uint32_t w[16];
        tmem_ld16(tO + HO * h + lane_off + c, w);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o[c + i] = __uint_as_float(w[i]);
      }
    }
    if constexpr (C::SPLIT == 2) xch[(4 + h) * TC_ROWS + r] = l;  // the row sum is the two halves' sums
    if (!ok) flags[1] = 1;
    tc_fence_before_sync();
    __syncthreads();  // the other warps' flags and the partial sums are visible past this point
    if (rv) {
      float lt = l;
      if constexpr (C::SPLIT == 2) lt += xch[(4 + (h ^ 1)) * TC_ROWS + r];
      const float inv = (!have || ctx_bad || flags[0] || flags[1]) ? NAN : 1.f / lt;
      T* dst = static_cast<T*>(p.out) + (static_cast<size_t>(q0 + t) * H + kvh * G + r % G) * HEAD_DIM + HO * h;
#pragma unroll
      for (int c = 0; c < HO; c += 8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = have ? pack2<T>(o[c + 2 * i] * inv, o[c + 2 * i + 1] * inv) : pack2<T>(NAN, NAN);
        *reinterpret_cast<uint4*>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
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
