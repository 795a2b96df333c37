// pa_prefill_tc.cuh -- paged prefill on the tcgen05 tensor cores: S = Q K^T and
// O += P V accumulate in tensor memory (TMEM); the softmax runs on one thread
// per query row between them.
//
//  paged_prefill_tc_kernel  one CTA per (query tile, KV head, sequence), 320
//                           threads.  A tile is 128 query rows: 128 / G new
//                           tokens of the sequence times the G query heads of
//                           the KV head, loaded by TMA as one box per 64 dims.
//                           Warp 9 loads K/V stages of 64 keys by TMA through
//                           the block table (a 32-lane register window of
//                           block ids); one lane of warp 8 issues the MMAs;
//                           warps 0-7 run the softmax, two threads per query
//                           row (warps w and w + 4 share TMEM lanes 32 (w % 4)
//                           .. + 31 and take half of the keys each): they
//                           read the row's scores, apply the causal mask and
//                           the online softmax, and write P (two buffers) to
//                           shared memory for the P V MMA.
//
// TMEM columns: S of block j in [64 (j % 2), 64 (j % 2) + 64) (two buffers, so
// the next block's Q K^T overlaps this block's softmax), O in [128, 128 + d).
// The running maximum used for the exponent moves only when a row's maximum
// grows by more than 2^8 (then O and l of that row are rescaled in place), so
// P stays within [0, 256] and the rescale is rare.
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
constexpr int TC_SOFT = 256;    // softmax threads: two per query row (warps w and w + 4)
constexpr int TC_THREADS = TC_SOFT + 64;  // + warp 8 (MMA issue) and warp 9 (loads)
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

template <typename T, int HEAD_DIM>
struct TcCfg {
  static constexpr int DBOX = HEAD_DIM / BOX_DIMS;       // 64-dim atoms per row
  static constexpr int QATOM = TC_ROWS * 128;            // 128 rows x 128 B
  static constexpr int KATOM = TC_KEYS * 128;            // 64 keys x 128 B
  static constexpr int KBYTES = DBOX * KATOM;            // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * KBYTES;
  // K/V stages in flight: 4, or 3 where bf16's second P tile would not fit
  static constexpr int STAGES = (std::is_same<T, __half>::value || HEAD_DIM < 128) ? 4 : 3;
  static constexpr int PBYTES = TC_ROWS * TC_KEYS * 2;   // one P tile: 128 rows x 64 keys
  static constexpr int NP = std::is_same<T, __half>::value ? 1 : 2;  // bf16: P and its residual
  static constexpr int PBUF = NP * PBYTES;               // one of the two P buffers
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = DBOX * QATOM;
  static constexpr int P_OFF = KV_OFF + STAGES * STAGE_BYTES;
  static constexpr int XCH_OFF = P_OFF + 2 * PBUF;      // [2 blocks][2 halves][128 rows] float row maxima
  static constexpr int BAR_OFF = XCH_OFF + 2 * 2 * TC_ROWS * 4;
  static constexpr int SMEM_BYTES = 1024 + BAR_OFF + 256;
  static constexpr uint32_t TMEM_COLS = 256;  // S0, S1 (64 each), O (<= 128)
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
__global__ void __launch_bounds__(TC_THREADS, 1)
paged_prefill_tc_kernel(const __grid_constant__ PrefillTcParams p) {
  using C = TcCfg<T, HEAD_DIM>;
  constexpr bool BF16 = !std::is_same<T, __half>::value;
  constexpr int DO = HEAD_DIM;  // O columns

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* full = bars;                   // [C::STAGES] K/V of a stage landed
  uint64_t* empty = bars + C::STAGES;      // [C::STAGES] the stage's MMAs are done
  uint64_t* sfull = bars + 2 * C::STAGES;  // [2] S of block j is in TMEM buffer j % 2
  uint64_t* pfull = sfull + 2;             // [2] P of block j is in buffer j % 2 (TC_SOFT arrivals)
  uint64_t* pvdone = pfull + 2;            // [2] P V of block j (buffer j % 2) has completed
  uint64_t* qbar = pvdone + 2;             // Q landed
  uint64_t* drain = qbar + 1;              // every MMA issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::BAR_OFF + 128);
  volatile int* flags = reinterpret_cast<volatile int*>(sm + C::BAR_OFF + 132);  // [0] bad block, [1] timeout

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
  const bool ctx_bad = ctx < qlen || ctx > cap;
  const int base = ctx - qlen;
  const int kend = ctx_bad ? 0 : base + t1;
  const int nblk = (kend + TC_KEYS - 1) / TC_KEYS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], TC_SOFT);
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
  const uint32_t sP = smem_addr(sm + C::P_OFF);

  if (warp == 9) {
    // ------------------------------------------------ K/V loads (lane 0 issues)
    // lane i holds the physical block of 16-token unit (wbase + i)
    const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
    const int units = (kend + CHUNK - 1) / CHUNK;
    auto win_load = [&](int wbase) -> int {
      const int u = wbase + lane;
      return u < units ? __ldg(bt + (u * CHUNK) / p.block_size) : 0;
    };
    int wbase = 0;
    int win = win_load(0);
    if (lane == 0 && nblk > 0) {
      mbar_arrive_expect_tx(qbar, C::DBOX * C::QATOM);
      for (int db = 0; db < C::DBOX; ++db)
        tma_load_3d(sm + C::Q_OFF + db * C::QATOM, &p.tmap_q, db * BOX_DIMS, kvh * G, q0 + t0, qbar);
    }
    int loaded = 0;
    for (int j = 0; j < nblk; ++j) {
      const int slot = j % C::STAGES;
      if (j >= C::STAGES &&
          !__all_sync(FULL_MASK, tc_wait(&empty[slot], ((j / C::STAGES) - 1) & 1))) {
        if (lane == 0) flags[1] = 1;
        break;
      }
      if (4 * j >= wbase + 32) {  // the next 32 units (8 stages)
        wbase += 32;
        win = win_load(wbase);
      }
      const int nsub = min(TC_KEYS / CHUNK, units - 4 * j);
      uint8_t* kd = sm + C::KV_OFF + slot * C::STAGE_BYTES;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], nsub * 2 * C::DBOX * BOX_BYTES);
      for (int sub = 0; sub < nsub; ++sub) {
        int phys = __shfl_sync(FULL_MASK, win, 4 * j + sub - wbase);
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
          if (lane == 0) flags[0] = 1;  // never read outside the pool; the tile's outputs become NaN
          phys = 0;
        }
        const int key0 = j * TC_KEYS + sub * CHUNK;
        const int y = phys * p.block_size + key0 % p.block_size;
        if (lane == 0) {
#pragma unroll
          for (int db = 0; db < C::DBOX; ++db) {
            tma_load_3d(kd + db * C::KATOM + sub * BOX_BYTES, &p.tmap_k, db * BOX_DIMS, kvh, y, &full[slot]);
            tma_load_3d(kd + C::KBYTES + db * C::KATOM + sub * BOX_BYTES, &p.tmap_v, db * BOX_DIMS, kvh, y,
                        &full[slot]);
          }
        }
      }
      loaded = j + 1;
    }
    // the copies of the last stages land before the shared memory is released
    for (int j = max(0, loaded - C::STAGES); j < loaded; ++j)
      (void)tc_wait(&full[j % C::STAGES], (j / C::STAGES) & 1);
  } else if (warp == 8) {
    // ------------------------------------------------ MMA issue (lane 0)
    if (lane == 0 && nblk > 0) {
      bool ok = tc_wait(qbar, 0);
      auto issue_qk = [&](int j) -> bool {
        const int slot = j % C::STAGES;
        if (!tc_wait(&full[slot], (j / C::STAGES) & 1)) return false;
        tc_fence_after_sync();
        const uint32_t kb = smem_addr(sm + C::KV_OFF + slot * C::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
          const uint32_t off = (ks & 3) << 5;  // 16 dims = 32 bytes along the swizzled row
          umma_f16(tmem + 64 * (j & 1), umma_desc_sw128(sQ + (ks >> 2) * C::QATOM + off, 16, 1024),
                   umma_desc_sw128(kb + (ks >> 2) * C::KATOM + off, 16, 1024), C::ID_S, ks > 0);
        }
        umma_commit(&sfull[j & 1]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && nblk > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < nblk; ++j) {
        const int b = j & 1;
        if (!tc_wait(&pfull[b], (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t vb = smem_addr(sm + C::KV_OFF + (j % C::STAGES) * C::STAGE_BYTES + C::KBYTES);
        const uint32_t pb = sP + b * C::PBUF;
#pragma unroll
        for (int kk = 0; kk < TC_KEYS / 16; ++kk) {
          const uint64_t bdesc = umma_desc_sw128(vb + kk * 2048, C::KATOM, 1024);
          umma_f16(tO, umma_desc_sw128(pb + (kk << 5), 16, 1024), bdesc, C::ID_PV, j > 0 || kk > 0);
          if constexpr (BF16)
            umma_f16(tO, umma_desc_sw128(pb + C::PBYTES + (kk << 5), 16, 1024), bdesc, C::ID_PV, true);
        }
        umma_commit(&pvdone[b]);
        umma_commit(&empty[j % C::STAGES]);
        if (j + 2 < nblk && !issue_qk(j + 2)) ok = false;
      }
      if (!ok) flags[1] = 1;
      umma_commit(drain);  // every MMA finishes before the TMEM is released
      if (!tc_wait(drain, 0)) flags[1] = 1;
    }
  } else {
    // ------------------------------------------------ softmax: two threads per query row
    // warp w (0-7) reads TMEM lanes 32 (w % 4) .. + 31: row r; half h = w / 4 takes keys
    // [32 h, 32 h + 32) of every block and O columns [h DO / 2, (h + 1) DO / 2)
    constexpr int HK = TC_KEYS / 2;
    constexpr int HO = DO / 2;
    const int h = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int t = t0 + r / G;
    const bool rv = t < t1;
    const int pos = rv ? base + t : -1;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    float* xch = reinterpret_cast<float*>(sm + C::XCH_OFF);  // [block % 2][half][row]
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // log2 units; l over this half's keys
    // Every softmax thread runs every block, so that all of them meet at the
    // named barrier each time; after a wait gives up (ok false, warp-uniform)
    // a warp skips its remaining waits and its results become NaN.
    bool ok = true;
    auto softmax_sync = []() { asm volatile("bar.sync 1, %0;" ::"n"(TC_SOFT) : "memory"); };
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
      float x[HK];  // raw scores of keys k0 + HK h + c; masked ones become -inf
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
      xch[(b * 2 + h) * TC_ROWS + r] = mx;
      softmax_sync();  // both halves of every row have published their maxima
      mx = fmaxf(mx, xch[(b * 2 + (h ^ 1)) * TC_ROWS + r]);
      const float m_new = fmaxf(m_used, mx * sl2);
      if (j >= 2) wait(&pvdone[b], ((j - 2) >> 1) & 1);  // P buffer b is free once P V of block j - 2 is done
      if (j == 0) {
        m_used = m_new;
      } else {
        const bool need = m_new > m_used + TC_RESCALE_LOG2;  // the same in both halves of a row
        if (__any_sync(FULL_MASK, need)) {
          // O must hold the P V of block j - 1 before this warp rescales its half rows
          wait(&pvdone[b ^ 1], ((j - 1) >> 1) & 1);
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
      // this half of the P row (32 keys, 64 bytes) into buffer b, 128-byte-swizzled K-major;
      // the sums add the float32 weights
      uint8_t* prow = sm + C::P_OFF + b * C::PBUF + r * 128;
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
        const int pu = ((4 * h + u) ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(prow + pu) = make_uint4(w[0], w[1], w[2], w[3]);
        if constexpr (BF16) *reinterpret_cast<uint4*>(prow + C::PBYTES + pu) = make_uint4(wr[0], wr[1], wr[2], wr[3]);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // keys at or past kend in the last stage hold stale data: zero those V rows
      if (j == nblk - 1 && kend < (j + 1) * TC_KEYS) {
        const int slot = j % C::STAGES;
        wait(&full[slot], (j / C::STAGES) & 1);
        uint8_t* vd = sm + C::KV_OFF + slot * C::STAGE_BYTES + C::KBYTES;
        const int key_lo = kend - j * TC_KEYS;
        const int units = (TC_KEYS - key_lo) * 8;  // 16-byte units per atom
        for (int i = threadIdx.x; i < units * C::DBOX; i += TC_SOFT) {
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
    xch[h * TC_ROWS + r] = l;  // the row sum is the two halves' sums
    tc_fence_before_sync();
    __syncthreads();  // the other warps' flags and the partial sums are visible past this point
    if (rv) {
      const float lt = l + xch[(h ^ 1) * TC_ROWS + r];
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
