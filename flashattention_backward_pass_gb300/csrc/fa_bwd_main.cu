// fa_bwd_main.cu — the FlashAttention backward main kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// One CTA owns one 128-key tile n of one kv-head (b, hk).  It walks every q-head h of the
// kv-head's group (GQA/MQA page: h_kv = h / (H/Hk)) and every 128-query tile m whose
// (m, n) pair has a visible entry, and per (h, m) it recomputes the probabilities and
// runs the five contractions of the `flash_bwd_sm90.py` page's `mma_one_m_block`:
//
//   S^T  = K Q^T            (M = 128 keys, N = 128 queries, K = Dp)   -> TMEM
//   dP^T = V dO^T           (same shape)                              -> TMEM
//   P    = exp2(S*scale*log2e - LSE2) (mask, softcap), dS = P*(dP - D) (* (1 - tanh^2))
//   dV  += P^T dO           (A = P^T from TMEM, B = dO, N = Dp, K = 128 queries)
//   dK  += dS^T Q           (A = dS^T from shared memory, B = Q)
//   dQ_t = dS K             (M = 128 queries, N = Dp, K = 128 keys)   -> fp32 adds to gmem
//
// dK and dV stay in tensor memory for the CTA's whole life, so the sum over the q-heads
// of the group (the call-trace page's GQA `sum_out`) is done in-kernel and in a fixed
// order.  dK is multiplied by the softmax scale once at the end (as the sm90 page does
// for MHA after its m-block loop); dQ partials are unscaled and the convert kernel
// applies the scale.
//
// Warp roles (16 warps, 512 threads):
//   warp 0      TMA producer: K, V once; Q+LSE2+D and dO per step into 2-stage rings
//   warp 1      TMEM allocator and the single MMA-issuing thread
//   warps 4-7   dQ drain: TMEM -> registers -> red.global.add.v4.f32 (or the ordered
//               path when deterministic)
//   warps 8-15  two compute warpgroups: warpgroup w handles queries [64w, 64w+64) of
//               the tile for every key row (thread = key = TMEM lane); epilogue dK / dV
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0, Dp)        dK accumulator          [128, 128+Dp)  dV accumulator
//   [256, 384)     S^T; P^T (bf16 pairs) is written back over the columns already read
//   [384, 512)     dP^T; reused for the dQ tile once dS has been formed
//
// Shared memory (1024-byte aligned tiles, 128B swizzle for 64-column panels, 32B/64B
// swizzle for a 16/32-column tail panel when Dp % 64 != 0):
//   K, V, Q[2], dO[2] (128 rows x Dp bf16 each), dS^T (128 keys x 128 queries bf16)
#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_tiles.h"

namespace fa {

namespace {

template <int DP>
struct Geo {
  static_assert(DP % 16 == 0 && DP >= 64 && DP <= 128, "Dp in [64, 128], multiple of 16");
  static constexpr int NFULL = DP / 64;        // 64-column panels (128B swizzle)
  static constexpr int TAIL = DP % 64;         // 0, 16 or 32 columns
  static_assert(TAIL == 0 || TAIL == 16 || TAIL == 32, "tail panel of 16 or 32 columns");
  static constexpr uint32_t FULL_BYTES = 128u * 128u;            // 128 rows x 128 B
  static constexpr uint32_t TAIL_ROWB = TAIL * 2;                // bytes per row in tail
  static constexpr uint32_t TAIL_OFF = NFULL * FULL_BYTES;
  static constexpr uint32_t TILE_BYTES = NFULL * FULL_BYTES + 128u * TAIL_ROWB;
  static constexpr uint32_t TAIL_SWZ = TAIL == 16 ? SWZ_32B : SWZ_64B;
  static constexpr int KSTEPS = DP / 16;

  // shared-memory layout (offsets from a 1024-aligned base)
  static constexpr uint32_t SMALL = 3072;
  static constexpr uint32_t OFF_K = SMALL;
  static constexpr uint32_t OFF_V = OFF_K + TILE_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;            // 2 stages
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * TILE_BYTES;       // 2 stages
  static constexpr uint32_t OFF_DS = OFF_DO + 2 * TILE_BYTES;
  static constexpr uint32_t DS_BYTES = 128u * 128u * 2u;
  static constexpr uint32_t TOTAL = OFF_DS + DS_BYTES;
  static_assert(TILE_BYTES % 1024 == 0, "tiles stay 1024-byte aligned");
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

// small-region layout
constexpr uint32_t SM_BAR = 0;          // 32 barriers x 8 B
constexpr uint32_t SM_TMEM = 256;       // TMEM base address slot
constexpr uint32_t SM_ABORT = 260;
constexpr uint32_t SM_TILE = 264;       // ticket -> tile id
constexpr uint32_t SM_LSE = 1024;       // 2 stages x 128 fp32
constexpr uint32_t SM_DSUM = 2048;      // 2 stages x 128 fp32

enum Bar : int {
  B_KV = 0, B_QF0, B_QF1, B_QE0, B_QE1, B_DOF0, B_DOF1, B_DOE0, B_DOE1,
  B_SFULL, B_DPFULL, B_PFULL, B_DSFULL, B_DVDONE, B_DQFULL, B_DQEMPTY, B_DSEMPTY,
  B_ACC, B_DRAIN, B_COUNT
};

// tensor-memory columns
constexpr uint32_t TM_DK = 0, TM_DV = 128, TM_S = 256, TM_DP = 384;

// Error codes written on a timed-out wait (all map to FA_ERR_DEVICE_TIMEOUT on the host;
// the low bits say which wait gave up).
constexpr int kTimeoutBase = -1100;

// K-major operand, 128 rows, K-step ks (16 columns) of a Dp-wide tile.
template <int DP>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int ks) {
  using G = Geo<DP>;
  if (ks < G::NFULL * 4) {
    uint32_t addr = tile + (ks >> 2) * G::FULL_BYTES + (ks & 3) * 32;
    return smem_desc(addr, 16, 1024, SWZ_128B);
  }
  int kk = ks - G::NFULL * 4;
  uint32_t addr = tile + G::TAIL_OFF + kk * 32;
  return smem_desc(addr, 16, 8 * G::TAIL_ROWB, G::TAIL_SWZ);
}

// MN-major operand whose rows are the contraction index (16 rows per K-step) and whose
// columns (Dp wide) are N: descriptor for the 64-column panels (all of them, LBO = panel
// stride) or for the tail panel.
template <int DP>
__device__ __forceinline__ uint64_t desc_mn_full(uint32_t tile, int ks) {
  return smem_desc(tile + ks * 16 * 128, Geo<DP>::FULL_BYTES, 1024, SWZ_128B);
}
template <int DP>
__device__ __forceinline__ uint64_t desc_mn_tail(uint32_t tile, int ks) {
  using G = Geo<DP>;
  return smem_desc(tile + G::TAIL_OFF + ks * 16 * G::TAIL_ROWB, 128u * G::TAIL_ROWB,
                   8 * G::TAIL_ROWB, G::TAIL_SWZ);
}

// Every lane waits (each needs the barrier's acquire), then the warp agrees: a lane
// that saw the abort flag makes the whole warp stop, so .sync.aligned tcgen05 ops that
// follow are always executed by all 32 lanes or by none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const AbortState& st,
                                          int code) {
  const bool ok = mbar_wait(bar, parity, st, code);
  return __all_sync(0xffffffffu, ok);
}

struct TileCoord {
  int n, b, hk;
};

__device__ __forceinline__ TileCoord decode_tile(const BwdMainParams& p, int t) {
  // key-tile-major order: all (b, hk) of key tile 0 first.  Under causal masking the low
  // key tiles see the most query tiles, so the longest work starts first, and in the
  // deterministic mode every tile a CTA waits for was claimed by a running CTA.
  TileCoord c;
  int per_n = p.B * p.Hk;
  c.n = t / per_n;
  int r = t - c.n * per_n;
  c.b = r / p.Hk;
  c.hk = r - c.b * p.Hk;
  return c;
}

}  // namespace

template <int DP, bool SOFTCAP>
__global__ void __launch_bounds__(512, 1)
    bwd_main_kernel(const __grid_constant__ BwdMainParams p,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t,
                    const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdo_t) {
  using G = Geo<DP>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* small = smem_raw;
  volatile int* s_abort = reinterpret_cast<volatile int*>(small + SM_ABORT);
  volatile int* s_tile = reinterpret_cast<volatile int*>(small + SM_TILE);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(small + SM_TMEM);
  const float* s_lse = reinterpret_cast<const float*>(small + SM_LSE);
  const float* s_dsum = reinterpret_cast<const float*>(small + SM_DSUM);
  auto bar = [&](int i) -> uint32_t { return sbase + SM_BAR + 8u * i; };

  if (threadIdx.x == 0) {
    *s_abort = 0;
    if ((sbase & 1023u) != 0) {
      // the tile layout assumes a 1024-byte aligned dynamic shared-memory base
      atomicExch(p.status, kTimeoutBase - 99);
      *s_abort = 1;
    }
    *s_tile = atomicAdd(p.ticket, 1);
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QF0 + s), 1);
      mbar_init(bar(B_QE0 + s), 1);
      mbar_init(bar(B_DOF0 + s), 1);
      mbar_init(bar(B_DOE0 + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_DSFULL), 8);
    mbar_init(bar(B_DVDONE), 1);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQEMPTY), 4);
    mbar_init(bar(B_DSEMPTY), 1);
    mbar_init(bar(B_ACC), 1);
    mbar_init(bar(B_DRAIN), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + SM_TMEM, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = *s_tmem;
  AbortState st{s_abort, p.status, p.wait_limit};

  const TileCoord tc = decode_tile(p, *s_tile);
  MaskGeom gm;
  gm.Sq = p.Sq;
  gm.Sk = p.Sk;
  gm.lo = p.lo64;
  gm.hi = p.hi64;
  gm.tm = kTileQ;
  gm.tn = kTileK;
  gm.Mb = p.Mb;
  gm.Nb = p.Nb;
  int64_t mb64, me64;
  m_range(gm, tc.n, &mb64, &me64);
  const int m_begin = (int)mb64;
  const int m_count = (int)(me64 - mb64);
  const int total = (*s_abort) ? 0 : m_count * p.G;  // steps: (g, m) with m fastest
  const int n0 = tc.n * kTileK;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      if (G::TAIL) {
        tma_prefetch_desc(&tq_t);
        tma_prefetch_desc(&tk_t);
        tma_prefetch_desc(&tv_t);
        tma_prefetch_desc(&tdo_t);
      }
      int issued_q[2] = {0, 0}, issued_do[2] = {0, 0};
      bool kv_issued = false;
      if (total > 0) {
        mbar_arrive_expect_tx(bar(B_KV), 2 * G::TILE_BYTES);
        for (int pnl = 0; pnl < G::NFULL; ++pnl) {
          tma_load_4d(sbase + G::OFF_K + pnl * G::FULL_BYTES, &tk, pnl * 64, tc.hk, n0, tc.b,
                      bar(B_KV));
          tma_load_4d(sbase + G::OFF_V + pnl * G::FULL_BYTES, &tv, pnl * 64, tc.hk, n0, tc.b,
                      bar(B_KV));
        }
        if (G::TAIL) {
          tma_load_4d(sbase + G::OFF_K + G::TAIL_OFF, &tk_t, G::NFULL * 64, tc.hk, n0, tc.b,
                      bar(B_KV));
          tma_load_4d(sbase + G::OFF_V + G::TAIL_OFF, &tv_t, G::NFULL * 64, tc.hk, n0, tc.b,
                      bar(B_KV));
        }
        kv_issued = true;
      }
      for (int it = 0; it < total; ++it) {
        const int s = it & 1;
        const int g = it / m_count;
        const int m = m_begin + (it - g * m_count);
        const int h = tc.hk * p.G + g;
        const int m0 = m * kTileQ;
        if (it >= 2 && !mbar_wait(bar(B_QE0 + s), ((it - 2) >> 1) & 1, st, kTimeoutBase - 1)) break;
        const uint32_t qdst = sbase + G::OFF_Q + s * G::TILE_BYTES;
        mbar_arrive_expect_tx(bar(B_QF0 + s), G::TILE_BYTES + 2 * 512);
        for (int pnl = 0; pnl < G::NFULL; ++pnl)
          tma_load_4d(qdst + pnl * G::FULL_BYTES, &tq, pnl * 64, h, m0, tc.b, bar(B_QF0 + s));
        if (G::TAIL) tma_load_4d(qdst + G::TAIL_OFF, &tq_t, G::NFULL * 64, h, m0, tc.b, bar(B_QF0 + s));
        const size_t row = ((size_t)tc.b * p.H + h) * p.Sq_r + m0;
        bulk_load(sbase + SM_LSE + s * 512, p.lse2 + row, 512, bar(B_QF0 + s));
        bulk_load(sbase + SM_DSUM + s * 512, p.dsum + row, 512, bar(B_QF0 + s));
        issued_q[s] = it / 2 + 1;

        if (it >= 2 && !mbar_wait(bar(B_DOE0 + s), ((it - 2) >> 1) & 1, st, kTimeoutBase - 2)) break;
        const uint32_t ddst = sbase + G::OFF_DO + s * G::TILE_BYTES;
        mbar_arrive_expect_tx(bar(B_DOF0 + s), G::TILE_BYTES);
        for (int pnl = 0; pnl < G::NFULL; ++pnl)
          tma_load_4d(ddst + pnl * G::FULL_BYTES, &tdo, pnl * 64, h, m0, tc.b, bar(B_DOF0 + s));
        if (G::TAIL) tma_load_4d(ddst + G::TAIL_OFF, &tdo_t, G::NFULL * 64, h, m0, tc.b, bar(B_DOF0 + s));
        issued_do[s] = it / 2 + 1;
      }
      // Before the CTA may exit, every copy this thread started must have landed (on an
      // abort the consumers may not have waited for them).
      AbortState drain{s_abort, p.status, p.wait_limit};
      volatile int no_abort = 0;
      drain.cta_abort = &no_abort;
      if (kv_issued) mbar_wait(bar(B_KV), 0, drain, kTimeoutBase - 3);
      for (int s = 0; s < 2; ++s) {
        if (issued_q[s]) mbar_wait(bar(B_QF0 + s), (issued_q[s] - 1) & 1, drain, kTimeoutBase - 3);
        if (issued_do[s]) mbar_wait(bar(B_DOF0 + s), (issued_do[s] - 1) & 1, drain, kTimeoutBase - 3);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_KV = idesc_bf16(128, G::NFULL * 64, false, true);
      constexpr uint32_t ID_KV_T = idesc_bf16(128, G::TAIL ? G::TAIL : 16, false, true);
      constexpr uint32_t ID_Q = idesc_bf16(128, G::NFULL * 64, true, true);
      constexpr uint32_t ID_Q_T = idesc_bf16(128, G::TAIL ? G::TAIL : 16, true, true);
      const uint32_t sK = sbase + G::OFF_K, sV = sbase + G::OFF_V, sDS = sbase + G::OFF_DS;
      uint32_t acc = 0;
      bool issued_any = false;
      for (int it = 0; it < total; ++it) {
        const int s = it & 1;
        const uint32_t ph2 = (it >> 1) & 1;
        const uint32_t sQ = sbase + G::OFF_Q + s * G::TILE_BYTES;
        const uint32_t sDO = sbase + G::OFF_DO + s * G::TILE_BYTES;
        if (it == 0 && !mbar_wait(bar(B_KV), 0, st, kTimeoutBase - 10)) break;
        if (!mbar_wait(bar(B_QF0 + s), ph2, st, kTimeoutBase - 11)) break;
        // P^T of the previous step (aliasing the S^T columns) must have been consumed
        if (it > 0 && !mbar_wait(bar(B_DVDONE), (it - 1) & 1, st, kTimeoutBase - 12)) break;
        tc_fence_after();
        for (int ks = 0; ks < G::KSTEPS; ++ks)
          mma_ss(tmem + TM_S, desc_kmajor<DP>(sK, ks), desc_kmajor<DP>(sQ, ks), ID_S, ks > 0);
        mma_commit(bar(B_SFULL));
        issued_any = true;

        if (!mbar_wait(bar(B_DOF0 + s), ph2, st, kTimeoutBase - 13)) break;
        // the previous dQ tile (aliasing the dP^T columns) must have been drained
        if (it > 0 && !mbar_wait(bar(B_DQEMPTY), (it - 1) & 1, st, kTimeoutBase - 14)) break;
        tc_fence_after();
        for (int ks = 0; ks < G::KSTEPS; ++ks)
          mma_ss(tmem + TM_DP, desc_kmajor<DP>(sV, ks), desc_kmajor<DP>(sDO, ks), ID_S, ks > 0);
        mma_commit(bar(B_DPFULL));

        // dV += P^T dO : A = P^T from TMEM (bf16 pairs), K = 128 queries in 8 steps
        if (!mbar_wait(bar(B_PFULL), it & 1, st, kTimeoutBase - 15)) break;
        tc_fence_after();
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a_t = tmem + TM_S + (ks >> 2) * 64 + (ks & 3) * 8;
          const uint32_t en = (acc | (uint32_t)ks) ? 1u : 0u;
          mma_ts(tmem + TM_DV, a_t, desc_mn_full<DP>(sDO, ks), ID_KV, en);
          if (G::TAIL) mma_ts(tmem + TM_DV + G::NFULL * 64, a_t, desc_mn_tail<DP>(sDO, ks), ID_KV_T, en);
        }
        mma_commit(bar(B_DOE0 + s));
        mma_commit(bar(B_DVDONE));

        // dK += dS^T Q : A = dS^T (K-major in shared memory), K = 128 queries
        if (!mbar_wait(bar(B_DSFULL), it & 1, st, kTimeoutBase - 16)) break;
        tc_fence_after();
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a = smem_desc(sDS + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, SWZ_128B);
          const uint32_t en = (acc | (uint32_t)ks) ? 1u : 0u;
          mma_ss(tmem + TM_DK, a, desc_mn_full<DP>(sQ, ks), ID_KV, en);
          if (G::TAIL) mma_ss(tmem + TM_DK + G::NFULL * 64, a, desc_mn_tail<DP>(sQ, ks), ID_KV_T, en);
        }
        mma_commit(bar(B_QE0 + s));
        // dQ tile = dS K : A = dS (M = queries, MN-major), B = K (N = Dp, MN-major), K = keys
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a = smem_desc(sDS + ks * 16 * 128, 16384, 1024, SWZ_128B);
          mma_ss(tmem + TM_DP, a, desc_mn_full<DP>(sK, ks), ID_Q, ks > 0);
          if (G::TAIL) mma_ss(tmem + TM_DP + G::NFULL * 64, a, desc_mn_tail<DP>(sK, ks), ID_Q_T, ks > 0);
        }
        mma_commit(bar(B_DQFULL));
        mma_commit(bar(B_DSEMPTY));
        acc = 1;
      }
      mma_commit(bar(B_ACC));
      if (issued_any) {
        // every MMA must be complete before the CTA releases tensor memory
        mma_commit(bar(B_DRAIN));
        AbortState drain{s_abort, p.status, p.wait_limit};
        volatile int no_abort = 0;
        drain.cta_abort = &no_abort;
        mbar_wait(bar(B_DRAIN), 0, drain, kTimeoutBase - 17);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ dQ drain
    const int qd = warp & 3;
    const int q = qd * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    volatile int* s_skip = reinterpret_cast<volatile int*>(small + SM_TILE + 4);
    for (int it = 0; it < total; ++it) {
      const int g = it / m_count;
      const int m = m_begin + (it - g * m_count);
      const int h = tc.hk * p.G + g;
      bool ok = warp_wait(bar(B_DQFULL), it & 1, st, kTimeoutBase - 20);
      const size_t tile_id = ((size_t)tc.b * p.H + h) * p.Mb + m;
      float* dst = p.dq_accum + tile_id * (size_t)(128 * DP);
      int* sem = p.sems + tile_id;
      if (p.deterministic) {
        // Ordered mode: contributions to one dQ tile are added in ascending key-tile
        // order.  No thread leaves this loop early, so the two named barriers per step
        // are always reached by all 128 drain threads.
        if (threadIdx.x == 128) {
          int stop = *s_abort;
          if (!stop) {
            int64_t nb, ne;
            n_range(gm, m, &nb, &ne);
            const int want = tc.n - (int)nb;
            long long t0 = clock64();
            while (true) {
              int cur;
              asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(cur) : "l"(sem) : "memory");
              if (cur == want) break;
              if (*s_abort) { stop = 1; break; }
              if (clock64() - t0 > p.wait_limit) {
                raise_timeout(st, kTimeoutBase - 21);
                stop = 1;
                break;
              }
            }
          }
          *s_skip = stop;
        }
        named_bar_sync(1, 128);
        ok = ok && (*s_skip == 0);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DP / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(t_lane + TM_DP + c * 16, r);
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            const int cg = c * 4 + g4;
            red_add_v4(dst + ((size_t)cg * 128 + q) * 4, __uint_as_float(r[4 * g4]),
                       __uint_as_float(r[4 * g4 + 1]), __uint_as_float(r[4 * g4 + 2]),
                       __uint_as_float(r[4 * g4 + 3]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DQEMPTY));
      }
      if (p.deterministic) {
        __threadfence();
        named_bar_sync(1, 128);
        if (threadIdx.x == 128 && *s_skip == 0)
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
      } else if (!ok) {
        break;
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------------ compute
    const int wg = (warp - 8) >> 2;        // query half of the tile
    const int qd = warp & 3;               // TMEM lane quadrant
    const int jl = qd * 32 + lane;         // key row inside the tile = TMEM lane
    const int col0 = wg * 64;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const uint32_t sDS = sbase + G::OFF_DS + wg * 16384 + jl * 128;
    const int j = n0 + jl;
    const bool row_ok = j < p.Sk;

    for (int it = 0; it < total; ++it) {
      const int s = it & 1;
      const int g = it / m_count;
      const int m = m_begin + (it - g * m_count);
      const int m0 = m * kTileQ;
      const bool need_mask = !tile_full(gm, m, tc.n);
      const int base = j - m0 - col0;       // (j - i) = base - local query index
      const float* lse = s_lse + s * 128 + col0;
      const float* dsum = s_dsum + s * 128 + col0;

      if (!warp_wait(bar(B_SFULL), it & 1, st, kTimeoutBase - 30)) break;
      tc_fence_after();
      uint32_t pc[32];  // P (times 1 - tanh^2 with softcap) as f16 pairs, reused for dS
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(t_lane + TM_S + col0 + c * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pv[2], pcv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int ql = c * 32 + e + u;
            const float sv = __uint_as_float(r[e + u]);
            float pr, fac = 1.f;
            if (SOFTCAP) {
              const float t = tanh_exp2(sv * p.cap_scale);
              pr = ex2_approx(fmaf(t, p.cap_log2, -lse[ql]));
              fac = fmaf(-t, t, 1.f);
            } else {
              pr = ex2_approx(fmaf(sv, p.scale_log2, -lse[ql]));
            }
            if (need_mask) {
              const int d = base - ql;
              const bool vis = row_ok && d >= p.lo && d <= p.hi;
              pr = vis ? pr : 0.f;
            }
            pv[u] = pr;
            pcv[u] = pr * fac;
          }
          pk[e >> 1] = pack_bf16(pv[0], pv[1]);
          pc[c * 16 + (e >> 1)] = pack_f16(pcv[0], pcv[1]);
        }
        tmem_st16(t_lane + TM_S + col0 + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));

      if (!warp_wait(bar(B_DPFULL), it & 1, st, kTimeoutBase - 31)) break;
      if (it > 0 && !warp_wait(bar(B_DSEMPTY), (it - 1) & 1, st, kTimeoutBase - 32)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(t_lane + TM_DP + col0 + c * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 pcv = unpack_f16(pc[c * 16 + (e >> 1)]);
          const int ql = c * 32 + e;
          const float d0 = pcv.x * (__uint_as_float(r[e]) - dsum[ql]);
          const float d1 = pcv.y * (__uint_as_float(r[e + 1]) - dsum[ql + 1]);
          pk[e >> 1] = pack_bf16(d0, d1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t chunk = (uint32_t)(c * 4 + u) ^ (uint32_t)(jl & 7);
          st_shared_v4(sDS + chunk * 16, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DSFULL));
    }

    // ------------------------------------------------------------------ dK / dV epilogue
    __nv_bfloat16* outp = wg == 0 ? p.dk : p.dv;
    const int64_t sb = wg == 0 ? p.dk_sb : p.dv_sb;
    const int64_t ss = wg == 0 ? p.dk_ss : p.dv_ss;
    const int64_t sh = wg == 0 ? p.dk_sh : p.dv_sh;
    const float sc = wg == 0 ? p.dk_scale : 1.f;
    const uint32_t tcol = wg == 0 ? TM_DK : TM_DV;
    __nv_bfloat16* rowp = outp + (int64_t)tc.b * sb + (int64_t)j * ss + (int64_t)tc.hk * sh;
    bool have = false;
    if (total > 0) have = warp_wait(bar(B_ACC), 0, st, kTimeoutBase - 33);
    if (have) tc_fence_after();
    const bool write = __all_sync(0xffffffffu, *s_abort == 0);
    if (write) {
#pragma unroll
      for (int c = 0; c < DP / 16; ++c) {
        uint32_t r[16];
        if (have) {
          tmem_ld16(t_lane + tcol + c * 16, r);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0u;
        }
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pk[e] = pack_bf16(__uint_as_float(r[2 * e]) * sc, __uint_as_float(r[2 * e + 1]) * sc);
        if (row_ok) {
          if (c * 16 < p.D)
            *reinterpret_cast<uint4*>(rowp + c * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          if (c * 16 + 8 < p.D)
            *reinterpret_cast<uint4*>(rowp + c * 16 + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t bwd_main_smem_bytes(int Dp) {
  switch (Dp) {
    case 64: return Geo<64>::TOTAL;
    case 80: return Geo<80>::TOTAL;
    case 96: return Geo<96>::TOTAL;
    case 128: return Geo<128>::TOTAL;
    default: return 0;
  }
}

template <int DP, bool SC>
static cudaError_t launch_one(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                              const OperandMaps& v, const OperandMaps& d, int num_ctas,
                              cudaStream_t s) {
  auto kern = bwd_main_kernel<DP, SC>;
  const size_t smem = Geo<DP>::TOTAL;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_ctas, 512, smem, s>>>(p, q.full, q.tail, k.full, k.tail, v.full, v.tail, d.full, d.tail);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                            const OperandMaps& v, const OperandMaps& d, int Dp, bool softcap,
                            int num_ctas, cudaStream_t s) {
  if (num_ctas <= 0) return cudaSuccess;
#define FA_CASE(DPV)                                                          \
  case DPV:                                                                   \
    return softcap ? launch_one<DPV, true>(p, q, k, v, d, num_ctas, s)        \
                   : launch_one<DPV, false>(p, q, k, v, d, num_ctas, s);
  switch (Dp) {
    FA_CASE(64)
    FA_CASE(80)
    FA_CASE(96)
    FA_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef FA_CASE
}

}  // namespace fa
