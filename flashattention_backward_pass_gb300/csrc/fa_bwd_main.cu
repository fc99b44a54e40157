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
//   warps 4-7   dQ drain (160 registers each via setmaxnreg): TMEM -> registers, release
//               the TMEM columns, then two 32 KB halves through a staging buffer into
//               cp.reduce.async.bulk fp32 adds (ordered by key tile when deterministic)
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
//   K, V, Q[2], dO (128 rows x Dp bf16 each), dS^T (128 keys x 128 queries bf16),
//   dQ staging (128 x 64 fp32)
#include "fa_bwd_common.cuh"

namespace fa {

namespace {

template <int DP>
struct Geo : Panels<DP> {
  using Panels<DP>::TILE_BYTES;
  // shared-memory layout (offsets from a 1024-aligned base)
  static constexpr uint32_t SMALL = 3072;
  static constexpr uint32_t OFF_K = SMALL;
  static constexpr uint32_t OFF_V = OFF_K + TILE_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;            // 2 stages
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * TILE_BYTES;       // 1 stage
  static constexpr uint32_t OFF_DS = OFF_DO + TILE_BYTES;
  static constexpr uint32_t DS_BYTES = 128u * 128u * 2u;
  static constexpr uint32_t OFF_STG = OFF_DS + DS_BYTES;           // dQ reduction staging
  static constexpr uint32_t STG_BYTES = 128u * 64u * 4u;           // 64 fp32 columns
  static constexpr uint32_t TOTAL = OFF_STG + STG_BYTES;
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

// small-region layout
constexpr uint32_t SM_BAR = 0;          // 32 barriers x 8 B
constexpr uint32_t SM_TMEM = 256;       // TMEM base address slot
constexpr uint32_t SM_ABORT = 260;
constexpr uint32_t SM_TILE = 264;       // drain scratch words
constexpr uint32_t SM_RING = 512;       // 2 tile descriptors x 32 B
constexpr uint32_t SM_LSE = 1024;       // 2 stages x 128 fp32
constexpr uint32_t SM_DSUM = 2048;      // 2 stages x 128 fp32

enum Bar : int {
  B_KV = 0, B_QF0, B_QF1, B_QE0, B_QE1, B_DOF0, B_DOF1, B_DOE0, B_DOE1,
  B_SFULL, B_DPFULL, B_PFULL, B_DSFULL, B_DVDONE, B_DQFULL, B_DQEMPTY, B_DSEMPTY,
  B_ACC, B_DRAIN, B_TILEF0, B_TILEF1, B_TILEE0, B_TILEE1, B_KVEMPTY, B_ACCEMPTY, B_NEXT,
  B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area holds 32 mbarriers");

// Consumers of a published tile descriptor: producer, MMA issuer, 4 drain warps and 8
// compute warps each arrive once on the slot's empty barrier.
constexpr int kTileConsumers = 14;

// One key tile of work as the scheduler publishes it in shared memory.
struct TileDesc {
  int valid, n, b, hk, m_begin, m_count, total, pad;
};

// tensor-memory columns
constexpr uint32_t TM_DK = 0, TM_DV = 128, TM_S = 256, TM_DP = 384;

// Error codes written on a timed-out wait (all map to FA_ERR_DEVICE_TIMEOUT on the host;
// the low bits say which wait gave up).
constexpr int kTimeoutBase = -1100;

#ifdef FA_TRACE
// Optional per-phase timestamps (clock64 relative to the CTA's start) of the first
// FA_TRACE_CTAS CTAs, for pipeline tuning.  Off in the normal build.
constexpr int FA_TRACE_CTAS = 4, FA_TRACE_ITERS = 64, FA_TRACE_EV = 12;
__device__ long long g_fa_trace[FA_TRACE_CTAS][FA_TRACE_ITERS][FA_TRACE_EV];
#define FA_TR(ev, it)                                                              \
  do {                                                                             \
    if (blockIdx.x < FA_TRACE_CTAS && (it) < FA_TRACE_ITERS)                       \
      g_fa_trace[blockIdx.x][(it)][(ev)] = clock64() - t_start;                    \
  } while (0)
#else
#define FA_TR(ev, it) \
  do {                \
  } while (0)
#endif

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

// Phase A of one step for one thread (key row = TMEM lane): reads its 64 S^T columns,
// forms P = exp2(S*scale*log2e - LSE2) (softcap: exp2(c*log2e*tanh(S*scale/c) - LSE2)),
// zeroes masked entries (MASK: visible iff qmin <= column <= qmax), writes P^T as bf16
// pairs back over the S^T columns already read (the A operand of dV += P^T dO), and keeps
// P (times 1 - tanh^2 under softcap) as f16 pairs in `pc` for dS.
template <bool MASK, bool SOFTCAP>
__device__ __forceinline__ void phase_p(const SoftmaxConsts& kc, uint32_t taddr, const float* lse,
                                        int qmin, int qmax, uint32_t (&pc)[32]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    uint32_t pk[16];
#pragma unroll
    for (int v4 = 0; v4 < 8; ++v4) {
      const float4 l4 = reinterpret_cast<const float4*>(lse + c * 32)[v4];
      const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
      float pv[4], pcv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ql = c * 32 + v4 * 4 + u;
        float fac;
        float pr = prob<SOFTCAP>(kc, __uint_as_float(r[v4 * 4 + u]), lv[u], &fac);
        if (MASK) pr = (ql >= qmin && ql <= qmax) ? pr : 0.f;
        pv[u] = pr;
        pcv[u] = SOFTCAP ? pr * fac : pr;
      }
      pk[v4 * 2] = pack_bf16(pv[0], pv[1]);
      pk[v4 * 2 + 1] = pack_bf16(pv[2], pv[3]);
      pc[c * 16 + v4 * 2] = pack_f16(pcv[0], pcv[1]);
      pc[c * 16 + v4 * 2 + 1] = pack_f16(pcv[2], pcv[3]);
    }
    tmem_st16(taddr + c * 16, pk);
  }
}

template <int DP, bool SOFTCAP>
__global__ void __launch_bounds__(512, 1)
    bwd_main_kernel(const __grid_constant__ BwdMainParams p,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t,
                    const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdo_t) {
  using G = Geo<DP>;
#ifdef FA_TRACE
  const long long t_start = clock64();
#endif
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
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QF0 + s), 1);
      mbar_init(bar(B_QE0 + s), 1);
      mbar_init(bar(B_DOF0 + s), 1);
      mbar_init(bar(B_DOE0 + s), 1);
      mbar_init(bar(B_TILEF0 + s), 1);
      mbar_init(bar(B_TILEE0 + s), kTileConsumers);
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
    mbar_init(bar(B_KVEMPTY), 1);
    mbar_init(bar(B_ACCEMPTY), 8);
    mbar_init(bar(B_NEXT), 1);
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
  MaskGeom gm;
  gm.Sq = p.Sq;
  gm.Sk = p.Sk;
  gm.lo = p.lo64;
  gm.hi = p.hi64;
  gm.tm = kTileQ;
  gm.tn = kTileK;
  gm.Mb = p.Mb;
  gm.Nb = p.Nb;

  // The CTA is persistent: it takes key tiles from the ticket counter until none are left.
  // A scheduler thread publishes each tile in a 2-slot ring; every role reads tile t from
  // slot t % 2 (full barrier), then frees the slot (empty barrier).  Per-step barriers use
  // a step counter that runs on across tiles (`git`); the K/V buffers and the dK/dV
  // accumulators are handed over between tiles with their own barriers, counted over the
  // tiles that have work (`kt`).
  TileDesc* ring = reinterpret_cast<TileDesc*>(small + SM_RING);
  auto read_tile = [&](int t, TileDesc& d) -> bool {
    const bool ok = mbar_wait(bar(B_TILEF0 + (t & 1)), (t >> 1) & 1, st, kTimeoutBase - 40);
    if (ok) d = ring[t & 1];
    return ok && d.valid;
  };

  // Register split (launch: 512 threads x 128 = 65536): the producer / MMA warpgroup
  // gives registers to the dQ drain warpgroup, which keeps a whole dQ row in registers.
  // 128 * (96 + 160 + 128 + 128) = 65536; the host refuses to launch unless the kernel
  // was compiled to exactly 128 registers per thread, so the split always fits.
  if (warp < 4) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
   if (warp == 2) {
    // ------------------------------------------------------------------ tile scheduler
    if (lane == 0) {
      for (int t = 0;; ++t) {
        const int k = t & 1;
        // Claim the next tile only when the current one is about to run out of work (the
        // producer starts its last step), so that tiles stay in longest-first order across
        // CTAs instead of being claimed a whole tile ahead.
        const bool ready =
            (t == 0 || mbar_wait(bar(B_NEXT), (t - 1) & 1, st, kTimeoutBase - 42)) &&
            (t < 2 || mbar_wait(bar(B_TILEE0 + k), ((t - 2) >> 1) & 1, st, kTimeoutBase - 41));
        if (!ready) {
          ring[k].valid = 0;
          mbar_arrive(bar(B_TILEF0 + k));
          break;
        }
        const int ticket = (*s_abort) ? p.num_tiles : atomicAdd(p.ticket, 1);
        TileDesc d{};
        d.valid = ticket < p.num_tiles;
        if (d.valid) {
          const TileCoord c = decode_tile(p, ticket);
          int64_t mb64, me64;
          m_range(gm, c.n, &mb64, &me64);
          d.n = c.n;
          d.b = c.b;
          d.hk = c.hk;
          d.m_begin = (int)mb64;
          d.m_count = (int)(me64 - mb64);
          d.total = d.m_count * p.G;  // steps (g, m), m fastest
        }
        ring[k] = d;
        mbar_arrive(bar(B_TILEF0 + k));
        if (!d.valid) break;
      }
    }
   } else if (warp == 0) {
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
      int git = 0, kt = 0, ndo = 0;
      bool alive = true;
      for (int t = 0; alive; ++t) {
        TileDesc d;
        if (!read_tile(t, d)) break;
        mbar_arrive(bar(B_TILEE0 + (t & 1)));
        if (d.total == 0) {
          mbar_arrive(bar(B_NEXT));
          continue;
        }
        const int n0 = d.n * kTileK;
        // K and V of the previous tile are free once all of its MMAs are complete
        if (kt > 0 && !mbar_wait(bar(B_KVEMPTY), (kt - 1) & 1, st, kTimeoutBase - 4)) break;
        mbar_arrive_expect_tx(bar(B_KV), 2 * G::TILE_BYTES);
        for (int pnl = 0; pnl < G::NFULL; ++pnl) {
          tma_load_4d(sbase + G::OFF_K + pnl * G::FULL_BYTES, &tk, pnl * 64, d.hk, n0, d.b, bar(B_KV));
          tma_load_4d(sbase + G::OFF_V + pnl * G::FULL_BYTES, &tv, pnl * 64, d.hk, n0, d.b, bar(B_KV));
        }
        if (G::TAIL) {
          tma_load_4d(sbase + G::OFF_K + G::TAIL_OFF, &tk_t, G::NFULL * 64, d.hk, n0, d.b, bar(B_KV));
          tma_load_4d(sbase + G::OFF_V + G::TAIL_OFF, &tv_t, G::NFULL * 64, d.hk, n0, d.b, bar(B_KV));
        }
        ++kt;
        for (int it = 0; it < d.total; ++it, ++git) {
          const int s = git & 1;
          const int g = it / d.m_count;
          const int m = d.m_begin + (it - g * d.m_count);
          const int h = d.hk * p.G + g;
          const int m0 = m * kTileQ;
          if (it == d.total - 1) mbar_arrive(bar(B_NEXT));  // time to claim the next tile
          if (git >= 2 && !mbar_wait(bar(B_QE0 + s), ((git - 2) >> 1) & 1, st, kTimeoutBase - 1)) {
            alive = false;
            break;
          }
          const uint32_t qdst = sbase + G::OFF_Q + s * G::TILE_BYTES;
          mbar_arrive_expect_tx(bar(B_QF0 + s), G::TILE_BYTES + 2 * 512);
          for (int pnl = 0; pnl < G::NFULL; ++pnl)
            tma_load_4d(qdst + pnl * G::FULL_BYTES, &tq, pnl * 64, h, m0, d.b, bar(B_QF0 + s));
          if (G::TAIL) tma_load_4d(qdst + G::TAIL_OFF, &tq_t, G::NFULL * 64, h, m0, d.b, bar(B_QF0 + s));
          const size_t row = ((size_t)d.b * p.H + h) * p.Sq_r + m0;
          bulk_load(sbase + SM_LSE + s * 512, p.lse2 + row, 512, bar(B_QF0 + s));
          bulk_load(sbase + SM_DSUM + s * 512, p.dsum + row, 512, bar(B_QF0 + s));
          FA_TR(10, git);
          // dO has one buffer: dO_i+1 may land once dV_i (its last reader) is complete
          if (git >= 1 && !mbar_wait(bar(B_DOE0), (git - 1) & 1, st, kTimeoutBase - 2)) {
            ++git;
            alive = false;
            break;
          }
          ++ndo;
          const uint32_t ddst = sbase + G::OFF_DO;
          mbar_arrive_expect_tx(bar(B_DOF0), G::TILE_BYTES);
          for (int pnl = 0; pnl < G::NFULL; ++pnl)
            tma_load_4d(ddst + pnl * G::FULL_BYTES, &tdo, pnl * 64, h, m0, d.b, bar(B_DOF0));
          if (G::TAIL) tma_load_4d(ddst + G::TAIL_OFF, &tdo_t, G::NFULL * 64, h, m0, d.b, bar(B_DOF0));
        }
      }
      // Before the CTA may exit, every copy this thread started must have landed (on an
      // abort the consumers may not have waited for them).  Only the latest phase of each
      // barrier can still be pending.
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      if (kt > 0) mbar_wait(bar(B_KV), (kt - 1) & 1, dr, kTimeoutBase - 3);
      for (int s = 0; s < 2; ++s) {
        const int nq = (git - s + 1) / 2;  // loads issued into Q stage s
        if (nq > 0) mbar_wait(bar(B_QF0 + s), (nq - 1) & 1, dr, kTimeoutBase - 3);
      }
      if (ndo > 0) mbar_wait(bar(B_DOF0), (ndo - 1) & 1, dr, kTimeoutBase - 3);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Per tile: S_0, dP_0 (after the previous tile's last dV and drained dQ), then per step i:
    //   dV_i  (needs P^T_i; the first one of a tile also needs the previous tile's dK/dV
    //         read out)                                 -> frees the dO buffer, dv_done
    //   S_i+1 (needs dv_done_i: P^T_i aliases the S^T columns) -- overlaps phase B_i
    //   dK_i, dQ_i (need dS_i)                          -> dq_full
    //   dP_i+1 (needs the dQ_i columns drained)
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_KV = idesc_bf16(128, G::NFULL * 64, false, true);
      constexpr uint32_t ID_KV_T = idesc_bf16(128, G::TAIL ? G::TAIL : 16, false, true);
      constexpr uint32_t ID_Q = idesc_bf16(128, G::NFULL * 64, true, true);
      constexpr uint32_t ID_Q_T = idesc_bf16(128, G::TAIL ? G::TAIL : 16, true, true);
      const uint32_t sK = sbase + G::OFF_K, sV = sbase + G::OFF_V, sDS = sbase + G::OFF_DS;
      const uint32_t sDO = sbase + G::OFF_DO;
      auto issue_S = [&](int g) -> bool {
        const int s = g & 1;
        if (!mbar_wait_spin(bar(B_QF0 + s), (g >> 1) & 1, st, kTimeoutBase - 11)) return false;
        tc_fence_after();
        FA_TR(0, g);
        const uint32_t sQ = sbase + G::OFF_Q + s * G::TILE_BYTES;
        for (int ks = 0; ks < G::KSTEPS; ++ks)
          mma_ss(tmem + TM_S, desc_kmajor<DP>(sK, ks), desc_kmajor<DP>(sQ, ks), ID_S, ks > 0);
        mma_commit(bar(B_SFULL));
        return true;
      };
      auto issue_dP = [&](int g) -> bool {
        if (!mbar_wait_spin(bar(B_DOF0), g & 1, st, kTimeoutBase - 13)) return false;
        tc_fence_after();
        FA_TR(1, g);
        for (int ks = 0; ks < G::KSTEPS; ++ks)
          mma_ss(tmem + TM_DP, desc_kmajor<DP>(sV, ks), desc_kmajor<DP>(sDO, ks), ID_S, ks > 0);
        mma_commit(bar(B_DPFULL));
        return true;
      };
      int git = 0, kt = 0;
      bool ok = true;
      for (int t = 0; ok; ++t) {
        TileDesc d;
        if (!read_tile(t, d)) break;
        mbar_arrive(bar(B_TILEE0 + (t & 1)));
        if (d.total == 0) continue;
        if (!mbar_wait_spin(bar(B_KV), kt & 1, st, kTimeoutBase - 10)) break;
        // the previous tile's last P^T and dQ columns must be consumed before S_0 / dP_0
        if (git > 0 && !mbar_wait_spin(bar(B_DVDONE), (git - 1) & 1, st, kTimeoutBase - 12)) break;
        if (!issue_S(git)) break;
        if (git > 0 && !mbar_wait_spin(bar(B_DQEMPTY), (git - 1) & 1, st, kTimeoutBase - 14)) break;
        if (!issue_dP(git)) break;
        uint32_t acc = 0;
        for (int it = 0; it < d.total; ++it, ++git) {
          const int s = git & 1;
          const uint32_t sQ = sbase + G::OFF_Q + s * G::TILE_BYTES;
          // dV += P^T dO : A = P^T from TMEM (bf16 pairs), K = 128 queries in 8 steps
          if (!mbar_wait_spin(bar(B_PFULL), git & 1, st, kTimeoutBase - 15)) { ok = false; break; }
          // the accumulators are overwritten by this tile's first dV / dK: the previous
          // tile's epilogue must have read them
          if (it == 0 && kt > 0 &&
              !mbar_wait_spin(bar(B_ACCEMPTY), (kt - 1) & 1, st, kTimeoutBase - 18)) {
            ok = false;
            break;
          }
          tc_fence_after();
          FA_TR(2, git);
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a_t = tmem + TM_S + (ks >> 2) * 64 + (ks & 3) * 8;
            const uint32_t en = (acc | (uint32_t)ks) ? 1u : 0u;
            mma_ts(tmem + TM_DV, a_t, desc_mn_full<DP>(sDO, ks), ID_KV, en);
            if (G::TAIL) mma_ts(tmem + TM_DV + G::NFULL * 64, a_t, desc_mn_tail<DP>(sDO, ks), ID_KV_T, en);
          }
          mma_commit(bar(B_DOE0));
          mma_commit(bar(B_DVDONE));
          if (it + 1 < d.total) {
            if (!mbar_wait_spin(bar(B_DVDONE), git & 1, st, kTimeoutBase - 12)) { ok = false; break; }
            if (!issue_S(git + 1)) { ok = false; break; }
          }
          // dK += dS^T Q : A = dS^T (K-major in shared memory), K = 128 queries
          if (!mbar_wait_spin(bar(B_DSFULL), git & 1, st, kTimeoutBase - 16)) { ok = false; break; }
          tc_fence_after();
          FA_TR(3, git);
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
          if (it + 1 < d.total) {
            if (!mbar_wait_spin(bar(B_DQEMPTY), git & 1, st, kTimeoutBase - 14)) { ok = false; break; }
            if (!issue_dP(git + 1)) { ok = false; break; }
          }
        }
        if (!ok) break;
        mma_commit(bar(B_ACC));      // this tile's dK / dV are final
        mma_commit(bar(B_KVEMPTY));  // and its K / V buffers may be refilled
        ++kt;
      }
      if (git > 0 || kt > 0) {
        // every MMA must be complete before the CTA releases tensor memory
        mma_commit(bar(B_DRAIN));
        volatile int no_abort = 0;
        AbortState dr{&no_abort, p.status, p.wait_limit};
        mbar_wait(bar(B_DRAIN), 0, dr, kTimeoutBase - 17);
      }
    }
   }
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 160;" ::: "memory");
    // ------------------------------------------------------------------ dQ drain
    // The whole dQ tile row of this thread (Dp fp32) is loaded from TMEM into registers
    // and the TMEM columns are released at once; the partial then reaches the fp32
    // accumulator through a dedicated staging buffer and bulk fp32 adds, at the L2's pace,
    // without holding anything the main loop needs.  The accumulator tile layout
    // (Dp/4, 128, 4) makes each staged half one contiguous range.
    const int qd = warp & 3;
    const int q = qd * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    volatile int* s_skip = reinterpret_cast<volatile int*>(small + SM_TILE + 4);
    int git = 0;
    for (int t = 0;; ++t) {
      TileDesc d;
      const bool have_tile = __all_sync(0xffffffffu, read_tile(t, d));
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TILEE0 + (t & 1)));
      if (!have_tile) break;
      for (int it = 0; it < d.total; ++it, ++git) {
        const int g = it / d.m_count;
        const int m = d.m_begin + (it - g * d.m_count);
        const int h = d.hk * p.G + g;
        bool ok = warp_wait(bar(B_DQFULL), git & 1, st, kTimeoutBase - 20);
        if (threadIdx.x == 128) FA_TR(8, git);
        uint32_t v[DP];
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < DP / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(t_lane + TM_DP + c * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[c * 32 + e] = r[e];
          }
          if (DP % 32) {
            uint32_t r[16];
            tmem_ld16(t_lane + TM_DP + (DP / 32) * 32, r);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[(DP / 32) * 32 + e] = r[e];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_DQEMPTY));
        }
        if (threadIdx.x == 128) FA_TR(9, git);
        const size_t tile_id = ((size_t)d.b * p.H + h) * p.Mb + m;
        float* dst = p.dq_accum + tile_id * (size_t)(128 * DP);
        int* sem = p.sems + tile_id;
        if (p.deterministic) {
          // Ordered mode: contributions to one dQ tile are added in ascending key-tile
          // order.  No drain thread leaves a step early, so the named barriers of a step
          // are always reached by all 128 drain threads.
          if (threadIdx.x == 128) {
            int stop = (*s_abort) || !ok;
            if (!stop) {
              int64_t nb, ne;
              n_range(gm, m, &nb, &ne);
              const int want = d.n - (int)nb;
              long long t0 = clock64();
              while (true) {
                int cur;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(cur) : "l"(sem) : "memory");
                if (cur == want) {
                  asm volatile("fence.proxy.async.global;" ::: "memory");
                  break;
                }
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
        }
        // Two halves (column groups [0, 16) and [16, Dp/4)) go through the 32 KB staging
        // buffer: all drain threads store a half, one thread issues the bulk fp32 add, and
        // the buffer is reused once the bulk engine has read it.  The bulk engine, not the
        // SM's load/store path, carries the reduction traffic to L2.
        constexpr int CGN = DP / 4;
        constexpr int NH = CGN > 16 ? 2 : 1;
        const uint32_t stg = sbase + G::OFF_STG;
#pragma unroll
        for (int hf = 0; hf < NH; ++hf) {
          const int cg0 = hf * 16;
          const int ncg = (CGN - cg0) < 16 ? (CGN - cg0) : 16;
          // the previous bulk add must have finished reading the buffer
          if (threadIdx.x == 128) bulk_wait_read_all();
          named_bar_sync(1, 128);
          if (ok) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              if (k < ncg) {
                const int cg = cg0 + k;
                st_shared_v4(stg + ((uint32_t)k * 128 + q) * 16, v[4 * cg], v[4 * cg + 1],
                             v[4 * cg + 2], v[4 * cg + 3]);
              }
            }
            fence_proxy_async_smem();
          }
          named_bar_sync(1, 128);
          if (threadIdx.x == 128 && ok) {
            bulk_reduce_add_f32(dst + (size_t)cg0 * 128 * 4, stg, (uint32_t)ncg * 128 * 16);
            bulk_commit();
          }
        }
        if (p.deterministic) {
          if (threadIdx.x == 128) {
            bulk_wait_all();
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __threadfence();
            if (*s_skip == 0)
              asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
          }
        }
        // no early exit: every drain thread reaches every named barrier of every step (on
        // an abort the waits return at once and the stores and bulk adds are skipped)
      }
    }
    if (threadIdx.x == 128) bulk_wait_all();
  } else if (warp >= 8) {
    // ------------------------------------------------------------------ compute
    const int wg = (warp - 8) >> 2;        // query half of the tile
    const int qd = warp & 3;               // TMEM lane quadrant
    const int jl = qd * 32 + lane;         // key row inside the tile = TMEM lane
    const int col0 = wg * 64;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const uint32_t sDS = sbase + G::OFF_DS + wg * 16384 + jl * 128;
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};
    int git = 0, kt = 0;
    bool alive = true;
    for (int t = 0; alive; ++t) {
      TileDesc d;
      const bool have_tile = __all_sync(0xffffffffu, read_tile(t, d));
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TILEE0 + (t & 1)));
      if (!have_tile) break;
      const int j = d.n * kTileK + jl;
      const bool row_ok = j < p.Sk;

      for (int it = 0; it < d.total; ++it, ++git) {
        const int s = git & 1;
        const int g = it / d.m_count;
        const int m = d.m_begin + (it - g * d.m_count);
        const int m0 = m * kTileQ;
        const bool need_mask = !tile_full(gm, m, d.n);
        // visible columns: lo <= (j - i) <= hi with i = m0 + col0 + ql  <=>  ql in [qmin, qmax]
        const int base = j - m0 - col0;
        const int qmin = row_ok ? max(base - p.hi, -1) : 1 << 20;
        const int qmax = row_ok ? min(base - p.lo, 1 << 20) : -1;
        const float* lse = s_lse + s * 128 + col0;
        const float* dsum = s_dsum + s * 128 + col0;

        if (!warp_wait(bar(B_SFULL), git & 1, st, kTimeoutBase - 30)) { alive = false; break; }
        tc_fence_after();
        if (threadIdx.x == 256) FA_TR(4, git);
        uint32_t pc[32];  // P (times 1 - tanh^2 with softcap) as f16 pairs, reused for dS
        if (need_mask)
          phase_p<true, SOFTCAP>(kc, t_lane + TM_S + col0, lse, qmin, qmax, pc);
        else
          phase_p<false, SOFTCAP>(kc, t_lane + TM_S + col0, lse, qmin, qmax, pc);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL));
        if (threadIdx.x == 256) FA_TR(5, git);
        if (threadIdx.x == 384) FA_TR(11, git);

        if (!warp_wait(bar(B_DPFULL), git & 1, st, kTimeoutBase - 31)) { alive = false; break; }
        if (git > 0 && !warp_wait(bar(B_DSEMPTY), (git - 1) & 1, st, kTimeoutBase - 32)) {
          alive = false;
          break;
        }
        tc_fence_after();
        if (threadIdx.x == 256) FA_TR(6, git);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(t_lane + TM_DP + col0 + c * 32, r);
          uint32_t pk[16];
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float4 d4 = reinterpret_cast<const float4*>(dsum + c * 32)[v4];
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int e = v4 * 4 + e2 * 2;
              const float2 pcv = unpack_f16(pc[c * 16 + (e >> 1)]);
              const float d0 = pcv.x * (__uint_as_float(r[e]) - dv[2 * e2]);
              const float d1 = pcv.y * (__uint_as_float(r[e + 1]) - dv[2 * e2 + 1]);
              pk[e >> 1] = pack_bf16(d0, d1);
            }
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
        if (threadIdx.x == 256) FA_TR(7, git);
      }
      if (!alive) break;

      // ---------------------------------------------------------------- dK / dV epilogue
      __nv_bfloat16* outp = wg == 0 ? p.dk : p.dv;
      const int64_t sb = wg == 0 ? p.dk_sb : p.dv_sb;
      const int64_t ss = wg == 0 ? p.dk_ss : p.dv_ss;
      const int64_t sh = wg == 0 ? p.dk_sh : p.dv_sh;
      const float sc = wg == 0 ? p.dk_scale : 1.f;
      const uint32_t tcol = wg == 0 ? TM_DK : TM_DV;
      __nv_bfloat16* rowp = outp + (int64_t)d.b * sb + (int64_t)j * ss + (int64_t)d.hk * sh;
      const bool have = d.total > 0;
      if (have) {
        if (!warp_wait(bar(B_ACC), kt & 1, st, kTimeoutBase - 33)) break;
        tc_fence_after();
      }
      const bool write = __all_sync(0xffffffffu, *s_abort == 0);
#pragma unroll
      for (int c = 0; c < DP / 16; ++c) {
        uint32_t r[16];
        if (have) {
          tmem_ld16(t_lane + tcol + c * 16, r);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0u;
        }
        if (have && c == DP / 16 - 1) {
          // all accumulator columns are read: the next tile's dV / dK may overwrite them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_ACCEMPTY));
        }
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pk[e] = pack_bf16(__uint_as_float(r[2 * e]) * sc, __uint_as_float(r[2 * e + 1]) * sc);
        if (write && row_ok) {
          if (c * 16 < p.D)
            *reinterpret_cast<uint4*>(rowp + c * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          if (c * 16 + 8 < p.D)
            *reinterpret_cast<uint4*>(rowp + c * 16 + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if (have) ++kt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

#ifdef FA_TRACE
cudaError_t bwd_trace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_fa_trace)) bytes = sizeof(g_fa_trace);
  return cudaMemcpyFromSymbol(host, g_fa_trace, bytes);
}
#endif

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
  // The in-kernel register split assumes exactly 128 registers per thread at launch.
  cudaFuncAttributes attr;
  cudaError_t ea = cudaFuncGetAttributes(&attr, kern);
  if (ea != cudaSuccess) return ea;
  if (attr.numRegs != 128) return cudaErrorInvalidConfiguration;
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
