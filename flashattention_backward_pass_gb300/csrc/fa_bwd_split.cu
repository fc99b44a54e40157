// fa_bwd_split.cu — the backward as two tcgen05 kernels with no atomics and no fp32 dQ
// accumulator in global memory.
//
// dK/dV kernel: one CTA owns a 128-key tile of one kv-head and walks the q-heads of its
// group and the query tiles with a visible entry, as in the `flash_bwd_sm90.py` page's
// `mma_one_m_block` minus the dQ product:
//   S^T = K Q^T, dP^T = V dO^T                        (tcgen05, fp32 in TMEM)
//   P^T = exp2(S^T*scale*log2e - LSE2)  -> bf16 over the S^T columns (A of dV)
//   dS^T = P^T*(dP^T - D) (* (1 - tanh^2))  -> bf16 over the dP^T columns (A of dK)
//   dV += P^T dO,  dK += dS^T Q                      (A operands straight from TMEM)
// dK/dV stay in TMEM over the whole GQA group (the call-trace page's `sum_out`, done
// in-kernel), dK gets the softmax scale once at the end.
//
// dQ kernel: persistent CTAs claim 128-query tiles of one q-head each and walk the key
// tiles with a visible entry (the Triton page's `_bwd_kernel_dq` loop, recomputing P):
//   S = Q K^T, dP = dO V^T, dS = P*(dP - D) -> bf16 over the S columns (A of dQ),
//   dQ += dS K  (fp32 in TMEM across all key tiles), then dQ = bf16(scale * dQ) once.
// Each output element is summed in one fixed order by one CTA, so the results are
// bitwise reproducible.
//
// Warp roles (both kernels, 12 warps): warp 0 TMA producer, warp 1 TMEM allocator and
// single MMA-issuing thread, warps 4-11 two compute warpgroups (warpgroup w owns 64 of the
// 128 columns of the score tile for all 128 TMEM lanes).
#include "fa_bwd_common.cuh"

namespace fa {

namespace {

constexpr int kThreads = 384;
constexpr int kTimeoutKV = -1200;
constexpr int kTimeoutQ = -1300;

// small shared region (both kernels)
constexpr uint32_t SM_BAR = 0;     // up to 32 mbarriers
constexpr uint32_t SM_TMEM = 256;  // TMEM base address slot
constexpr uint32_t SM_ABORT = 260;
constexpr uint32_t SM_TILE = 264;  // dK/dV kernel: its ticket; dQ kernel: 2-slot tile ring
constexpr uint32_t SM_LSE = 1024;  // dK/dV kernel: 2 stages x 128 fp32
constexpr uint32_t SM_DSUM = 2048; // dK/dV kernel: 2 stages x 128 fp32
constexpr uint32_t SMALL = 3072;

template <int DP>
struct GeoKV : Panels<DP> {
  using Panels<DP>::TILE_BYTES;
  static constexpr uint32_t OFF_K = SMALL;
  static constexpr uint32_t OFF_V = OFF_K + TILE_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;       // 2 stages
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * TILE_BYTES;  // 2 stages
  static constexpr uint32_t TOTAL = OFF_DO + 2 * TILE_BYTES;
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

template <int DP>
struct GeoQ : Panels<DP> {
  using Panels<DP>::TILE_BYTES;
  static constexpr int KST = 3;                               // K ring stages
  static constexpr uint32_t OFF_Q = SMALL;
  static constexpr uint32_t OFF_DO = OFF_Q + TILE_BYTES;
  static constexpr uint32_t OFF_K = OFF_DO + TILE_BYTES;      // KST stages
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE_BYTES; // 2 stages
  static constexpr uint32_t TOTAL = OFF_V + 2 * TILE_BYTES;
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

enum KvBar : int {
  KB_KV = 0, KB_QF0, KB_QF1, KB_QE0, KB_QE1, KB_DOF0, KB_DOF1, KB_DOE0, KB_DOE1,
  KB_SFULL, KB_DPFULL, KB_PFULL, KB_DSFULL, KB_ACC, KB_DRAIN, KB_COUNT
};
enum QBar : int {
  QB_QDO = 0, QB_KF0, QB_KF1, QB_KF2, QB_KE0, QB_KE1, QB_KE2, QB_VF0, QB_VF1, QB_VE0, QB_VE1,
  QB_SF0, QB_SF1, QB_DPFULL, QB_DPFREE, QB_DSFULL0, QB_DSFULL1, QB_ACC, QB_DRAIN,
  QB_QDOE, QB_TF0, QB_TF1, QB_TE0, QB_TE1, QB_COUNT
};

// tensor-memory columns
constexpr uint32_t KV_DK = 0, KV_DV = 128, KV_S = 256, KV_DP = 384;
constexpr uint32_t QT_S0 = 0, QT_S1 = 128, QT_DP = 256, QT_DQ = 384;

#ifdef FA_TRACE
// Optional per-phase timestamps (clock64 relative to the CTA's start) of the first CTAs of
// each split kernel, for pipeline tuning.  Off in the normal build.
constexpr int ST_CTAS = 4, ST_ITERS = 64, ST_EV = 12;
__device__ long long g_split_trace[2][ST_CTAS][ST_ITERS][ST_EV];
#define ST_TR(kern, ev, it)                                                       \
  do {                                                                            \
    if (blockIdx.x < ST_CTAS && (it) < ST_ITERS)                                  \
      g_split_trace[kern][blockIdx.x][(it)][(ev)] = clock64() - t_start;          \
  } while (0)
#define ST_START const long long t_start = clock64()
#else
#define ST_TR(kern, ev, it) \
  do {                      \
  } while (0)
#define ST_START
#endif

__device__ __forceinline__ MaskGeom geom_of(const BwdMainParams& p) {
  MaskGeom g;
  g.Sq = p.Sq;
  g.Sk = p.Sk;
  g.lo = p.lo64;
  g.hi = p.hi64;
  g.tm = kTileQ;
  g.tn = kTileK;
  g.Mb = p.Mb;
  g.Nb = p.Nb;
  return g;
}

// Common prologue: barrier init, TMEM allocation (512 columns), ticket (claimed here when
// `ticket` is not null).  Returns the TMEM base; *tile receives the ticket.
__device__ __forceinline__ uint32_t cta_setup(uint8_t* smem_raw, uint32_t sbase, int nbar,
                                              const uint32_t* counts, int* ticket, int* status,
                                              int* tile_out) {
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem_raw + SM_ABORT);
  volatile int* s_tile = reinterpret_cast<volatile int*>(smem_raw + SM_TILE);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    *s_abort = 0;
    if ((sbase & 1023u) != 0) {
      atomicExch(status, -1999);
      *s_abort = 1;
    }
    *s_tile = ticket ? atomicAdd(ticket, 1) : 0;
    for (int i = 0; i < nbar; ++i) mbar_init(sbase + SM_BAR + 8u * i, counts[i]);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + SM_TMEM, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  *tile_out = *s_tile;
  return *reinterpret_cast<uint32_t*>(smem_raw + SM_TMEM);
}

// bf16 stores of a 16-column chunk of a TMEM accumulator row (times sc), clipped to D.
__device__ __forceinline__ void store_row16(__nv_bfloat16* rowp, int c16, int D, const uint32_t (&r)[16],
                                            float sc, bool ok) {
  uint32_t pk[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    pk[e] = pack_bf16(__uint_as_float(r[2 * e]) * sc, __uint_as_float(r[2 * e + 1]) * sc);
  if (ok) {
    if (c16 * 16 < D)
      *reinterpret_cast<uint4*>(rowp + c16 * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    if (c16 * 16 + 8 < D)
      *reinterpret_cast<uint4*>(rowp + c16 * 16 + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
}

// dK/dV kernel, phase A for one thread (key row = TMEM lane, 64 query columns): P^T =
// exp2(S^T*scale*log2e - LSE2) (MASK: zero outside [cmin, cmax]) written back as bf16 pairs
// over the S^T columns already read; P (times 1 - tanh^2 under softcap) kept as f16 pairs.
// The mask is a template parameter so that unmasked tiles carry no per-element test.
template <bool MASK, bool SOFTCAP>
__device__ __forceinline__ void kv_phase_p(const SoftmaxConsts& kc, uint32_t taddr,
                                           const float* lse, int cmin, int cmax,
                                           uint32_t (&pc)[32]) {
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
        const int cc = c * 32 + v4 * 4 + u;
        float fac;
        float pr = prob<SOFTCAP>(kc, __uint_as_float(r[v4 * 4 + u]), lv[u], &fac);
        if (MASK) pr = (cc >= cmin && cc <= cmax) ? pr : 0.f;
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

// dQ kernel, one thread (query row = TMEM lane, 64 key columns): dS = P*(dP - D) with P
// recomputed from S (MASK: zero outside [cmin, cmax]), written as bf16 pairs over the S
// columns already read (the A operand of dQ += dS K).
template <bool MASK, bool SOFTCAP>
__device__ __forceinline__ void q_phase_ds(const SoftmaxConsts& kc, uint32_t sbuf, float lse2,
                                           float dsum, int cmin, int cmax,
                                           const uint32_t (&dp)[64]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    tmem_ld32(sbuf + c * 32, r);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float d2[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int cc = c * 32 + e + u;
        float fac;
        float pr = prob<SOFTCAP>(kc, __uint_as_float(r[e + u]), lse2, &fac);
        if (MASK) pr = (cc >= cmin && cc <= cmax) ? pr : 0.f;
        d2[u] = (SOFTCAP ? pr * fac : pr) * (__uint_as_float(dp[cc]) - dsum);
      }
      pk[e >> 1] = pack_bf16(d2[0], d2[1]);
    }
    tmem_st16(sbuf + c * 16, pk);
  }
}

}  // namespace

// ============================================================================ dK / dV

template <int DP, bool SOFTCAP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ BwdMainParams p,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t,
                    const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdo_t) {
  using G = GeoKV<DP>;
  ST_START;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem_raw + SM_ABORT);
  const float* s_lse = reinterpret_cast<const float*>(smem_raw + SM_LSE);
  const float* s_dsum = reinterpret_cast<const float*>(smem_raw + SM_DSUM);
  auto bar = [&](int i) -> uint32_t { return sbase + SM_BAR + 8u * i; };

  uint32_t counts[KB_COUNT];
  for (int i = 0; i < KB_COUNT; ++i) counts[i] = 1;
  counts[KB_PFULL] = 8;
  counts[KB_DSFULL] = 8;
  int tile;
  const uint32_t tmem = cta_setup(smem_raw, sbase, KB_COUNT, counts, p.ticket, p.status, &tile);
  // the dQ kernel reads nothing this kernel writes: let it start filling the SMs that this
  // kernel's last CTAs leave
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  AbortState st{s_abort, p.status, p.wait_limit};

  // key-tile-major order: under causal masking the low key tiles see the most query tiles
  const int per_n = p.B * p.Hk;
  const int n = tile / per_n;
  const int bk = tile - n * per_n;
  const int b = bk / p.Hk;
  const int hk = bk - b * p.Hk;
  const MaskGeom gm = geom_of(p);
  int64_t mb64, me64;
  m_range(gm, n, &mb64, &me64);
  const int m_begin = (int)mb64;
  const int m_count = (int)(me64 - mb64);
  const int total = (*s_abort) ? 0 : m_count * p.G;  // steps (g, m), m fastest
  const int n0 = n * kTileK;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      int issued_q[2] = {0, 0}, issued_do[2] = {0, 0};
      const bool kv = total > 0;
      if (kv) {
        mbar_arrive_expect_tx(bar(KB_KV), 2 * G::TILE_BYTES);
        for (int pn = 0; pn < G::NFULL; ++pn) {
          tma_load_4d(sbase + G::OFF_K + pn * G::FULL_BYTES, &tk, pn * 64, hk, n0, b, bar(KB_KV));
          tma_load_4d(sbase + G::OFF_V + pn * G::FULL_BYTES, &tv, pn * 64, hk, n0, b, bar(KB_KV));
        }
        if (G::TAIL) {
          tma_load_4d(sbase + G::OFF_K + G::TAIL_OFF, &tk_t, G::NFULL * 64, hk, n0, b, bar(KB_KV));
          tma_load_4d(sbase + G::OFF_V + G::TAIL_OFF, &tv_t, G::NFULL * 64, hk, n0, b, bar(KB_KV));
        }
      }
      for (int it = 0; it < total; ++it) {
        const int s = it & 1;
        const int g = it / m_count;
        const int m0 = (m_begin + (it - g * m_count)) * kTileQ;
        const int h = hk * p.G + g;
        if (it >= 2 && !mbar_wait(bar(KB_QE0 + s), ((it - 2) >> 1) & 1, st, kTimeoutKV - 1)) break;
        const uint32_t qdst = sbase + G::OFF_Q + s * G::TILE_BYTES;
        mbar_arrive_expect_tx(bar(KB_QF0 + s), G::TILE_BYTES + 2 * 512);
        for (int pn = 0; pn < G::NFULL; ++pn)
          tma_load_4d(qdst + pn * G::FULL_BYTES, &tq, pn * 64, h, m0, b, bar(KB_QF0 + s));
        if (G::TAIL) tma_load_4d(qdst + G::TAIL_OFF, &tq_t, G::NFULL * 64, h, m0, b, bar(KB_QF0 + s));
        const size_t row = ((size_t)b * p.H + h) * p.Sq_r + m0;
        bulk_load(sbase + SM_LSE + s * 512, p.lse2 + row, 512, bar(KB_QF0 + s));
        bulk_load(sbase + SM_DSUM + s * 512, p.dsum + row, 512, bar(KB_QF0 + s));
        issued_q[s] = it / 2 + 1;
        ST_TR(0, 8, it);
        if (it >= 2 && !mbar_wait(bar(KB_DOE0 + s), ((it - 2) >> 1) & 1, st, kTimeoutKV - 2)) break;
        const uint32_t ddst = sbase + G::OFF_DO + s * G::TILE_BYTES;
        mbar_arrive_expect_tx(bar(KB_DOF0 + s), G::TILE_BYTES);
        for (int pn = 0; pn < G::NFULL; ++pn)
          tma_load_4d(ddst + pn * G::FULL_BYTES, &tdo, pn * 64, h, m0, b, bar(KB_DOF0 + s));
        if (G::TAIL) tma_load_4d(ddst + G::TAIL_OFF, &tdo_t, G::NFULL * 64, h, m0, b, bar(KB_DOF0 + s));
        issued_do[s] = it / 2 + 1;
      }
      // every copy this thread started must land before the CTA may exit
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      if (kv) mbar_wait(bar(KB_KV), 0, dr, kTimeoutKV - 3);
      for (int s = 0; s < 2; ++s) {
        if (issued_q[s]) mbar_wait(bar(KB_QF0 + s), (issued_q[s] - 1) & 1, dr, kTimeoutKV - 3);
        if (issued_do[s]) mbar_wait(bar(KB_DOF0 + s), (issued_do[s] - 1) & 1, dr, kTimeoutKV - 3);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // prologue S_0, dP_0; then per step i:
    //   dV_i (needs P^T_i) ; dK_i (needs dS^T_i) ;
    //   S_i+1 (needs dV_i done: P^T_i aliases the S^T columns) ;
    //   dP_i+1 (needs dK_i done: dS^T_i aliases the dP^T columns)
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_N = idesc_bf16(128, G::NFULL * 64, false, true);
      constexpr uint32_t ID_N_T = idesc_bf16(128, G::TAIL ? G::TAIL : 16, false, true);
      const uint32_t sK = sbase + G::OFF_K, sV = sbase + G::OFF_V;
      uint32_t acc_v = 0, acc_k = 0;
      auto issue_S = [&](int it) -> bool {
        const int s = it & 1;
        if (!mbar_wait_spin(bar(KB_QF0 + s), (it >> 1) & 1, st, kTimeoutKV - 11)) return false;
        tc_fence_after();
        ST_TR(0, 0, it);
        const uint32_t sQ = sbase + G::OFF_Q + s * G::TILE_BYTES;
        for (int ks = 0; ks < G::KSTEPS; ++ks)
          mma_ss(tmem + KV_S, desc_kmajor<DP>(sK, ks), desc_kmajor<DP>(sQ, ks), ID_S, ks > 0);
        mma_commit(bar(KB_SFULL));
        return true;
      };
      auto issue_dP = [&](int it) -> bool {
        const int s = it & 1;
        if (!mbar_wait_spin(bar(KB_DOF0 + s), (it >> 1) & 1, st, kTimeoutKV - 13)) return false;
        tc_fence_after();
        ST_TR(0, 1, it);
        const uint32_t sDO = sbase + G::OFF_DO + s * G::TILE_BYTES;
        for (int ks = 0; ks < G::KSTEPS; ++ks)
          mma_ss(tmem + KV_DP, desc_kmajor<DP>(sV, ks), desc_kmajor<DP>(sDO, ks), ID_S, ks > 0);
        mma_commit(bar(KB_DPFULL));
        return true;
      };
      bool ok = total > 0 && mbar_wait_spin(bar(KB_KV), 0, st, kTimeoutKV - 10);
      const bool issued_any = ok;
      if (ok) ok = issue_S(0) && issue_dP(0);
      for (int it = 0; ok && it < total; ++it) {
        const int s = it & 1;
        const uint32_t sQ = sbase + G::OFF_Q + s * G::TILE_BYTES;
        const uint32_t sDO = sbase + G::OFF_DO + s * G::TILE_BYTES;
        // dV += P^T dO : A = P^T (bf16 pairs over the S^T columns), K = 128 queries
        if (!mbar_wait_spin(bar(KB_PFULL), it & 1, st, kTimeoutKV - 15)) break;
        tc_fence_after();
        ST_TR(0, 2, it);
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a_t = tmem + KV_S + (ks >> 2) * 64 + (ks & 3) * 8;
          const uint32_t en = (acc_v | (uint32_t)ks) ? 1u : 0u;
          mma_ts(tmem + KV_DV, a_t, desc_mn_full<DP>(sDO, ks), ID_N, en);
          if (G::TAIL) mma_ts(tmem + KV_DV + G::NFULL * 64, a_t, desc_mn_tail<DP>(sDO, ks), ID_N_T, en);
        }
        acc_v = 1;
        mma_commit(bar(KB_DOE0 + s));
        // dK += dS^T Q : A = dS^T (bf16 pairs over the dP^T columns), K = 128 queries
        if (!mbar_wait_spin(bar(KB_DSFULL), it & 1, st, kTimeoutKV - 16)) break;
        tc_fence_after();
        ST_TR(0, 3, it);
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a_t = tmem + KV_DP + (ks >> 2) * 64 + (ks & 3) * 8;
          const uint32_t en = (acc_k | (uint32_t)ks) ? 1u : 0u;
          mma_ts(tmem + KV_DK, a_t, desc_mn_full<DP>(sQ, ks), ID_N, en);
          if (G::TAIL) mma_ts(tmem + KV_DK + G::NFULL * 64, a_t, desc_mn_tail<DP>(sQ, ks), ID_N_T, en);
        }
        acc_k = 1;
        mma_commit(bar(KB_QE0 + s));
        if (it + 1 < total) {
          // S_i+1 overwrites P^T_i (read by dV_i) and dP_i+1 overwrites dS^T_i (read by
          // dK_i): both products were issued before by this thread, and tcgen05.mma
          // operations from one thread execute in issue order, so they queue right behind
          if (!issue_S(it + 1)) break;
          if (!issue_dP(it + 1)) break;
        }
      }
      mma_commit(bar(KB_ACC));
      if (issued_any) {
        mma_commit(bar(KB_DRAIN));
        volatile int no_abort = 0;
        AbortState dr{&no_abort, p.status, p.wait_limit};
        mbar_wait(bar(KB_DRAIN), 0, dr, kTimeoutKV - 17);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ compute
    const int wg = (warp - 4) >> 2;        // query half of the score tile
    const int qd = warp & 3;               // TMEM lane quadrant
    const int jl = qd * 32 + lane;         // key row inside the tile = TMEM lane
    const int col0 = wg * 64;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const int j = n0 + jl;
    const bool row_ok = j < p.Sk;
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};

    for (int it = 0; it < total; ++it) {
      const int s = it & 1;
      const int g = it / m_count;
      const int m = m_begin + (it - g * m_count);
      const int m0 = m * kTileQ;
      const bool need_mask = !tile_full(gm, m, n);
      // visible columns: lo <= (j - i) <= hi with i = m0 + col0 + c  <=>  c in [cmin, cmax]
      const int base = j - m0 - col0;
      const int cmin = row_ok ? max(base - p.hi, -1) : 1 << 20;
      const int cmax = row_ok ? min(base - p.lo, 1 << 20) : -1;
      const float* lse = s_lse + s * 128 + col0;
      const float* dsum = s_dsum + s * 128 + col0;

      if (!warp_wait(bar(KB_SFULL), it & 1, st, kTimeoutKV - 30)) break;
      tc_fence_after();
      if (threadIdx.x == 128) ST_TR(0, 4, it);
      uint32_t pc[32];  // P (times 1 - tanh^2 under softcap) as f16 pairs, reused for dS
      if (need_mask)
        kv_phase_p<true, SOFTCAP>(kc, t_lane + KV_S + col0, lse, cmin, cmax, pc);
      else
        kv_phase_p<false, SOFTCAP>(kc, t_lane + KV_S + col0, lse, cmin, cmax, pc);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_PFULL));
      if (threadIdx.x == 128) ST_TR(0, 5, it);

      if (!warp_wait(bar(KB_DPFULL), it & 1, st, kTimeoutKV - 31)) break;
      tc_fence_after();
      if (threadIdx.x == 128) ST_TR(0, 6, it);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(t_lane + KV_DP + col0 + c * 32, r);
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
        tmem_st16(t_lane + KV_DP + col0 + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_DSFULL));
      if (threadIdx.x == 128) ST_TR(0, 7, it);
    }

    // ------------------------------------------------------------------ dK / dV epilogue
    __nv_bfloat16* outp = wg == 0 ? p.dk : p.dv;
    const int64_t sb = wg == 0 ? p.dk_sb : p.dv_sb;
    const int64_t ss = wg == 0 ? p.dk_ss : p.dv_ss;
    const int64_t sh = wg == 0 ? p.dk_sh : p.dv_sh;
    const float sc = wg == 0 ? p.dk_scale : 1.f;
    const uint32_t tcol = wg == 0 ? KV_DK : KV_DV;
    __nv_bfloat16* rowp = outp + (int64_t)b * sb + (int64_t)j * ss + (int64_t)hk * sh;
    bool have = false;
    if (total > 0) have = warp_wait(bar(KB_ACC), 0, st, kTimeoutKV - 33);
    if (have) tc_fence_after();
    if (__all_sync(0xffffffffu, *s_abort == 0)) {
#pragma unroll
      for (int c = 0; c < DP / 16; ++c) {
        uint32_t r[16];
        if (have) {
          tmem_ld16(t_lane + tcol + c * 16, r);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0u;
        }
        store_row16(rowp, c, p.D, r, sc, row_ok);
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

// ============================================================================ dQ

// One query tile of the dQ kernel as every role decodes it from its ticket: query tiles
// with the most key tiles first (under causal masking: the last ones).
struct QTile {
  int m0, b, h, hk, n_begin, total;
};

__device__ __forceinline__ QTile q_tile_of(const BwdMainParams& p, const MaskGeom& gm, int tile) {
  QTile t;
  const int per_m = p.B * p.H;
  const int m = p.Mb - 1 - tile / per_m;
  const int bh = tile - (p.Mb - 1 - m) * per_m;
  t.b = bh / p.H;
  t.h = bh - t.b * p.H;
  t.hk = t.h / p.G;
  int64_t nb64, ne64;
  n_range(gm, m, &nb64, &ne64);
  t.n_begin = (int)nb64;
  t.total = (int)(ne64 - nb64);
  t.m0 = m * kTileQ;
  return t;
}

// Persistent: one CTA per SM claims query tiles from a ticket until none is left.  The TMA
// producer claims each tile when it reaches it and hands the ticket to the MMA thread and
// the compute warps through a two-slot ring (tile-full / tile-empty barriers).  Every
// per-step barrier phase, the K / V ring stages and the S buffers follow the CTA's global
// step count, so the next tile's Q / dO load starts as soon as the current tile's last
// S and dP products are complete, and its K / V loads run ahead across the boundary.
template <int DP, bool SOFTCAP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ BwdMainParams p,
                  const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t,
                  const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdo_t) {
  using G = GeoQ<DP>;
  ST_START;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem_raw + SM_ABORT);
  volatile int* s_tiles = reinterpret_cast<volatile int*>(smem_raw + SM_TILE);  // 2 slots
  auto bar = [&](int i) -> uint32_t { return sbase + SM_BAR + 8u * i; };

  uint32_t counts[QB_COUNT];
  for (int i = 0; i < QB_COUNT; ++i) counts[i] = 1;
  counts[QB_DPFREE] = 8;
  counts[QB_DSFULL0] = counts[QB_DSFULL1] = 8;
  counts[QB_TE0] = counts[QB_TE1] = 9;  // the MMA thread and the 8 compute warps
  int unused;
  const uint32_t tmem = cta_setup(smem_raw, sbase, QB_COUNT, counts, nullptr, p.status, &unused);
  AbortState st{s_abort, p.status, p.wait_limit};
  const int num_tiles = p.B * p.H * p.Mb;
  const MaskGeom gm = geom_of(p);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      int issued_k[G::KST] = {0, 0, 0}, issued_v[2] = {0, 0};
      int q_loads = 0;  // Q / dO loads issued (tiles with a visible key tile)
      int j = 0;        // steps (key tiles) loaded, over all tiles of the CTA
      bool ok = true;
      for (int T = 0; ok; ++T) {
        const int slot = T & 1;
        if (T >= 2 && !mbar_wait(bar(QB_TE0 + slot), ((T - 2) >> 1) & 1, st, kTimeoutQ - 4)) break;
        int tile = *s_abort ? -1 : atomicAdd(p.ticket_dq, 1);
        if (tile >= num_tiles) tile = -1;
        s_tiles[slot] = tile;
        mbar_arrive(bar(QB_TF0 + slot));  // release: the waiters see the slot
        if (tile < 0) break;
        const QTile q = q_tile_of(p, gm, tile);
        if (q.total == 0) continue;
        // Q / dO are free once the previous tile's last S and dP products are complete
        if (q_loads > 0 && !mbar_wait(bar(QB_QDOE), (q_loads - 1) & 1, st, kTimeoutQ - 5)) break;
        mbar_arrive_expect_tx(bar(QB_QDO), 2 * G::TILE_BYTES);
        for (int pn = 0; pn < G::NFULL; ++pn) {
          tma_load_4d(sbase + G::OFF_Q + pn * G::FULL_BYTES, &tq, pn * 64, q.h, q.m0, q.b, bar(QB_QDO));
          tma_load_4d(sbase + G::OFF_DO + pn * G::FULL_BYTES, &tdo, pn * 64, q.h, q.m0, q.b, bar(QB_QDO));
        }
        if (G::TAIL) {
          tma_load_4d(sbase + G::OFF_Q + G::TAIL_OFF, &tq_t, G::NFULL * 64, q.h, q.m0, q.b, bar(QB_QDO));
          tma_load_4d(sbase + G::OFF_DO + G::TAIL_OFF, &tdo_t, G::NFULL * 64, q.h, q.m0, q.b, bar(QB_QDO));
        }
        ++q_loads;
        for (int it = 0; it < q.total; ++it, ++j) {
          const int n0 = (q.n_begin + it) * kTileK;
          const int ks = j % G::KST;
          if (j >= G::KST &&
              !mbar_wait(bar(QB_KE0 + ks), ((j - G::KST) / G::KST) & 1, st, kTimeoutQ - 1)) {
            ok = false;
            break;
          }
          const uint32_t kdst = sbase + G::OFF_K + ks * G::TILE_BYTES;
          mbar_arrive_expect_tx(bar(QB_KF0 + ks), G::TILE_BYTES);
          for (int pn = 0; pn < G::NFULL; ++pn)
            tma_load_4d(kdst + pn * G::FULL_BYTES, &tk, pn * 64, q.hk, n0, q.b, bar(QB_KF0 + ks));
          if (G::TAIL) tma_load_4d(kdst + G::TAIL_OFF, &tk_t, G::NFULL * 64, q.hk, n0, q.b, bar(QB_KF0 + ks));
          issued_k[ks] = j / G::KST + 1;
          ST_TR(1, 8, j);
          const int vs = j & 1;
          if (j >= 2 && !mbar_wait(bar(QB_VE0 + vs), ((j - 2) >> 1) & 1, st, kTimeoutQ - 2)) {
            ok = false;
            break;
          }
          const uint32_t vdst = sbase + G::OFF_V + vs * G::TILE_BYTES;
          mbar_arrive_expect_tx(bar(QB_VF0 + vs), G::TILE_BYTES);
          for (int pn = 0; pn < G::NFULL; ++pn)
            tma_load_4d(vdst + pn * G::FULL_BYTES, &tv, pn * 64, q.hk, n0, q.b, bar(QB_VF0 + vs));
          if (G::TAIL) tma_load_4d(vdst + G::TAIL_OFF, &tv_t, G::NFULL * 64, q.hk, n0, q.b, bar(QB_VF0 + vs));
          issued_v[vs] = j / 2 + 1;
        }
      }
      // every copy this thread issued lands before the CTA ends
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      if (q_loads) mbar_wait(bar(QB_QDO), (q_loads - 1) & 1, dr, kTimeoutQ - 3);
      for (int s = 0; s < G::KST; ++s)
        if (issued_k[s]) mbar_wait(bar(QB_KF0 + s), (issued_k[s] - 1) & 1, dr, kTimeoutQ - 3);
      for (int s = 0; s < 2; ++s)
        if (issued_v[s]) mbar_wait(bar(QB_VF0 + s), (issued_v[s] - 1) & 1, dr, kTimeoutQ - 3);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // per tile: S_0, dP_0, S_1; then per key tile i:
    //   dP_i+1 (needs dP_i read: runs while dS_i is formed) ; dQ += dS_i K_i (needs dS_i) ;
    //   S_i+2 (dS_i aliases S_i's columns, which S_i+2 reuses: it queues right behind
    //   dQ_i, since tcgen05.mma operations from this one thread execute in issue order).
    // Across tiles the step index j runs on: the S buffers, the dP buffer and every
    // per-step barrier phase follow it.
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_N = idesc_bf16(128, G::NFULL * 64, false, true);
      constexpr uint32_t ID_N_T = idesc_bf16(128, G::TAIL ? G::TAIL : 16, false, true);
      const uint32_t sQ = sbase + G::OFF_Q, sDO = sbase + G::OFF_DO;
      // j: the CTA's global step index of the product being issued
      auto issue_S = [&](int j) -> bool {
        const int ks = j % G::KST;
        if (!mbar_wait_spin(bar(QB_KF0 + ks), (j / G::KST) & 1, st, kTimeoutQ - 11)) return false;
        tc_fence_after();
        ST_TR(1, 0, j);
        const uint32_t sK = sbase + G::OFF_K + ks * G::TILE_BYTES;
        const uint32_t dst = tmem + ((j & 1) ? QT_S1 : QT_S0);
        for (int k = 0; k < G::KSTEPS; ++k)
          mma_ss(dst, desc_kmajor<DP>(sQ, k), desc_kmajor<DP>(sK, k), ID_S, k > 0);
        mma_commit(bar(QB_SF0 + (j & 1)));
        return true;
      };
      auto issue_dP = [&](int j) -> bool {
        const int vs = j & 1;
        if (!mbar_wait_spin(bar(QB_VF0 + vs), (j >> 1) & 1, st, kTimeoutQ - 13)) return false;
        tc_fence_after();
        ST_TR(1, 1, j);
        const uint32_t sV = sbase + G::OFF_V + vs * G::TILE_BYTES;
        for (int k = 0; k < G::KSTEPS; ++k)
          mma_ss(tmem + QT_DP, desc_kmajor<DP>(sDO, k), desc_kmajor<DP>(sV, k), ID_S, k > 0);
        mma_commit(bar(QB_DPFULL));
        mma_commit(bar(QB_VE0 + vs));
        return true;
      };
      int j0 = 0, tq = 0;  // steps issued before this tile, tiles with work
      bool ok = true;
      for (int T = 0; ok; ++T) {
        const int slot = T & 1;
        if (!mbar_wait(bar(QB_TF0 + slot), (T >> 1) & 1, st, kTimeoutQ - 18)) break;
        const int tile = s_tiles[slot];
        mbar_arrive(bar(QB_TE0 + slot));
        if (tile < 0) break;
        const int total = q_tile_of(p, gm, tile).total;
        if (total == 0) continue;
        if (!mbar_wait_spin(bar(QB_QDO), tq & 1, st, kTimeoutQ - 10)) break;
        // S_0 / S_1 reuse the buffers of the previous tile's last two steps (issue order
        // puts them behind those steps' dQ products) and dP_0 the dP buffer (read once the
        // previous tile's last DPFREE phase completes).
        if (j0 > 0 && !mbar_wait_spin(bar(QB_DPFREE), (j0 - 1) & 1, st, kTimeoutQ - 14)) break;
        ok = issue_S(j0) && issue_dP(j0);
        if (ok && total == 1) mma_commit(bar(QB_QDOE));
        if (ok && total > 1) ok = issue_S(j0 + 1);
        for (int it = 0; ok && it < total; ++it) {
          const int j = j0 + it;
          if (it + 1 < total) {
            if (!mbar_wait_spin(bar(QB_DPFREE), j & 1, st, kTimeoutQ - 14)) { ok = false; break; }
            if (!issue_dP(j + 1)) { ok = false; break; }
            // the tile's last S and dP products are issued: Q / dO free once they complete
            if (it + 2 == total) mma_commit(bar(QB_QDOE));
          }
          // dQ += dS K : A = dS (bf16 pairs over S_j's columns), B = K_j MN-major, K = keys
          // (one dS barrier per step parity: a warp that has finished step j may finish step
          // j+1 (its S and dP are already issued) before a slower warp finishes step j, and
          // an arrival for j+1 must not complete the phase of j)
          if (!mbar_wait_spin(bar(QB_DSFULL0 + (j & 1)), (j >> 1) & 1, st, kTimeoutQ - 16)) {
            ok = false;
            break;
          }
          tc_fence_after();
          ST_TR(1, 2, j);
          const int ks = j % G::KST;
          const uint32_t sK = sbase + G::OFF_K + ks * G::TILE_BYTES;
          const uint32_t sbuf = tmem + ((j & 1) ? QT_S1 : QT_S0);
          for (int k = 0; k < 8; ++k) {
            const uint32_t a_t = sbuf + (k >> 2) * 64 + (k & 3) * 8;
            const uint32_t en = (it > 0 || k > 0) ? 1u : 0u;
            mma_ts(tmem + QT_DQ, a_t, desc_mn_full<DP>(sK, k), ID_N, en);
            if (G::TAIL) mma_ts(tmem + QT_DQ + G::NFULL * 64, a_t, desc_mn_tail<DP>(sK, k), ID_N_T, en);
          }
          mma_commit(bar(QB_KE0 + ks));
          // S_j+2 overwrites dS_j (read by dQ_j, issued just above): issue order suffices
          if (it + 2 < total && !issue_S(j + 2)) { ok = false; break; }
        }
        if (!ok) break;
        mma_commit(bar(QB_ACC));
        j0 += total;
        ++tq;
      }
      if (j0 > 0 || tq > 0 || !ok) {
        // every product issued is complete before tensor memory is released
        mma_commit(bar(QB_DRAIN));
        volatile int no_abort = 0;
        AbortState dr{&no_abort, p.status, p.wait_limit};
        mbar_wait(bar(QB_DRAIN), 0, dr, kTimeoutQ - 17);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ compute
    const int wg = (warp - 4) >> 2;        // key half of the score tile
    const int qd = warp & 3;               // TMEM lane quadrant
    const int ql = qd * 32 + lane;         // query row inside the tile = TMEM lane
    const int col0 = wg * 64;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};
    int j0 = 0, tq = 0;  // steps before this tile, tiles with work
    for (int T = 0;; ++T) {
      const int slot = T & 1;
      if (!warp_wait(bar(QB_TF0 + slot), (T >> 1) & 1, st, kTimeoutQ - 34)) break;
      const int tile = s_tiles[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QB_TE0 + slot));
      if (tile < 0) break;
      const QTile q = q_tile_of(p, gm, tile);
      const int i = q.m0 + ql;
      const bool row_ok = i < p.Sq;
      const size_t row = ((size_t)q.b * p.H + q.h) * p.Sq_r + (size_t)(q.m0 + ql);
      const float lse2 = p.lse2[row];  // +inf on padded rows, so P = 0 there
      const float dsum = p.dsum[row];
      bool ok = true;
      for (int it = 0; it < q.total; ++it) {
        const int j = j0 + it;
        const int n = q.n_begin + it;
        const int kb = n * kTileK + col0;  // key index of this thread's column 0
        const bool need_mask = !tile_full(gm, q.m0 / kTileQ, n);
        // visible columns: lo <= (key - i) <= hi and key < Sk  <=>  c in [cmin, cmax]
        const int cmin = max(i + p.lo - kb, -1);
        const int cmax = min(min(i + p.hi - kb, p.Sk - 1 - kb), 1 << 20);
        const uint32_t sbuf = t_lane + ((j & 1) ? QT_S1 : QT_S0) + col0;

        if (!warp_wait(bar(QB_SF0 + (j & 1)), (j >> 1) & 1, st, kTimeoutQ - 30)) { ok = false; break; }
        if (!warp_wait(bar(QB_DPFULL), j & 1, st, kTimeoutQ - 31)) { ok = false; break; }
        tc_fence_after();
        if (threadIdx.x == 128) ST_TR(1, 4, j);
        uint32_t dp[64];
        {
          uint32_t r[32];
          tmem_ld32(t_lane + QT_DP + col0, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) dp[e] = r[e];
          tmem_ld32(t_lane + QT_DP + col0 + 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) dp[32 + e] = r[e];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_DPFREE));
        if (threadIdx.x == 128) ST_TR(1, 5, j);
        if (need_mask)
          q_phase_ds<true, SOFTCAP>(kc, sbuf, lse2, dsum, cmin, cmax, dp);
        else
          q_phase_ds<false, SOFTCAP>(kc, sbuf, lse2, dsum, cmin, cmax, dp);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_DSFULL0 + (j & 1)));
        if (threadIdx.x == 128) ST_TR(1, 7, j);
      }

      // -------------------------------------------------------------- dQ epilogue
      // (the accumulator columns are read before this warp's next dS arrival, which the
      // next tile's first dQ product waits for)
      __nv_bfloat16* rowp =
          p.dq + (int64_t)q.b * p.dq_sb + (int64_t)i * p.dq_ss + (int64_t)q.h * p.dq_sh;
      bool have = false;
      if (ok && q.total > 0) have = warp_wait(bar(QB_ACC), tq & 1, st, kTimeoutQ - 33);
      if (have) tc_fence_after();
      if (__all_sync(0xffffffffu, ok && *s_abort == 0)) {
#pragma unroll
        for (int c = wg; c < DP / 16; c += 2) {
          uint32_t r[16];
          if (have) {
            tmem_ld16(t_lane + QT_DQ + c * 16, r);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = 0u;
          }
          store_row16(rowp, c, p.D, r, p.dk_scale, row_ok);
        }
      } else {
        break;
      }
      if (q.total > 0) {
        j0 += q.total;
        ++tq;
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

// ============================================================================ launch

namespace {

template <typename Kern>
cudaError_t launch_kernel(Kern kern, size_t smem, const BwdMainParams& p, const OperandMaps& q,
                          const OperandMaps& k, const OperandMaps& v, const OperandMaps& d,
                          int num_ctas, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_ctas, kThreads, smem, s>>>(p, q.full, q.tail, k.full, k.tail, v.full, v.tail, d.full,
                                        d.tail);
  return cudaGetLastError();
}

// The dQ kernel as a programmatic dependent of the dK / dV kernel before it on the stream:
// it may start once every dK / dV CTA has started (they signal it at once), and needs no
// result of theirs.
template <typename Kern>
cudaError_t launch_dependent(Kern kern, size_t smem, const BwdMainParams& p, const OperandMaps& q,
                             const OperandMaps& k, const OperandMaps& v, const OperandMaps& d,
                             int num_ctas, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p, q.full, q.tail, k.full, k.tail, v.full, v.tail, d.full, d.tail);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_split(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                             const OperandMaps& v, const OperandMaps& d, int Dp, bool softcap,
                             int num_kv_ctas, int num_q_ctas, cudaStream_t s) {
  // the dQ kernel is persistent: one CTA per SM at most, each claiming query tiles
  int q_ctas = num_q_ctas;
  if (num_q_ctas > 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (q_ctas > sms) q_ctas = sms;
  }
#define FA_SPLIT_CASE(DPV)                                                                     \
  case DPV: {                                                                                  \
    cudaError_t e = cudaSuccess;                                                               \
    if (num_kv_ctas > 0)                                                                       \
      e = softcap ? launch_kernel(bwd_dkdv_kernel<DPV, true>, GeoKV<DPV>::TOTAL, p, q, k, v, d, \
                                  num_kv_ctas, s)                                              \
                  : launch_kernel(bwd_dkdv_kernel<DPV, false>, GeoKV<DPV>::TOTAL, p, q, k, v, d, \
                                  num_kv_ctas, s);                                             \
    if (e != cudaSuccess) return e;                                                            \
    if (num_q_ctas > 0)                                                                        \
      e = softcap ? launch_dependent(bwd_dq_kernel<DPV, true>, GeoQ<DPV>::TOTAL, p, q, k, v, d, \
                                     q_ctas, s)                                                \
                  : launch_dependent(bwd_dq_kernel<DPV, false>, GeoQ<DPV>::TOTAL, p, q, k, v,  \
                                     d, q_ctas, s);                                            \
    return e;                                                                                  \
  }
  switch (Dp) {
    FA_SPLIT_CASE(64)
    FA_SPLIT_CASE(80)
    FA_SPLIT_CASE(96)
    FA_SPLIT_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef FA_SPLIT_CASE
}

#ifdef FA_TRACE
cudaError_t split_trace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_split_trace)) bytes = sizeof(g_split_trace);
  return cudaMemcpyFromSymbol(host, g_split_trace, bytes);
}
#endif

}  // namespace fa
