// fa_fwd_tc.cu — the forward (O and the natural-log LSE) on tcgen05 / TMEM / TMA for sm_103a.
//
// It computes what the Triton page's `_attn_fwd_inner` computes — per key block, scores,
// running row maximum, rescaled running sum and accumulator, and at the end O = acc / l,
// LSE = (m + log2 l) * ln 2 — with the same mask (bottom-right aligned band lo <= j - i
// <= hi, j < Sk) and softcap (z = c * tanh(scale * s / c)) as the backward.
//
// One CTA owns one 128-query tile of one (batch, q-head) and walks the key tiles with a
// visible entry (GQA/MQA page: the kv-head is h / (H / Hk)):
//   S = Q K^T        (M = 128 queries, N = 128 keys, K = Dp; both operands K-major)
//   P = exp2(z * log2e - m)  written as 16-bit pairs over the S columns already read
//   O (+)= P V       (A = P from tensor memory, B = V read MN-major, N = Dp)
// Two softmax warpgroups split the 128 key columns of the score tile: thread (warpgroup
// w, TMEM lane r) owns query row r and columns [64w, 64w + 64).  The two halves of a
// row's maximum meet through shared memory once per key tile; each warpgroup keeps the
// row sum of its own columns and the two are added at the end.
//
// The running maximum m is only moved (and O, l rescaled by exp2(m_old - m_new)) when
// a new score exceeds it by more than 8 in log2 units; otherwise the stale m is kept and
// P may reach 2^8, well inside bf16 / f16 and the fp32 sums.  O = acc / l and the LSE use
// the same m, so the result is exact up to rounding either way.  After the first key
// tiles a rescale is rare.
//
// Warp roles (12 warps): warp 0 TMA producer of Q (once) and of the 3-stage K ring;
// warp 2 TMA producer of the 2-stage V ring; warp 1 TMEM allocator and single
// MMA-issuing thread; warps 4-11 two softmax / epilogue warpgroups (warp w reads TMEM
// lanes 32 (w % 4) .. +31).  Warp 3 only joins the CTA barriers.
//
// Tensor memory: S double buffer [0, 128) and [128, 256) (P written over its first 32
// columns of each 64-column half), O accumulator [256, 256 + Dp).
#include "fa_bwd_common.cuh"

#include <math.h>

namespace fa {

namespace {

constexpr int kFwdThreads = 384;
constexpr int kFwdTimeout = -1400;

constexpr uint32_t FSM_BAR = 0;     // mbarriers
constexpr uint32_t FSM_TMEM = 256;  // TMEM base address slot
constexpr uint32_t FSM_ABORT = 260;
constexpr uint32_t FSM_MAX = 1024;  // [2 parities][2 warpgroups][128 rows] fp32 row maxima
constexpr uint32_t FSM_L = 3072;    // [2 warpgroups][128 rows] fp32 row sums (epilogue)
constexpr uint32_t FSMALL = 4096;

template <int DP>
struct GeoF : Panels<DP> {
  using Panels<DP>::TILE_BYTES;
  static constexpr int KST = 3;  // K ring stages
  static constexpr int VST = 2;  // V ring stages
  static constexpr uint32_t OFF_Q = FSMALL;
  static constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE_BYTES;
  static constexpr uint32_t TOTAL = OFF_V + VST * TILE_BYTES;
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

enum FBar : int {
  F_Q = 0, F_KF0, F_KF1, F_KF2, F_KE0, F_KE1, F_KE2, F_VF0, F_VF1, F_VE0, F_VE1,
  F_SF0, F_SF1, F_PF0, F_PF1, F_OD, F_ACC, F_DRAIN, F_COUNT
};
static_assert(F_COUNT <= 32, "barrier area holds 32 mbarriers");

constexpr uint32_t FT_S0 = 0, FT_S1 = 128, FT_O = 256;

constexpr float kNegInf = -__builtin_huge_valf();

// Scores of this thread's 64 columns of its row in log2 units (scale * s * log2e, or
// with softcap c * log2e * tanh(scale * s / c)); `sbuf` addresses column col0 of the
// row; masked columns (MASK: visible iff cmin <= column <= cmax, columns of the whole
// tile) are -inf.  Returns the maximum over the 64.
template <bool MASK, bool SOFTCAP>
__device__ __forceinline__ float fwd_scores(const SoftmaxConsts& kc, uint32_t sbuf, int col0,
                                            int cmin, int cmax, float (&x)[64]) {
  float mx = kNegInf;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    tmem_ld32(sbuf + c * 32, r);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int col = col0 + c * 32 + e;
      const float s = __uint_as_float(r[e]);
      float v = SOFTCAP ? kc.cap_log2 * tanh_exp2(s * kc.cap_scale) : s * kc.scale_log2;
      if (MASK) v = (col >= cmin && col <= cmax) ? v : kNegInf;
      x[c * 32 + e] = v;
      mx = fmaxf(mx, v);
    }
  }
  return mx;
}

// P = exp2(x - m) for the thread's 64 columns as 16-bit pairs over the first 32 of them
// (`sbuf` = column col0): columns [0, 64) of the row land in TMEM columns [0, 32),
// columns [64, 128) in [64, 96), the A layout the P V product reads.  Returns the sum of
// the 64 P values (fp32, before rounding).
template <bool F16>
__device__ __forceinline__ float fwd_probs(uint32_t sbuf, float m, const float (&x)[64]) {
  float sum = 0.f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float p0 = ex2_approx(x[q * 32 + 2 * e] - m);
      const float p1 = ex2_approx(x[q * 32 + 2 * e + 1] - m);
      sum += p0 + p1;
      pk[e] = pack_h2<F16>(p0, p1);
    }
    tmem_st16(sbuf + q * 16, pk);
  }
  return sum;
}

}  // namespace

template <int DP, bool SOFTCAP, bool F16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tc_kernel(const __grid_constant__ FwdTcParams p,
                  const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t) {
  using G = GeoF<DP>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem_raw + FSM_ABORT);
  auto bar = [&](int i) -> uint32_t { return sbase + FSM_BAR + 8u * i; };

  if (threadIdx.x == 0) {
    *s_abort = 0;
    if ((sbase & 1023u) != 0) {
      // the tile layout assumes a 1024-byte aligned dynamic shared-memory base
      if (p.status) atomicExch(p.status, kFwdTimeout - 99);
      *s_abort = 1;
    }
    for (int i = 0; i < F_COUNT; ++i) mbar_init(bar(i), (i == F_PF0 || i == F_PF1) ? 8 : 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + FSM_TMEM, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<uint32_t*>(smem_raw + FSM_TMEM);
  AbortState st{s_abort, p.status, p.wait_limit};

  // query tiles with the most key tiles first (under causal masking: the last ones)
  const int per_m = p.B * p.H;
  const int m = p.Mb - 1 - (int)(blockIdx.x / (unsigned)per_m);
  const int bh = (int)blockIdx.x - (p.Mb - 1 - m) * per_m;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int hk = h / p.G;
  MaskGeom gm;
  int q_off = 0, k_off = 0, tb = b, lo = p.lo, hi = p.hi;  // tb: batch coordinate of the maps
  if (p.varlen) {
    // sequence b: rows [cu[b], cu[b+1]) clamped into the packed tensors, so that malformed
    // offsets cannot move a load or a store outside them
    const int q0 = min(max(p.cu_q[b], 0), p.total_q), q1 = min(max(p.cu_q[b + 1], q0), p.total_q);
    const int k0 = min(max(p.cu_k[b], 0), p.total_k), k1 = min(max(p.cu_k[b + 1], k0), p.total_k);
    q_off = q0;
    k_off = k0;
    tb = 0;
    gm = make_geom(q1 - q0, k1 - k0, p.causal, p.window_left, p.window_right, kTileQ, kTileK);
    lo = (int)max64(min64(gm.lo, 1ll << 30), -(1ll << 30));
    hi = (int)max64(min64(gm.hi, 1ll << 30), -(1ll << 30));
  } else {
    gm.Sq = p.Sq;
    gm.Sk = p.Sk;
    gm.lo = p.lo64;
    gm.hi = p.hi64;
    gm.tm = kTileQ;
    gm.tn = kTileK;
    gm.Mb = p.Mb;
    gm.Nb = p.Nb;
  }
  const int Sq = (int)gm.Sq, Sk = (int)gm.Sk;
  int64_t nb64 = 0, ne64 = 0;
  if (m < gm.Mb) n_range(gm, m, &nb64, &ne64);  // a shorter sequence may have no tile m
  const int n_begin = (int)nb64;
  // Block sparsity: the key tiles of [n_begin, n_end) whose block-mask byte is set, in
  // ascending order.  Every warp counts them (lanes striding the row) and every role walks
  // them with its own cursor, so all roles agree on the sequence without exchanging it.
  const uint8_t* brow = p.block_mask
                            ? p.block_mask + (((size_t)b * p.H + h) * p.Mb + m) * (size_t)p.Nb
                            : nullptr;
  int nvis = (int)(ne64 - nb64);
  if (brow) {
    int c = 0;
    for (int n = (int)nb64 + lane; n < (int)ne64; n += 32) c += brow[n] != 0;
    nvis = __reduce_add_sync(0xffffffffu, c);
  }
  auto next_tile = [&](int nc) -> int {  // the visible key tile after nc
    ++nc;
    if (brow)
      while (brow[nc] == 0) ++nc;
    return nc;
  };
  const int total = (*s_abort) ? 0 : nvis;
  const int m0 = m * kTileQ;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ TMA producers
    // Warp 0 loads Q and the K ring, warp 2 the V ring: each refills a stage as soon as
    // its own last reader is done (K: the stage's S product, V: its P V product), so a K
    // load never waits behind a V stage that is still being read.
    if (lane == 0) {
      const bool kside = warp == 0;
      const CUtensorMap* tm = kside ? &tk : &tv;
      const CUtensorMap* tm_t = kside ? &tk_t : &tv_t;
      const int nst = kside ? G::KST : G::VST;
      const uint32_t base = sbase + (kside ? G::OFF_K : G::OFF_V);
      const int full0 = kside ? F_KF0 : F_VF0, empty0 = kside ? F_KE0 : F_VE0;
      tma_prefetch_desc(tm);
      int issued[G::KST] = {};
      if (kside && total > 0) {
        tma_prefetch_desc(&tq);
        mbar_arrive_expect_tx(bar(F_Q), G::TILE_BYTES);
        for (int pn = 0; pn < G::NFULL; ++pn)
          tma_load_4d(sbase + G::OFF_Q + pn * G::FULL_BYTES, &tq, pn * 64, h, q_off + m0, tb, bar(F_Q));
        if (G::TAIL) tma_load_4d(sbase + G::OFF_Q + G::TAIL_OFF, &tq_t, G::NFULL * 64, h, q_off + m0, tb, bar(F_Q));
      }
      int ncur = n_begin - 1;
      for (int it = 0; it < total; ++it) {
        ncur = next_tile(ncur);
        const int n0 = k_off + ncur * kTileK;
        const int ks = it % nst;
        if (it >= nst && !mbar_wait(bar(empty0 + ks), ((it - nst) / nst) & 1, st, kFwdTimeout - 1))
          break;
        const uint32_t dst = base + ks * G::TILE_BYTES;
        mbar_arrive_expect_tx(bar(full0 + ks), G::TILE_BYTES);
        for (int pn = 0; pn < G::NFULL; ++pn)
          tma_load_4d(dst + pn * G::FULL_BYTES, tm, pn * 64, hk, n0, tb, bar(full0 + ks));
        if (G::TAIL) tma_load_4d(dst + G::TAIL_OFF, tm_t, G::NFULL * 64, hk, n0, tb, bar(full0 + ks));
        issued[ks] = it / nst + 1;
      }
      // every copy this thread started must land before the CTA may exit
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      if (kside && total > 0) mbar_wait(bar(F_Q), 0, dr, kFwdTimeout - 3);
      for (int s2 = 0; s2 < nst; ++s2)
        if (issued[s2]) mbar_wait(bar(full0 + s2), (issued[s2] - 1) & 1, dr, kFwdTimeout - 3);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // S_0, S_1; then per key tile j: O (+)= P_j V_j once P_j is written (and O rescaled),
    // then S_j+2 once that product is done (P_j lives in S_j's columns, which S_j+2 reuses).
    if (lane == 0) {
      const TileDescs dQ_ = tile_descs<DP>(sbase + G::OFF_Q);
      auto issue_S = [&](int it) -> bool {
        const int ks = it % G::KST;
        if (!mbar_wait_spin(bar(F_KF0 + ks), (it / G::KST) & 1, st, kFwdTimeout - 11)) return false;
        tc_fence_after();
        const TileDescs dK_ = tile_descs<DP>(sbase + G::OFF_K + ks * G::TILE_BYTES);
        mma_kmajor<DP, F16>(tmem + ((it & 1) ? FT_S1 : FT_S0), dQ_, dK_);
        mma_commit(bar(F_SF0 + (it & 1)));
        mma_commit(bar(F_KE0 + ks));
        return true;
      };
      bool ok = total > 0 && mbar_wait_spin(bar(F_Q), 0, st, kFwdTimeout - 10);
      const bool issued_any = ok;
      if (ok) ok = issue_S(0);
      if (ok && total > 1) ok = issue_S(1);
      for (int it = 0; ok && it < total; ++it) {
        const int sb = it & 1;
        if (!mbar_wait_spin(bar(F_PF0 + sb), (it >> 1) & 1, st, kFwdTimeout - 12)) break;
        const int vs = it % G::VST;
        if (!mbar_wait_spin(bar(F_VF0 + vs), (it / G::VST) & 1, st, kFwdTimeout - 13)) break;
        tc_fence_after();
        const TileDescs dV_ = tile_descs<DP>(sbase + G::OFF_V + vs * G::TILE_BYTES);
        mma_dv<DP, F16>(tmem + FT_O, tmem + (sb ? FT_S1 : FT_S0), dV_, it > 0 ? 1u : 0u);
        mma_commit(bar(F_VE0 + vs));
        mma_commit(bar(F_OD));
        if (it + 2 < total) {
          if (!mbar_wait_spin(bar(F_OD), it & 1, st, kFwdTimeout - 14)) break;
          if (!issue_S(it + 2)) break;
        }
      }
      if (issued_any) {
        mma_commit(bar(F_ACC));
        mma_commit(bar(F_DRAIN));
        volatile int no_abort = 0;
        AbortState dr{&no_abort, p.status, p.wait_limit};
        mbar_wait(bar(F_DRAIN), 0, dr, kFwdTimeout - 15);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - 4) >> 2;        // key half of the score tile (columns 64 wg ..)
    const int qd = warp & 3;               // TMEM lane quadrant
    const int r = qd * 32 + lane;          // query row inside the tile = TMEM lane
    const int col0 = wg * 64;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const int i = m0 + r;
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};
    float* s_max = reinterpret_cast<float*>(smem_raw + FSM_MAX);
    float* s_l = reinterpret_cast<float*>(smem_raw + FSM_L);
    // O columns this warpgroup rescales and stores: 16-column chunks [c_lo, c_hi)
    constexpr int NCH = DP / 16;
    constexpr int NCH0 = (NCH + 1) / 2;
    const int c_lo = wg ? NCH0 : 0, c_hi = wg ? NCH : NCH0;
    float mrow = kNegInf;  // running maximum (log2 units); moved only by more than 8
    float lrow = 0.f;      // running sum of this warpgroup's P relative to mrow
    int ncur = n_begin - 1;
    for (int it = 0; it < total; ++it) {
      const int n = ncur = next_tile(ncur);
      const int kb = n * kTileK;  // key index of column 0
      const bool need_mask = !tile_full(gm, m, n);
      // visible columns: lo <= key - i <= hi and key < Sk  <=>  c in [cmin, cmax]
      const int cmin = max(i + lo - kb, -1);
      const int cmax = min(min(i + hi - kb, Sk - 1 - kb), 1 << 20);
      const uint32_t sbuf = t_lane + ((it & 1) ? FT_S1 : FT_S0) + col0;
      const bool ok = warp_wait(bar(F_SF0 + (it & 1)), (it >> 1) & 1, st, kFwdTimeout - 30);
      float x[64];
      float mx = kNegInf;
      if (ok) {
        tc_fence_after();
        mx = need_mask ? fwd_scores<true, SOFTCAP>(kc, sbuf, col0, cmin, cmax, x)
                       : fwd_scores<false, SOFTCAP>(kc, sbuf, col0, cmin, cmax, x);
      }
      // the row maximum over both halves; both warpgroups always reach this barrier, and
      // after it both see the abort flag that a failed wait of either one has raised
      s_max[((it & 1) * 2 + wg) * 128 + r] = mx;
      named_bar_sync(1, 256);
      if (*s_abort) break;
      mx = fmaxf(mx, s_max[((it & 1) * 2 + (wg ^ 1)) * 128 + r]);
      // move the reference maximum only when a score passes it by more than 8 (log2);
      // both warpgroups take the same decision for a row
      float alpha = 1.f;
      if (it == 0) {
        mrow = mx;
      } else if (mx > mrow + 8.f) {
        alpha = ex2_approx(mrow - mx);  // mrow finite here, or -inf: alpha = 0
        mrow = mx;
      }
      const float muse = mrow == kNegInf ? 0.f : mrow;  // all-masked so far: P = 0
      lrow = lrow * alpha + fwd_probs<F16>(sbuf, muse, x);
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds the products up to key tile it-1: wait for the last one, then rescale
        // this warpgroup's columns of it (on a failed wait the next barrier ends the loop)
        if (!warp_wait(bar(F_OD), (it - 1) & 1, st, kFwdTimeout - 31)) continue;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < NCH0; ++c) {
          if (c_lo + c < c_hi) {
            uint32_t o[16];
            tmem_ld16(t_lane + FT_O + (c_lo + c) * 16, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(t_lane + FT_O + (c_lo + c) * 16, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(F_PF0 + (it & 1)));
    }

    // O = acc / l and LSE = (m + log2 l) * ln 2 with l the sum of both halves; a row with
    // no visible key gives O = 0 and LSE = +inf
    bool have = false;
    if (!*s_abort && total > 0) have = warp_wait(bar(F_ACC), 0, st, kFwdTimeout - 32);
    s_l[wg * 128 + r] = lrow;
    named_bar_sync(1, 256);
    const float lsum = lrow + s_l[(wg ^ 1) * 128 + r];
    if (have) tc_fence_after();
    if (__all_sync(0xffffffffu, *s_abort == 0)) {
      const bool row_ok = i < Sq;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + (int64_t)tb * p.o_sb +
                       (int64_t)(q_off + i) * p.o_ss + (int64_t)h * p.o_sh;
#pragma unroll
      for (int cc = 0; cc < NCH0; ++cc) {
        const int c = c_lo + cc;
        if (c < c_hi) {
          uint32_t o[16];
          if (have) {
            tmem_ld16(t_lane + FT_O + c * 16, o);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = 0u;
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pk[e] = pack_h2<F16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          if (row_ok) {
            if (c * 16 < p.D)
              *reinterpret_cast<uint4*>(orow + c * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (c * 16 + 8 < p.D)
              *reinterpret_cast<uint4*>(orow + c * 16 + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      if (row_ok && wg == 0) {
        const float lse = lsum > 0.f ? (mrow + log2f(lsum)) * 0.69314718055994531f
                                     : __int_as_float(0x7f800000);
        p.lse[(int64_t)tb * p.lse_sb + (int64_t)h * p.lse_sh + (int64_t)(q_off + i) * p.lse_ss] = lse;
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

namespace {

// Sk == 0: no row has a visible key, so O = 0 and LSE = +inf everywhere (the rows-without-
// keys convention of the main kernel's epilogue).  One thread per (b, i, h) row.
__global__ void __launch_bounds__(256) fwd_empty_kernel(const FwdTcParams p) {
  const int64_t rows = (int64_t)p.B * p.Sq * p.H;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = r / ((int64_t)p.Sq * p.H);
    const int64_t rem = r - b * p.Sq * p.H;
    const int64_t i = rem / p.H, h = rem - (rem / p.H) * p.H;
    uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + b * p.o_sb + i * p.o_ss + h * p.o_sh;
    for (int c = 0; c < p.D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0u, 0u, 0u, 0u);
    p.lse[b * p.lse_sb + h * p.lse_sh + i * p.lse_ss] = __int_as_float(0x7f800000);
  }
}

template <int DP, bool SC, bool F16>
cudaError_t launch_fwd_one(const FwdTcParams& p, const OperandMaps& q, const OperandMaps& k,
                           const OperandMaps& v, cudaStream_t s) {
  auto kern = fwd_tc_kernel<DP, SC, F16>;
  // at least 116 KB, so that one CTA (which allocates all 512 TMEM columns) runs per SM
  const size_t smem = GeoF<DP>::TOTAL > 118784u ? GeoF<DP>::TOTAL : 118784u;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t ctas = (int64_t)p.Mb * p.B * p.H;
  if (ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kFwdThreads, smem, s>>>(p, q.full, q.tail, k.full, k.tail, v.full, v.tail);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_empty(const FwdTcParams& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.Sq * p.H;
  if (rows <= 0) return cudaSuccess;
  int64_t blocks = (rows + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  fwd_empty_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const FwdTcParams& p, const OperandMaps& q, const OperandMaps& k,
                          const OperandMaps& v, int Dp, bool softcap, bool f16, cudaStream_t s) {
  if (p.Mb <= 0 || p.B <= 0 || p.H <= 0) return cudaSuccess;
#define FA_FWD_TC_CASE(DPV)                                                             \
  case DPV:                                                                             \
    if (f16)                                                                            \
      return softcap ? launch_fwd_one<DPV, true, true>(p, q, k, v, s)                   \
                     : launch_fwd_one<DPV, false, true>(p, q, k, v, s);                 \
    return softcap ? launch_fwd_one<DPV, true, false>(p, q, k, v, s)                    \
                   : launch_fwd_one<DPV, false, false>(p, q, k, v, s);
  switch (Dp) {
    FA_FWD_TC_CASE(64)
    FA_FWD_TC_CASE(80)
    FA_FWD_TC_CASE(96)
    FA_FWD_TC_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef FA_FWD_TC_CASE
}

}  // namespace fa
