// fa_wide.cu — forward and backward for head dims above 128 and for a V head dim that
// differs from the Q / K one (the call-trace page's `run_mha_bwd_constexpr` dispatches
// head dims up to 256; the `flash_bwd_sm90.py` page's kernel takes `head_dim` and
// `head_dim_v` separately), on tcgen05 / TMEM / TMA for sm_103a.
//
// The arithmetic is the one of the 128-wide kernels (fa_fwd_tc.cu, fa_bwd_main.cu); what
// changes is the tiling, because at a head dim of 256 the dK and dV accumulators of a
// 128-key tile alone fill tensor memory and four 256-column operand tiles exceed shared
// memory.  Both padded head dims (DPK for q / k, DPV for v) are multiples of 64, at most
// 256, held as 64-column 128B-swizzled panels.
//
// Forward (one CTA per 128-query tile of one (batch, q-head)):
//   S = Q K^T          M = 128 queries, N = 128 keys, K = DPK      -> TMEM, two buffers
//   P = exp2(z * log2e - m), written as 16-bit pairs over the S columns
//   O (+)= P V         A = P from TMEM, B = V read MN-major, N = DPV (<= 256)
// with the online softmax of the Triton page's `_attn_fwd_inner` (the running maximum is
// moved only when a score passes it by more than 8 in log2 units, as in fa_fwd_tc.cu).
// Tensor memory: S buffers [0, 128) and [128, 256), O [256, 256 + DPV).
//
// Backward (one CTA per (128-key tile, batch, kv-head, output slice); in the deterministic
// mode the CTAs claim the tiles from a ticket counter, highest key tile first, and add the
// dQ partials of a block from the highest key tile down): slice s owns the
// dK / dQ columns [128 s, 128 s + 128) of DPK and the dV columns [128 s, 128 s + 128) of
// DPV; every slice recomputes the scores over the full head dims.  Per (q-head of the
// group, 64-query block):
//   S^T  = K Q^T       M = 128 keys, N = 64 queries, K = DPK
//   dP^T = V dO^T      M = 128 keys, N = 64 queries, K = DPV
//   P^T, dS^T = P^T (dP^T - D) (x (1 - tanh^2)) as 16-bit pairs over the S^T / dP^T
//                      columns, dS^T also into shared memory
//   dV_s += P^T dO_s   A = P^T from TMEM, K = 64 queries
//   dK_s += dS^T Q_s   A = dS^T from TMEM
//   dQ_s^T = K_s^T dS^T  M = 128 head-dim rows, N = 64 queries, K = 128 keys: the dQ
//                      partial is formed transposed, so no M = 64 product is needed
// and the dQ partial is added into an fp32 accumulator with bulk reductions.  Tensor
// memory: dK_s [0, 128), dV_s [128, 256), S^T [256, 320), dP^T [320, 384), dQ^T
// [384, 448).  Shared memory at DPK = DPV = 256: K 64 KB, V 64 KB, Q 32 KB, dO 32 KB,
// dS^T 16 KB and a 16 KB staging buffer, 227 KB in all, so Q and dO have one buffer each
// there; where two fit (smaller head dims), Q and dO are double-buffered and the MMAs of
// consecutive steps overlap.
//
// dQ accumulator layout: per (b, h, 64-query block, slice) one block of 128 head-dim rows
// x 64 queries fp32 (32 KB); in row d, the 16-byte chunk of queries 4c..4c+3 sits at
// chunk position c ^ (d & 15), so that the drain's stores of whole rows do not collide
// in shared memory banks.  The convert kernel reads the same layout.
#include "fa_bwd_common.cuh"

#include <math.h>

namespace fa {

namespace {

constexpr int kWideTimeout = -1500;
constexpr uint32_t W_PANEL128 = 128u * 128u;  // 64-column panel of 128 rows (16 KB)
constexpr uint32_t W_PANEL64 = 64u * 128u;    // 64-column panel of 64 rows (8 KB)
constexpr float kNegInfW = -__builtin_huge_valf();
constexpr uint32_t kMinSmem = 118784u;        // one CTA per SM (each allocates all TMEM)

// D = A B^T, both operands K-major over nks 16-column K-steps held in 64-column panels
// (panel strides given in 16-byte units).
__device__ __forceinline__ void mma_kk(uint32_t d, DescWords a, uint32_t a_panel16, DescWords b,
                                       uint32_t b_panel16, int nks, uint32_t idesc) {
#pragma unroll 1
  for (int ks = 0; ks < nks; ++ks) {
    const uint32_t ao = (uint32_t)(ks >> 2) * a_panel16 + (uint32_t)(ks & 3) * 2;
    const uint32_t bo = (uint32_t)(ks >> 2) * b_panel16 + (uint32_t)(ks & 3) * 2;
    if (ks == 0)
      mma_ss_w<0>(d, a, ao, b, bo, idesc);
    else
      mma_ss_w<1>(d, a, ao, b, bo, idesc);
  }
}

// ------------------------------------------------------------------ forward

struct WideFwdGeo {
  uint32_t off_q, off_k, off_v, kb, vb, total;
  int nst;  // K / V ring stages (2 when they fit, else 1)
};

__host__ __device__ inline WideFwdGeo wide_fwd_geo(int DPK, int DPV) {
  WideFwdGeo g;
  g.off_q = 2048;
  const uint32_t qb = (uint32_t)(DPK / 64) * W_PANEL128;
  g.kb = (uint32_t)(DPK / 64) * W_PANEL128;
  g.vb = (uint32_t)(DPV / 64) * W_PANEL128;
  g.nst = (g.off_q + qb + 2u * (g.kb + g.vb) <= 232448u) ? 2 : 1;
  g.off_k = g.off_q + qb;
  g.off_v = g.off_k + (uint32_t)g.nst * g.kb;
  g.total = g.off_v + (uint32_t)g.nst * g.vb;
  return g;
}

enum WFBar : int {
  WF_Q = 0, WF_KF0, WF_KF1, WF_KE0, WF_KE1, WF_VF0, WF_VF1, WF_VE0, WF_VE1, WF_SF0, WF_SF1,
  WF_PF0, WF_PF1, WF_PD0, WF_PD1, WF_ACC, WF_DRAIN, WF_COUNT
};
constexpr uint32_t WF_TMEM = 256, WF_ABORT = 260;
constexpr uint32_t WFT_O = 256;

}  // namespace

// Warps: 0 TMA producer (Q once, the K and V rings), 1 TMEM allocator and MMA issue (lane
// 0), 2-3 idle, 4-7 softmax and epilogue (thread = query row = TMEM lane).
template <bool SOFTCAP, bool F16>
__global__ void __launch_bounds__(256, 1)
    fwd_wide_kernel(const __grid_constant__ WideParams p, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem_raw + WF_ABORT);
  auto bar = [&](int i) -> uint32_t { return sbase + 8u * (uint32_t)i; };
  const WideFwdGeo geo = wide_fwd_geo(p.DPK, p.DPV);
  const int nst = geo.nst;

  // the work item: query tiles longest first (under causal masking the last ones see the
  // most keys)
  const int per_m = p.B * p.H;
  const int m = p.Mb - 1 - (int)(blockIdx.x / (unsigned)per_m);
  const int bh = (int)(blockIdx.x % (unsigned)per_m);
  const int b = bh / p.H, h = bh - (bh / p.H) * p.H, hk = h / p.G;
  MaskGeom gm;
  gm.Sq = p.Sq; gm.Sk = p.Sk; gm.lo = p.lo64; gm.hi = p.hi64;
  gm.tm = 128; gm.tn = 128; gm.Mb = p.Mb; gm.Nb = p.Nb;
  int64_t nb64 = 0, ne64 = 0;
  n_range(gm, m, &nb64, &ne64);
  const int n_begin = (int)nb64, nvis = (int)(ne64 - nb64);

  if (threadIdx.x == 0) {
    *s_abort = 0;
    if ((sbase & 1023u) != 0) {
      // the tile layout assumes a 1024-byte aligned dynamic shared-memory base
      if (p.status) atomicExch(p.status, kWideTimeout - 99);
      *s_abort = 1;
    }
    for (int i = 0; i < WF_COUNT; ++i) mbar_init(bar(i), (i == WF_PF0 || i == WF_PF1) ? 4 : 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + WF_TMEM, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<uint32_t*>(smem_raw + WF_TMEM);
  AbortState st{s_abort, p.status, p.wait_limit};

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && nvis > 0 && *s_abort == 0) {
      const int npk = p.DPK / 64, npv = p.DPV / 64;
      mbar_arrive_expect_tx(bar(WF_Q), (uint32_t)npk * W_PANEL128);
      for (int pn = 0; pn < npk; ++pn)
        tma_load_4d(sbase + geo.off_q + pn * W_PANEL128, &tq, pn * 64, h, m * 128, b, bar(WF_Q));
      int nk = 0, nv = 0;
      for (int t = 0; t < nvis; ++t) {
        const int n0 = (n_begin + t) * 128;
        const int ks = t % nst;
        if (t >= nst && !mbar_wait(bar(WF_KE0 + ks), ((t - nst) / nst) & 1, st, kWideTimeout - 1)) break;
        mbar_arrive_expect_tx(bar(WF_KF0 + ks), geo.kb);
        for (int pn = 0; pn < npk; ++pn)
          tma_load_4d(sbase + geo.off_k + ks * geo.kb + pn * W_PANEL128, &tk, pn * 64, hk, n0, b,
                      bar(WF_KF0 + ks));
        ++nk;
        if (t >= nst && !mbar_wait(bar(WF_VE0 + ks), ((t - nst) / nst) & 1, st, kWideTimeout - 2)) break;
        mbar_arrive_expect_tx(bar(WF_VF0 + ks), geo.vb);
        for (int pn = 0; pn < npv; ++pn)
          tma_load_4d(sbase + geo.off_v + ks * geo.vb + pn * W_PANEL128, &tv, pn * 64, hk, n0, b,
                      bar(WF_VF0 + ks));
        ++nv;
      }
      // every copy started here must land before the CTA may exit: the last load of each
      // ring stage (and Q)
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      mbar_wait(bar(WF_Q), 0, dr, kWideTimeout - 3);
      for (int k2 = 0; k2 < nst && k2 < nk; ++k2) {
        const int last = nk - 1 - ((nk - 1 - k2) % nst);
        mbar_wait(bar(WF_KF0 + last % nst), (last / nst) & 1, dr, kWideTimeout - 3);
      }
      for (int k2 = 0; k2 < nst && k2 < nv; ++k2) {
        const int last = nv - 1 - ((nv - 1 - k2) % nst);
        mbar_wait(bar(WF_VF0 + last % nst), (last / nst) & 1, dr, kWideTimeout - 3);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // S_0, S_1, then per key tile t: O (+)= P_t V_t once P_t is written (and O rescaled),
    // then S_t+2 into the buffer P_t occupies (one thread's MMAs run in issue order).
    if (lane == 0 && nvis > 0) {
      const uint32_t idS = idesc_h<F16>(128, 128, false, false);
      const uint32_t idO = idesc_h<F16>(128, p.DPV, false, true);
      const DescWords dq = desc_words(sbase + geo.off_q, 16, 1024, SWZ_128B);
      bool ok = mbar_wait_spin(bar(WF_Q), 0, st, kWideTimeout - 10);
      auto issue_S = [&](int x) -> bool {
        const int ks = x % nst;
        if (!mbar_wait_spin(bar(WF_KF0 + ks), (x / nst) & 1, st, kWideTimeout - 11)) return false;
        tc_fence_after();
        const DescWords dk = desc_words(sbase + geo.off_k + ks * geo.kb, 16, 1024, SWZ_128B);
        mma_kk(tmem + (x & 1) * 128, dq, W_PANEL128 >> 4, dk, W_PANEL128 >> 4, p.DPK / 16, idS);
        mma_commit(bar(WF_SF0 + (x & 1)));
        mma_commit(bar(WF_KE0 + ks));
        return true;
      };
      if (ok) ok = issue_S(0);
      if (ok && nvis > 1) ok = issue_S(1);
      for (int t = 0; ok && t < nvis; ++t) {
        if (!mbar_wait_spin(bar(WF_PF0 + (t & 1)), (t >> 1) & 1, st, kWideTimeout - 12)) {
          ok = false;
          break;
        }
        const int vs = t % nst;
        if (!mbar_wait_spin(bar(WF_VF0 + vs), (t / nst) & 1, st, kWideTimeout - 13)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const DescWords dv = desc_words(sbase + geo.off_v + vs * geo.vb, W_PANEL128, 1024, SWZ_128B);
        // A = P: keys [0, 64) as pairs in columns [0, 32), keys [64, 128) in [64, 96)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a_t = tmem + (t & 1) * 128 + (ks >> 2) * 64 + (ks & 3) * 8;
          if (ks == 0)
            mma_ts_wp(tmem + WFT_O, a_t, dv, 0, idO, t > 0 ? 1u : 0u);
          else
            mma_ts_w<1>(tmem + WFT_O, a_t, dv, ks * 128, idO);
        }
        mma_commit(bar(WF_VE0 + vs));
        mma_commit(bar(WF_PD0 + (t & 1)));
        if (t + 2 < nvis && !issue_S(t + 2)) {
          ok = false;
          break;
        }
      }
      if (ok) mma_commit(bar(WF_ACC));
      // every MMA must be complete before the CTA releases tensor memory
      mma_commit(bar(WF_DRAIN));
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      mbar_wait(bar(WF_DRAIN), 0, dr, kWideTimeout - 15);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // query row in the tile = TMEM lane
    const int i = m * 128 + r;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};
    float mrow = kNegInfW;  // running maximum (log2 units); moved only by more than 8
    float lrow = 0.f;       // running sum of P relative to mrow
    bool ok = true;
    for (int t = 0; t < nvis; ++t) {
      const int n = n_begin + t;
      const int kb = n * 128;
      const bool need_mask = !tile_full(gm, m, n);
      // visible columns: lo <= key - i <= hi and key < Sk  <=>  c in [cmin, cmax]
      const int cmin = max(i + p.lo - kb, -1);
      const int cmax = min(min(i + p.hi - kb, p.Sk - 1 - kb), 1 << 20);
      const uint32_t sbuf = t_lane + (t & 1) * 128;
      if (!warp_wait(bar(WF_SF0 + (t & 1)), (t >> 1) & 1, st, kWideTimeout - 30)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[128];
      float mx = kNegInfW;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32(sbuf + c * 32, rr);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = c * 32 + e;
          const float s = __uint_as_float(rr[e]);
          float v = SOFTCAP ? kc.cap_log2 * tanh_exp2(s * kc.cap_scale) : s * kc.scale_log2;
          if (need_mask) v = (col >= cmin && col <= cmax) ? v : kNegInfW;
          x[col] = v;
          mx = fmaxf(mx, v);
        }
      }
      float alpha = 1.f;
      if (t == 0) {
        mrow = mx;
      } else if (mx > mrow + 8.f) {
        alpha = ex2_approx(mrow - mx);  // mrow finite, or -inf: alpha = 0
        mrow = mx;
      }
      const float muse = mrow == kNegInfW ? 0.f : mrow;  // all masked so far: P = 0
      float sum = 0.f;
#pragma unroll
      for (int hq = 0; hq < 4; ++hq) {  // 32-key groups; pairs of keys per column
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(x[hq * 32 + 2 * e] - muse);
          const float p1 = ex2_approx(x[hq * 32 + 2 * e + 1] - muse);
          sum += p0 + p1;
          pk[e] = pack_h2<F16>(p0, p1);
        }
        tmem_st16(sbuf + (hq >> 1) * 64 + (hq & 1) * 16, pk);
      }
      lrow = lrow * alpha + sum;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds the products up to key tile t-1: wait for the last one, then rescale
        if (!warp_wait(bar(WF_PD0 + ((t - 1) & 1)), ((t - 1) >> 1) & 1, st, kWideTimeout - 31)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < p.DPV / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(t_lane + WFT_O + c * 16, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(t_lane + WFT_O + c * 16, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(WF_PF0 + (t & 1)));
    }
    // O = acc / l, LSE = (m + log2 l) * ln 2; no visible key: O = 0, LSE = +inf
    bool acc_ok = ok && nvis > 0;
    if (acc_ok) {
      acc_ok = warp_wait(bar(WF_ACC), 0, st, kWideTimeout - 32);
      if (acc_ok) tc_fence_after();
    }
    const bool store = i < p.Sq && (nvis == 0 || acc_ok) && *s_abort == 0;
    const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
    uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + (int64_t)b * p.o_sb + (int64_t)i * p.o_ss +
                     (int64_t)h * p.o_sh;
#pragma unroll 1
    for (int c = 0; c < p.DPV / 16; ++c) {
      uint32_t o[16];
      if (acc_ok) {
        tmem_ld16(t_lane + WFT_O + c * 16, o);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = 0u;
      }
      uint32_t pk[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        pk[e] = pack_h2<F16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
      if (store) {
        if (c * 16 < p.Dv) *reinterpret_cast<uint4*>(orow + c * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        if (c * 16 + 8 < p.Dv)
          *reinterpret_cast<uint4*>(orow + c * 16 + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    if (store) {
      const float lse = lrow > 0.f ? (mrow + log2f(lrow)) * 0.69314718055994531f
                                   : __int_as_float(0x7f800000);
      p.lse[(int64_t)b * p.lse_sb + (int64_t)h * p.lse_sh + (int64_t)i * p.lse_ss] = lse;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ backward

namespace {

struct WideBwdGeo {
  uint32_t off_k, off_v, off_q, off_do, off_ds, off_stg, total, kb, vb, qb, dob;
  int nst;  // Q / dO stages: 2 when they fit in shared memory, else 1
};

__host__ __device__ inline WideBwdGeo wide_bwd_geo(int DPK, int DPV) {
  WideBwdGeo g;
  g.kb = (uint32_t)(DPK / 64) * W_PANEL128;
  g.vb = (uint32_t)(DPV / 64) * W_PANEL128;
  g.qb = (uint32_t)(DPK / 64) * W_PANEL64;
  g.dob = (uint32_t)(DPV / 64) * W_PANEL64;
  g.off_k = 3072;
  g.off_v = g.off_k + g.kb;
  g.off_q = g.off_v + g.vb;
  g.nst = (g.off_q + 2u * (g.qb + g.dob) + 32768u <= 232448u) ? 2 : 1;
  g.off_do = g.off_q + (uint32_t)g.nst * g.qb;
  g.off_ds = g.off_do + (uint32_t)g.nst * g.dob;
  g.off_stg = g.off_ds + 16384;
  g.total = g.off_stg + 16384;
  return g;
}

enum WBBar : int {
  WB_KV = 0, WB_QF0, WB_QF1, WB_QE0, WB_QE1, WB_DOF0, WB_DOF1, WB_DOE0, WB_DOE1, WB_SF, WB_DPF,
  WB_PF, WB_DSF, WB_DQF, WB_DQE, WB_DSE, WB_ACC, WB_DRAIN, WB_COUNT
};
// small region: barriers, TMEM slot, abort flag, ticket, and per Q stage the step's LSE2 and
// D (64 fp32 each)
constexpr uint32_t WB_TMEM = 512, WB_ABORT = 516, WB_TICKET = 520, WB_LSE = 1024, WB_DSUM = 1536;
constexpr uint32_t WBT_DK = 0, WBT_DV = 128, WBT_S = 256, WBT_DP = 320, WBT_DQ = 384;

}  // namespace

// Warps: 0 TMA producer, 1 TMEM allocator and MMA issue (whole warp, one elected lane
// issues), 2-3 idle, 4-7 dQ drain (thread = head-dim row of the slice = TMEM lane), 8-15
// two compute warpgroups (thread = key row = TMEM lane; warpgroup w owns queries
// [32 w, 32 w + 32) of each 64-query block).
template <bool SOFTCAP, bool F16>
__global__ void __launch_bounds__(512, 1)
    bwd_wide_kernel(const __grid_constant__ WideParams p, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tdo) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem_raw + WB_ABORT);
  auto bar = [&](int i) -> uint32_t { return sbase + 8u * (uint32_t)i; };
  const WideBwdGeo geo = wide_bwd_geo(p.DPK, p.DPV);
  const int nst = geo.nst;

  if (threadIdx.x == 0) {
    // the tile index: the block index, or in the ordered mode a ticket, so that every key
    // tile whose dQ partials this one must wait for was claimed by a CTA already running
    *reinterpret_cast<volatile int*>(smem_raw + WB_TICKET) =
        p.deterministic ? atomicAdd(p.ticket, 1) : (int)blockIdx.x;
    *s_abort = 0;
    if ((sbase & 1023u) != 0) {
      atomicExch(p.status, kWideTimeout - 98);
      *s_abort = 1;
    }
    for (int i = 0; i < WB_COUNT; ++i) {
      const int cnt = (i == WB_PF || i == WB_DSF) ? 8 : (i == WB_DQE ? 4 : 1);
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + WB_TMEM, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<uint32_t*>(smem_raw + WB_TMEM);
  AbortState st{s_abort, p.status, p.wait_limit};

  // the tile: key-tile major (under causal masking the low key tiles see the most queries;
  // in the ordered mode the highest key tile comes first, since dQ partials are added from
  // the highest key tile down), then batch, kv-head, slice
  const int tix = *reinterpret_cast<volatile int*>(smem_raw + WB_TICKET);
  const int per_n = p.B * p.Hk * p.nslice;
  const int n0t = tix / per_n;
  const int n = p.deterministic ? p.Nb - 1 - n0t : n0t;
  int rem = tix - n0t * per_n;
  const int s = rem % p.nslice;
  rem /= p.nslice;
  const int hk = rem % p.Hk;
  const int b = rem / p.Hk;
  const int kcols = min(max(p.DPK - 128 * s, 0), 128);  // dK / dQ columns of this slice
  const int vcols = min(max(p.DPV - 128 * s, 0), 128);  // dV columns of this slice
  MaskGeom gm;  // 64-query blocks x 128-key tiles
  gm.Sq = p.Sq; gm.Sk = p.Sk; gm.lo = p.lo64; gm.hi = p.hi64;
  gm.tm = 64; gm.tn = 128; gm.Mb = p.Mb; gm.Nb = p.Nb;
  int64_t mb64 = 0, me64 = 0;
  m_range(gm, n, &mb64, &me64);
  const int m_begin = (int)mb64, m_count = (int)(me64 - mb64);
  const int total = m_count * p.G;  // steps (g, m), m fastest

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && total > 0 && *s_abort == 0) {
      const int npk = p.DPK / 64, npv = p.DPV / 64;
      const int n0 = n * 128;
      mbar_arrive_expect_tx(bar(WB_KV), geo.kb + geo.vb);
      for (int pn = 0; pn < npk; ++pn)
        tma_load_4d(sbase + geo.off_k + pn * W_PANEL128, &tk, pn * 64, hk, n0, b, bar(WB_KV));
      for (int pn = 0; pn < npv; ++pn)
        tma_load_4d(sbase + geo.off_v + pn * W_PANEL128, &tv, pn * 64, hk, n0, b, bar(WB_KV));
      int nq = 0, ndo = 0;
      for (int it = 0; it < total; ++it) {
        const int g = it / m_count;
        const int mb = m_begin + (it - g * m_count);
        const int h = hk * p.G + g;
        const int q0 = mb * 64;
        const int sq = it % nst;
        // Q, LSE2 and D of step it go to stage it % nst once that stage's last reader (the
        // dK product nst steps back) is done
        if (it >= nst && !mbar_wait(bar(WB_QE0 + sq), ((it - nst) / nst) & 1, st, kWideTimeout - 41)) break;
        mbar_arrive_expect_tx(bar(WB_QF0 + sq), geo.qb + 512);
        for (int pn = 0; pn < npk; ++pn)
          tma_load_4d(sbase + geo.off_q + sq * geo.qb + pn * W_PANEL64, &tq, pn * 64, h, q0, b,
                      bar(WB_QF0 + sq));
        const size_t row = ((size_t)b * p.H + h) * p.Sq_r + q0;
        bulk_load(sbase + WB_LSE + sq * 256, p.lse2 + row, 256, bar(WB_QF0 + sq));
        bulk_load(sbase + WB_DSUM + sq * 256, p.dsum + row, 256, bar(WB_QF0 + sq));
        ++nq;
        // dO of step it once the dV product nst steps back is done
        if (it >= nst && !mbar_wait(bar(WB_DOE0 + sq), ((it - nst) / nst) & 1, st, kWideTimeout - 42)) break;
        mbar_arrive_expect_tx(bar(WB_DOF0 + sq), geo.dob);
        for (int pn = 0; pn < npv; ++pn)
          tma_load_4d(sbase + geo.off_do + sq * geo.dob + pn * W_PANEL64, &tdo, pn * 64, h, q0, b,
                      bar(WB_DOF0 + sq));
        ++ndo;
      }
      // every copy started here must land before the CTA may exit: the last load of each
      // stage
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      mbar_wait(bar(WB_KV), 0, dr, kWideTimeout - 43);
      for (int k2 = 0; k2 < nst && k2 < nq; ++k2) {
        const int last = nq - 1 - ((nq - 1 - k2) % nst);
        mbar_wait(bar(WB_QF0 + last % nst), (last / nst) & 1, dr, kWideTimeout - 43);
      }
      for (int k2 = 0; k2 < nst && k2 < ndo; ++k2) {
        const int last = ndo - 1 - ((ndo - 1 - k2) % nst);
        mbar_wait(bar(WB_DOF0 + last % nst), (last / nst) & 1, dr, kWideTimeout - 43);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Per step i: S^T, dP^T; dV (after P^T) -> dO free; dK (after dS^T) -> Q free; dQ^T
    // (after the previous dQ^T is drained) -> dq_full; dS free.  With two Q / dO stages
    // the next step's S^T follows dV_i and its dP^T follows dK_i (they overwrite P^T_i and
    // dS^T_i, which those products read: issue order), so the compute warps find the next
    // scores ready; with one stage the next Q can only land after dK_i, so the steps run
    // one after another.
    if (total > 0) {
      const bool leader = elect_one();
      auto wspin = [&](uint32_t bb, uint32_t par, int code) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_spin(bb, par, st, code));
      };
      const uint32_t idS = idesc_h<F16>(128, 64, false, false);
      const uint32_t idV = idesc_h<F16>(128, vcols > 0 ? vcols : 64, false, true);
      const uint32_t idK = idesc_h<F16>(128, kcols > 0 ? kcols : 64, false, true);
      const uint32_t idQ = idesc_h<F16>(128, 64, true, true);
      const DescWords aK = desc_words(sbase + geo.off_k, 16, 1024, SWZ_128B);
      const DescWords aV = desc_words(sbase + geo.off_v, 16, 1024, SWZ_128B);
      const DescWords aKt = desc_words(sbase + geo.off_k + 2 * s * W_PANEL128, W_PANEL128, 1024, SWZ_128B);
      const DescWords bDS = desc_words(sbase + geo.off_ds, W_PANEL64, 1024, SWZ_128B);
      auto do_S = [&](int i) -> bool {
        const int sq = i % nst;
        if (!wspin(bar(WB_QF0 + sq), (i / nst) & 1, kWideTimeout - 11)) return false;
        tc_fence_after();
        const DescWords bQ = desc_words(sbase + geo.off_q + sq * geo.qb, 16, 1024, SWZ_128B);
        if (leader) mma_kk(tmem + WBT_S, aK, W_PANEL128 >> 4, bQ, W_PANEL64 >> 4, p.DPK / 16, idS);
        if (leader) mma_commit(bar(WB_SF));
        return true;
      };
      auto do_dP = [&](int i) -> bool {
        const int sq = i % nst;
        if (!wspin(bar(WB_DOF0 + sq), (i / nst) & 1, kWideTimeout - 12)) return false;
        tc_fence_after();
        const DescWords bDO = desc_words(sbase + geo.off_do + sq * geo.dob, 16, 1024, SWZ_128B);
        if (leader) mma_kk(tmem + WBT_DP, aV, W_PANEL128 >> 4, bDO, W_PANEL64 >> 4, p.DPV / 16, idS);
        if (leader) mma_commit(bar(WB_DPF));
        return true;
      };
      // dV_s += P^T dO_s: A = P^T (queries [0, 32) as pairs in columns [0, 16) of S^T,
      // [32, 64) in [32, 48)), K = 64 queries in 4 steps
      auto do_dV = [&](int i) -> bool {
        const int sq = i % nst;
        if (!wspin(bar(WB_PF), i & 1, kWideTimeout - 13)) return false;
        tc_fence_after();
        const DescWords bDOs =
            desc_words(sbase + geo.off_do + sq * geo.dob + 2 * s * W_PANEL64, W_PANEL64, 1024, SWZ_128B);
        if (leader && vcols > 0) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_wp(tmem + WBT_DV, tmem + WBT_S + (ks >> 1) * 32 + (ks & 1) * 8, bDOs, ks * 128, idV,
                      (i > 0 || ks > 0) ? 1u : 0u);
        }
        if (leader) mma_commit(bar(WB_DOE0 + sq));
        return true;
      };
      // dK_s += dS^T Q_s: A = dS^T over the dP^T columns, same layout
      auto do_dK = [&](int i) -> bool {
        const int sq = i % nst;
        if (!wspin(bar(WB_DSF), i & 1, kWideTimeout - 14)) return false;
        tc_fence_after();
        const DescWords bQs =
            desc_words(sbase + geo.off_q + sq * geo.qb + 2 * s * W_PANEL64, W_PANEL64, 1024, SWZ_128B);
        if (leader && kcols > 0) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_wp(tmem + WBT_DK, tmem + WBT_DP + (ks >> 1) * 32 + (ks & 1) * 8, bQs, ks * 128, idK,
                      (i > 0 || ks > 0) ? 1u : 0u);
        }
        if (leader) mma_commit(bar(WB_QE0 + sq));
        return true;
      };
      // dQ_s^T = K_s^T dS^T: A = the K tile's slice panels read MN-major (M = 128 head-dim
      // rows), B = dS^T from shared memory (N = 64 queries), K = 128 keys in 8 steps
      auto do_dQ = [&](int i) -> bool {
        if (kcols > 0) {
          if (i >= 1 && !wspin(bar(WB_DQE), (i - 1) & 1, kWideTimeout - 15)) return false;
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              if (ks == 0)
                mma_ss_w<0>(tmem + WBT_DQ, aKt, 0, bDS, 0, idQ);
              else
                mma_ss_w<1>(tmem + WBT_DQ, aKt, ks * 128, bDS, ks * 128, idQ);
            }
          }
          if (leader) mma_commit(bar(WB_DQF));
        }
        if (leader) mma_commit(bar(WB_DSE));
        return true;
      };
      bool ok = wspin(bar(WB_KV), 0, kWideTimeout - 10);
      if (nst == 1) {
        for (int it = 0; ok && it < total; ++it)
          ok = do_S(it) && do_dP(it) && do_dV(it) && do_dK(it) && do_dQ(it);
      } else {
        ok = ok && do_S(0) && do_dP(0);
        for (int it = 0; ok && it < total; ++it) {
          const bool more = it + 1 < total;
          ok = do_dV(it) && (!more || do_S(it + 1)) && do_dK(it) && (!more || do_dP(it + 1)) &&
               do_dQ(it);
        }
      }
      if (ok && leader) mma_commit(bar(WB_ACC));
      if (leader) mma_commit(bar(WB_DRAIN));
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      mbar_wait(bar(WB_DRAIN), 0, dr, kWideTimeout - 16);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ dQ drain
    const int qd = warp & 3;
    const int dl = qd * 32 + lane;  // head-dim row of the slice = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const uint32_t stg = sbase + geo.off_stg;
    if (kcols > 0) {
      for (int it = 0; it < total; ++it) {
        const int g = it / m_count;
        const int mb = m_begin + (it - g * m_count);
        const int h = hk * p.G + g;
        bool ok = warp_wait(bar(WB_DQF), it & 1, st, kWideTimeout - 20);
        uint32_t v[64];
        if (ok) {
          tc_fence_after();
          uint32_t r0[32], r1[32];
          tmem_ld32(t_lane + WBT_DQ, r0);
          tmem_ld32(t_lane + WBT_DQ + 32, r1);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            v[e] = r0[e];
            v[32 + e] = r1[e];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(WB_DQE));
        }
        const size_t blk = (((size_t)b * p.H + h) * p.Mb + mb) * (size_t)p.nks + s;
        float* dst = p.dq_accum + blk * 8192;
        // ordered mode: the block takes this key tile's partial once every higher key tile
        // that reaches it has added its own (its counter equals this tile's rank from the
        // top); a wait that runs out stops the CTA
        if (p.deterministic && threadIdx.x == 128 && ok) {
          int64_t nb = 0, ne = 0;
          n_range(gm, mb, &nb, &ne);
          const int want = (int)ne - 1 - n;
          const int* sem = p.sems + blk;
          const long long t0 = clock64();
          while (true) {
            int cur;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(cur) : "l"(sem) : "memory");
            if (cur == want) break;
            if (*s_abort) break;
            if (clock64() - t0 > p.wait_limit) {
              raise_timeout(st, kWideTimeout - 21);
              break;
            }
          }
          // the bulk adds (async proxy) come after the acquire
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        // two halves of 64 rows each through the 16 KB staging buffer; every drain thread
        // reaches every named barrier
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          if (threadIdx.x == 128) bulk_wait_read_all();
          named_bar_sync(1, 128);
          if (ok && (qd >> 1) == hf && dl < kcols) {
            const uint32_t row = stg + (uint32_t)(dl - 64 * hf) * 256u;
#pragma unroll
            for (int c = 0; c < 16; ++c)
              st_shared_v4(row + (uint32_t)((c ^ (dl & 15)) * 16), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                           v[4 * c + 3]);
            fence_proxy_async_smem();
          }
          named_bar_sync(1, 128);
          if (threadIdx.x == 128 && 64 * hf < kcols && *s_abort == 0) {
            bulk_reduce_add_f32(dst + hf * 64 * 64, stg, 16384);
            bulk_commit();
          }
        }
        // ordered mode: hand the block on once the adds have landed
        if (p.deterministic && threadIdx.x == 128 && *s_abort == 0) {
          bulk_wait_all();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.sems + blk) : "memory");
        }
      }
    }
    if (threadIdx.x == 128) bulk_wait_all();
  } else if (warp >= 8) {
    // ------------------------------------------------------------------ compute
    const int wg = (warp - 8) >> 2;
    const int qd = warp & 3;
    const int jl = qd * 32 + lane;  // key row in the tile = TMEM lane
    const int col0 = wg * 32;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};
    const int j = n * 128 + jl;
    const bool row_ok = j < p.Sk;
    const uint32_t sDS = sbase + geo.off_ds + (uint32_t)jl * 128u;
    bool alive = true;
    for (int it = 0; it < total; ++it) {
      const int mb = m_begin + (it - (it / m_count) * m_count);
      const int m0 = mb * 64;
      const bool need_mask = !tile_full(gm, mb, n);
      // visible columns: lo <= (j - i) <= hi with i = m0 + col0 + ql  <=>  ql in [qmin, qmax]
      const int base = j - m0 - col0;
      const int qmin = row_ok ? max(base - p.hi, -1) : 1 << 20;
      const int qmax = row_ok ? min(base - p.lo, 1 << 20) : -1;
      if (!warp_wait(bar(WB_SF), it & 1, st, kWideTimeout - 30)) { alive = false; break; }
      tc_fence_after();
      const float* s_lse = reinterpret_cast<const float*>(smem_raw + WB_LSE + (it % nst) * 256);
      const float* s_dsum = reinterpret_cast<const float*>(smem_raw + WB_DSUM + (it % nst) * 256);
      uint32_t r[32];
      tmem_ld32(t_lane + WBT_S + col0, r);
      float pc[32];  // P (times 1 - tanh^2 under softcap), kept for dS
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float pr[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ql = e + u;
          float fac;
          float pv = prob<SOFTCAP>(kc, __uint_as_float(r[ql]), s_lse[col0 + ql], &fac);
          if (need_mask) pv = (ql >= qmin && ql <= qmax) ? pv : 0.f;
          pr[u] = pv;
          pc[ql] = SOFTCAP ? pv * fac : pv;
        }
        pk[e >> 1] = pack_h2<F16>(pr[0], pr[1]);
      }
      tmem_st16(t_lane + WBT_S + col0, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(WB_PF));

      if (!warp_wait(bar(WB_DPF), it & 1, st, kWideTimeout - 31)) { alive = false; break; }
      if (it >= 1 && !warp_wait(bar(WB_DSE), (it - 1) & 1, st, kWideTimeout - 32)) { alive = false; break; }
      tc_fence_after();
      tmem_ld32(t_lane + WBT_DP + col0, r);
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float d0 = pc[e] * (__uint_as_float(r[e]) - s_dsum[col0 + e]);
        const float d1 = pc[e + 1] * (__uint_as_float(r[e + 1]) - s_dsum[col0 + e + 1]);
        pk[e >> 1] = pack_h2<F16>(d0, d1);
      }
      // dS^T row jl: this warpgroup's 64 bytes are 16-byte chunks 4 wg .. 4 wg + 3 of the
      // 128-byte row, 128B-swizzled
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t chunk = (uint32_t)(wg * 4 + u) ^ (uint32_t)(jl & 7);
        st_shared_v4(sDS + chunk * 16, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      tmem_st16(t_lane + WBT_DP + col0, pk);
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(WB_DSF));
    }

    // ---------------------------------------------------------------- dK / dV epilogue
    // Each warpgroup writes half of the 16-column chunks of the slice's columns.  A key
    // tile with no visible query writes zero rows.
    const bool have = total > 0;
    bool acc_ok = alive;
    if (have && acc_ok) {
      acc_ok = warp_wait(bar(WB_ACC), 0, st, kWideTimeout - 33);
      if (acc_ok) tc_fence_after();
    }
    const bool store = acc_ok && *s_abort == 0 && row_ok;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      const int ncols = which ? kcols : vcols;
      const int c_base = 128 * s;  // first column of the slice
      const int dlim = which ? p.Dk : p.Dv;
      const uint32_t tcol = which ? WBT_DK : WBT_DV;
      const float sc = which ? p.dk_scale : 1.f;
      uint16_t* row = which ? reinterpret_cast<uint16_t*>(p.dk) + (int64_t)b * p.dk_sb +
                                  (int64_t)j * p.dk_ss + (int64_t)hk * p.dk_sh
                            : reinterpret_cast<uint16_t*>(p.dv) + (int64_t)b * p.dv_sb +
                                  (int64_t)j * p.dv_ss + (int64_t)hk * p.dv_sh;
      const int nch = ncols / 16;
      const int nch0 = (nch + 1) / 2;
      const int c0 = wg ? nch0 : 0;
      const int c1 = wg ? nch : nch0;
#pragma unroll 1
      for (int c = c0; c < c1; ++c) {
        uint32_t rr[16];
        if (have && acc_ok) {
          tmem_ld16(t_lane + tcol + c * 16, rr);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) rr[e] = 0u;
        }
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          o[e] = pack_h2<F16>(__uint_as_float(rr[2 * e]) * sc, __uint_as_float(rr[2 * e + 1]) * sc);
        const int col = c_base + c * 16;
        if (store) {
          if (col < dlim) *reinterpret_cast<uint4*>(row + col) = make_uint4(o[0], o[1], o[2], o[3]);
          if (col + 8 < dlim) *reinterpret_cast<uint4*>(row + col + 8) = make_uint4(o[4], o[5], o[6], o[7]);
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

namespace {

// dQ = scale * accumulator, from the transposed, chunk-swizzled blocks of the wide
// backward.  One block of 256 threads per accumulator block (128 head-dim rows x 64
// queries): the 32 KB block is staged in shared memory with coalesced loads, then each
// thread writes 32 columns of one query row.
template <bool F16>
__global__ void __launch_bounds__(256) convert_wide_kernel(const WideParams p) {
  __shared__ float4 tile[2048];
  size_t id = blockIdx.x;
  const int s = (int)(id % (size_t)p.nks);
  id /= (size_t)p.nks;
  const int mb = (int)(id % (size_t)p.Mb);
  const size_t bh = id / (size_t)p.Mb;
  const int b = (int)(bh / (size_t)p.H);
  const int h = (int)(bh - (size_t)b * p.H);
  const float4* src = reinterpret_cast<const float4*>(p.dq_accum) + (size_t)blockIdx.x * 2048;
  for (int k = threadIdx.x; k < 2048; k += 256) tile[k] = __ldcs(src + k);
  __syncthreads();
  const float* t = reinterpret_cast<const float*>(tile);
  const int q = threadIdx.x >> 2;          // query in the block
  const int d0 = (threadIdx.x & 3) * 32;   // first head-dim row of this thread
  const int i = mb * 64 + q;
  if (i >= p.Sq) return;
  uint16_t* out = reinterpret_cast<uint16_t*>(p.dq) + (int64_t)b * p.dq_sb + (int64_t)i * p.dq_ss +
                  (int64_t)h * p.dq_sh;
#pragma unroll
  for (int g8 = 0; g8 < 4; ++g8) {
    const int dd = d0 + g8 * 8;
    const int col = 128 * s + dd;
    if (col >= p.Dk) break;
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int da = dd + 2 * e, db = da + 1;
      const float va = t[da * 64 + (((q >> 2) ^ (da & 15)) << 2) + (q & 3)];
      const float vb = t[db * 64 + (((q >> 2) ^ (db & 15)) << 2) + (q & 3)];
      pk[e] = pack_h2<F16>(va * p.scale, vb * p.scale);
    }
    *reinterpret_cast<uint4*>(out + col) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

size_t wide_fwd_smem_bytes(int DPK, int DPV) {
  const size_t t = wide_fwd_geo(DPK, DPV).total;
  return t > kMinSmem ? t : kMinSmem;
}

size_t wide_bwd_smem_bytes(int DPK, int DPV) {
  const size_t t = wide_bwd_geo(DPK, DPV).total;
  return t > kMinSmem ? t : kMinSmem;
}

cudaError_t launch_fwd_wide(const WideParams& p, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, bool softcap, bool f16, cudaStream_t s) {
  const int64_t items = (int64_t)p.Mb * p.B * p.H;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const size_t smem = wide_fwd_smem_bytes(p.DPK, p.DPV);
  if (smem > 232448) return cudaErrorInvalidConfiguration;
  auto kern = f16 ? (softcap ? fwd_wide_kernel<true, true> : fwd_wide_kernel<false, true>)
                  : (softcap ? fwd_wide_kernel<true, false> : fwd_wide_kernel<false, false>);
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)items, 256, smem, s>>>(p, q, k, v);
  return cudaGetLastError();
}

cudaError_t launch_bwd_wide(const WideParams& p, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const CUtensorMap& dout, bool softcap, bool f16,
                            cudaStream_t s) {
  const int64_t tiles = (int64_t)p.Nb * p.B * p.Hk * p.nslice;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const size_t smem = wide_bwd_smem_bytes(p.DPK, p.DPV);
  if (smem > 232448) return cudaErrorInvalidConfiguration;
  auto kern = f16 ? (softcap ? bwd_wide_kernel<true, true> : bwd_wide_kernel<false, true>)
                  : (softcap ? bwd_wide_kernel<true, false> : bwd_wide_kernel<false, false>);
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)tiles, 512, smem, s>>>(p, q, k, v, dout);
  return cudaGetLastError();
}

cudaError_t launch_convert_wide(const WideParams& p, bool f16, cudaStream_t s) {
  const int64_t blocks = (int64_t)p.B * p.H * p.Mb * p.nks;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  if (f16)
    convert_wide_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(p);
  else
    convert_wide_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
