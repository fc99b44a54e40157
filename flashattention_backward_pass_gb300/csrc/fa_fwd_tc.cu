// fa_fwd_tc.cu — the forward (O and the natural-log LSE) on tcgen05 / TMEM / TMA for sm_103a.
//
// It computes what the Triton page's `_attn_fwd_inner` computes — per key block, scores,
// running row maximum, rescaled running sum and accumulator, and at the end O = acc / l,
// LSE = (m + log2 l) * ln 2 — with the same mask (bottom-right aligned band lo <= j - i
// <= hi, j < Sk) and softcap (z = c * tanh(scale * s / c)) as the backward.
//
// Work item: one 128-query tile of one (batch, q-head), walking the key tiles with a
// visible entry (GQA/MQA page: the kv-head is h / (H / Hk)):
//   S = Q K^T        (M = 128 queries, N = 128 keys, K = Dp; both operands K-major)
//   P = exp2(z * log2e - m)  written as 16-bit pairs over the S columns already read
//   O (+)= P V       (A = P from tensor memory, B = V read MN-major, N = Dp)
// The grid is persistent: the CTAs take the items of a list ordered longest first (under
// causal masking the last query tiles see the most keys) in snake order.  Consecutive
// items overlap: the next item's Q and first K / V tiles load and its first S products
// run while the softmax warps finish the current item and write its O, which lives in
// the other of two TMEM accumulators.  A CTA therefore pays its set-up once, not per
// query tile.
//
// Two softmax warpgroups split the 128 key columns of the score tile: thread (warpgroup
// w, TMEM lane r) owns query row r and columns [64w, 64w + 64).  The two halves of a
// row's maximum meet through shared memory once per key tile (a barrier of the two warps
// that own the row); each warpgroup keeps the row sum of its own columns and the two are
// added at the end.
//
// The running maximum m is only moved (and O, l rescaled by exp2(m_old - m_new)) when
// a new score exceeds it by more than 8 in log2 units; otherwise the stale m is kept and
// P may reach 2^8, well inside bf16 / f16 and the fp32 sums.  O = acc / l and the LSE use
// the same m, so the result is exact up to rounding either way.  After the first key
// tiles a rescale is rare.
//
// Warp roles (12 warps): warp 0 TMA producer of Q (two buffers) and of the K ring; warp 2
// TMA producer of the V ring; warp 1 TMEM allocator and issuer of the P V products, warp
// 3 issuer of the score products (one lane of each issues); warps 4-11 two softmax /
// epilogue warpgroups (warp w reads TMEM lanes 32 (w % 4) .. +31).  Every role walks the
// same item list and counts key tiles and items with work the same way, so the ring and
// buffer phases agree without any exchange.
//
// Tensor memory: S buffers [0, 128) and [128, 256) (P written over the first 32 columns
// of each 64-column half), O accumulators [256, 256 + Dp) and [384, 384 + Dp).
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
constexpr uint32_t FSM_L = 3072;    // [2 item parities][2 warpgroups][128 rows] fp32 row sums
constexpr uint32_t FSMALL = 6144;

template <int DP>
struct GeoF : Panels<DP> {
  using Panels<DP>::TILE_BYTES;
  static constexpr int KST = 2;  // K ring stages
  static constexpr int VST = 2;  // V ring stages
  static constexpr uint32_t OFF_Q = FSMALL;  // 2 buffers (this item and the next)
  static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE_BYTES;
  static constexpr uint32_t TOTAL = OFF_V + VST * TILE_BYTES;
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

// Barriers.  Sx / Px / PDx by score buffer, Qx / ACCx / OEx by item parity (items with
// work), K / V by ring stage.
enum FBar : int {
  F_QF0 = 0, F_QF1, F_QE0, F_QE1, F_KF0, F_KF1, F_KE0, F_KE1, F_VF0, F_VF1, F_VE0, F_VE1,
  F_SF0, F_SF1, F_PF0, F_PF1, F_PD0, F_PD1, F_ACC0, F_ACC1, F_OE0, F_OE1, F_DRAIN,
  F_OS0, F_OS1, F_DRAIN2, F_COUNT
};
static_assert(F_COUNT <= 32, "barrier area holds 32 mbarriers");

constexpr uint32_t FT_S0 = 0, FT_O0 = 256;

constexpr float kNegInf = -__builtin_huge_valf();

template <int N>
struct IntC {
  static constexpr int value = N;
};

// Scores of this thread's 64 columns of its row (`sbuf` addresses column col0 of the row;
// masked columns, MASK: visible iff cmin <= column <= cmax, columns of the whole tile,
// are -inf).  Without softcap x holds the raw scores s (the scale is applied together
// with the subtraction of the maximum in fwd_probs, one fused multiply-add); with softcap
// c x holds z = c * log2e * tanh(scale * s / c).  Returns the maximum over the 64 in
// log2 units (scale * log2e > 0, so the raw maximum scales to the scaled one).
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
      float v = SOFTCAP ? kc.cap_log2 * tanh_exp2(s * kc.cap_scale) : s;
      if (MASK) v = (col >= cmin && col <= cmax) ? v : kNegInf;
      x[c * 32 + e] = v;
      mx = fmaxf(mx, v);
    }
  }
  return SOFTCAP ? mx : mx * kc.scale_log2;
}

// P = exp2(x * mul - m) for the thread's 64 columns (mul = scale * log2e on raw scores,
// 1 on softcapped ones) as 16-bit pairs over the first 32 of them (`sbuf` = column col0):
// columns [0, 64) of the row land in TMEM columns [0, 32), columns [64, 128) in [64, 96),
// the A layout the P V product reads.  Returns the sum of the 64 P values (fp32, before
// rounding).
template <bool F16>
__device__ __forceinline__ float fwd_probs(uint32_t sbuf, float mul, float m, const float (&x)[64]) {
  const uint64_t mul2 = f2_pack(mul, mul), negm2 = f2_pack(-m, -m);
  uint64_t sum2 = 0;  // (+0, +0)
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint64_t t = f2_fma(f2_pack(x[q * 32 + 2 * e], x[q * 32 + 2 * e + 1]), mul2, negm2);
      const float p0 = ex2_approx(f2_lo(t));
      const float p1 = ex2_approx(f2_hi(t));
      sum2 = f2_add(sum2, f2_pack(p0, p1));
      pk[e] = pack_h2<F16>(p0, p1);
    }
    tmem_st16(sbuf + q * 16, pk);
  }
  return f2_lo(sum2) + f2_hi(sum2);
}


// One work item as every role sees it: the query tile, its (batch, head), the sequence's
// geometry and offsets, and the visible key tiles (the element mask's range, filtered by
// the block mask).  Must be called by a whole warp (the block-mask count is a warp sum).
struct FwdItem {
  int m, b, h, hk, tb, q_off, k_off, lo, hi, Sq, Sk, n_begin, nvis;
  MaskGeom gm;
  const uint8_t* brow;
};

__device__ __forceinline__ FwdItem fwd_item(const FwdTcParams& p, int idx, int lane) {
  FwdItem it;
  const int per_m = p.B * p.H;
  it.m = p.Mb - 1 - idx / per_m;  // longest first
  const int bh = idx - (p.Mb - 1 - it.m) * per_m;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  it.hk = it.h / p.G;
  it.q_off = 0;
  it.k_off = 0;
  it.tb = it.b;
  it.lo = p.lo;
  it.hi = p.hi;
  if (p.varlen) {
    // sequence b: rows [cu[b], cu[b+1]) clamped into the packed tensors, so that malformed
    // offsets cannot move a load or a store outside them
    const int q0 = min(max(p.cu_q[it.b], 0), p.total_q);
    int q1 = min(max(p.cu_q[it.b + 1], q0), p.total_q);
    const int k0 = min(max(p.cu_k[it.b], 0), p.total_k);
    int k1 = min(max(p.cu_k[it.b + 1], k0), p.total_k);
    // used lengths: only the first used[b] rows of the range are computed
    if (p.used_q != nullptr) q1 = q0 + min(max(p.used_q[it.b], 0), q1 - q0);
    if (p.used_k != nullptr) k1 = k0 + min(max(p.used_k[it.b], 0), k1 - k0);
    it.q_off = q0;
    it.k_off = k0;
    it.tb = 0;
    it.gm = make_geom(q1 - q0, k1 - k0, p.causal, p.window_left, p.window_right, kTileQ, kTileK);
    it.lo = (int)max64(min64(it.gm.lo, 1ll << 30), -(1ll << 30));
    it.hi = (int)max64(min64(it.gm.hi, 1ll << 30), -(1ll << 30));
  } else {
    it.gm.Sq = p.Sq;
    it.gm.Sk = p.Sk;
    it.gm.lo = p.lo64;
    it.gm.hi = p.hi64;
    it.gm.tm = kTileQ;
    it.gm.tn = kTileK;
    it.gm.Mb = p.Mb;
    it.gm.Nb = p.Nb;
  }
  it.Sq = (int)it.gm.Sq;
  it.Sk = (int)it.gm.Sk;
  int64_t nb = 0, ne = 0;
  if (it.m < it.gm.Mb) n_range(it.gm, it.m, &nb, &ne);  // a shorter sequence may have no tile m
  it.n_begin = (int)nb;
  it.nvis = (int)(ne - nb);
  it.brow = p.block_mask ? p.block_mask + (((size_t)it.b * p.H + it.h) * p.Mb + it.m) * (size_t)p.Nb
                         : nullptr;
  if (it.brow) {
    int c = 0;
    for (int n = (int)nb + lane; n < (int)ne; n += 32) c += it.brow[n] != 0;
    it.nvis = __reduce_add_sync(0xffffffffu, c);
  }
  return it;
}

// The visible key tile after nc (block sparsity skips the removed ones).
__device__ __forceinline__ int fwd_next_tile(const FwdItem& it, int nc) {
  ++nc;
  if (it.brow)
    while (it.brow[nc] == 0) ++nc;
  return nc;
}

}  // namespace

template <int DP, bool SOFTCAP, bool F16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tc_kernel(const __grid_constant__ FwdTcParams p,
                  const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t,
                  const __grid_constant__ CUtensorMap to, const __grid_constant__ CUtensorMap to_t) {
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
    for (int i = 0; i < F_COUNT; ++i) {
      const bool eight = (i == F_PF0 || i == F_PF1 || i == F_OE0 || i == F_OE1 || i == F_OS0 ||
                          i == F_OS1);
      mbar_init(bar(i), eight ? 8 : 1);  // softmax warps arrive on P-full, O-empty, O-staged
    }
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
  const int num_items = p.Mb * p.B * p.H;
  // The items are ordered longest first; round k gives CTA c item k * grid + c on even
  // rounds and k * grid + (grid - 1 - c) on odd ones, so a CTA that got a long item in
  // one round gets a short one in the next (snake order) and the sums even out.
  auto item_of = [&](int k) -> int {
    const int c = (k & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    return k * (int)gridDim.x + c;
  };

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ TMA producers
    // Warp 0 loads each item's Q (two buffers, so the next item's Q lands while this one
    // runs) and the K ring, warp 2 the V ring; each refills a stage as soon as its own last
    // reader is done (Q: the item's last MMA, K: its S product, V: its P V product).
    const bool kside = warp == 0;
    const CUtensorMap* tm = kside ? &tk : &tv;
    const CUtensorMap* tm_t = kside ? &tk_t : &tv_t;
    const int nst = kside ? G::KST : G::VST;
    const uint32_t base = sbase + (kside ? G::OFF_K : G::OFF_V);
    const int full0 = kside ? F_KF0 : F_VF0, empty0 = kside ? F_KE0 : F_VE0;
    if (lane == 0) {
      tma_prefetch_desc(tm);
      if (kside) tma_prefetch_desc(&tq);
    }
    int c = 0, qn = 0, qarmed = 0;  // tiles loaded into the ring, items with work, Q loads
    bool alive = true;
    for (int k = 0, idx = item_of(0); alive && idx < num_items; idx = item_of(++k)) {
      const FwdItem I = fwd_item(p, idx, lane);
      if (*s_abort) break;
      if (I.nvis == 0) continue;
      if (lane == 0) {
        if (kside) {
          const int qb = qn & 1;
          // the buffer's item two back: its S products are done and its O, staged there,
          // has been read by the tensor stores
          if (qn >= 2 && (!mbar_wait(bar(F_QE0 + qb), ((qn - 2) >> 1) & 1, st, kFwdTimeout - 4) ||
                          !mbar_wait(bar(F_OS0 + qb), ((qn - 2) >> 1) & 1, st, kFwdTimeout - 5))) {
            alive = false;
          } else {
            const uint32_t qdst = sbase + G::OFF_Q + qb * G::TILE_BYTES;
            mbar_arrive_expect_tx(bar(F_QF0 + qb), G::TILE_BYTES);
            for (int pn = 0; pn < G::NFULL; ++pn)
              tma_load_4d(qdst + pn * G::FULL_BYTES, &tq, pn * 64, I.h, I.q_off + I.m * kTileQ, I.tb, bar(F_QF0 + qb));
            if (G::TAIL) tma_load_4d(qdst + G::TAIL_OFF, &tq_t, G::NFULL * 64, I.h, I.q_off + I.m * kTileQ, I.tb, bar(F_QF0 + qb));
            ++qarmed;
          }
        }
        int ncur = I.n_begin - 1;
        for (int t = 0; alive && t < I.nvis; ++t, ++c) {
          ncur = fwd_next_tile(I, ncur);
          const int n0 = I.k_off + ncur * kTileK;
          const int ks = c % nst;
          if (c >= nst && !mbar_wait(bar(empty0 + ks), ((c - nst) / nst) & 1, st, kFwdTimeout - 1)) {
            alive = false;
            break;
          }
          const uint32_t dst = base + ks * G::TILE_BYTES;
          mbar_arrive_expect_tx(bar(full0 + ks), G::TILE_BYTES);
          for (int pn = 0; pn < G::NFULL; ++pn)
            tma_load_4d(dst + pn * G::FULL_BYTES, tm, pn * 64, I.hk, n0, I.tb, bar(full0 + ks));
          if (G::TAIL) tma_load_4d(dst + G::TAIL_OFF, tm_t, G::NFULL * 64, I.hk, n0, I.tb, bar(full0 + ks));
        }
      }
      ++qn;
      alive = __shfl_sync(0xffffffffu, alive, 0);
    }
    // every copy this thread started must land before the CTA may exit: the last phase of
    // each stage (and of each Q buffer) that it armed
    if (lane == 0) {
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      for (int k2 = 0; k2 < nst && k2 < c; ++k2) {
        const int last = c - 1 - ((c - 1 - k2) % nst);  // the last load into stage k2
        mbar_wait(bar(full0 + (last % nst)), (last / nst) & 1, dr, kFwdTimeout - 3);
      }
      if (kside)
        for (int k2 = 0; k2 < 2 && k2 < qarmed; ++k2) {
          const int last = qarmed - 1 - k2;
          mbar_wait(bar(F_QF0 + (last & 1)), (last >> 1) & 1, dr, kFwdTimeout - 3);
        }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 1 issues the P V products, warp 3 the score products.  Per key tile j (counted
    // across items): S_j once K_j is loaded (and, at an item's first tile, its Q) and the
    // P V product of key tile j-2 is complete (P_j-2 lives in the buffer S_j overwrites);
    // O (+)= P_j V_j once P_j is written (and O rescaled).  A thread's tcgen05.mma issue
    // stalls while the products before it drain, so one thread issuing both kinds in
    // turn held each P V product back behind the score product issued before it; with two
    // issuers, P V starts as soon as P is ready.
    const bool s_side = warp == 3;
    int g = 0, on = 0;  // key tiles issued, items with work
    bool ok = true;
    for (int k = 0, idx = item_of(0); ok && idx < num_items; idx = item_of(++k)) {
      const FwdItem I = fwd_item(p, idx, lane);
      if (*s_abort) break;
      if (I.nvis == 0) continue;
      if (lane == 0) {
        const int qb = on & 1;
        if (s_side) {
          const TileDescs dQ_ = tile_descs<DP>(sbase + G::OFF_Q + qb * G::TILE_BYTES);
          ok = mbar_wait_spin(bar(F_QF0 + qb), (on >> 1) & 1, st, kFwdTimeout - 10);
          for (int t = 0; ok && t < I.nvis; ++t) {
            const int x = g + t;  // global key tile x into score buffer x % 2
            const int ks = x % G::KST;
            if (x >= 2 &&
                !mbar_wait_spin(bar(F_PD0 + (x & 1)), ((x - 2) >> 1) & 1, st, kFwdTimeout - 14)) {
              ok = false;
              break;
            }
            if (!mbar_wait_spin(bar(F_KF0 + ks), (x / G::KST) & 1, st, kFwdTimeout - 11)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const TileDescs dK_ = tile_descs<DP>(sbase + G::OFF_K + ks * G::TILE_BYTES);
            mma_kmajor<DP, F16>(tmem + FT_S0 + (x & 1) * 128, dQ_, dK_);
            mma_commit(bar(F_SF0 + (x & 1)));
            mma_commit(bar(F_KE0 + ks));
          }
          if (ok) mma_commit(bar(F_QE0 + qb));  // every S of the item has been issued
        } else {
          const uint32_t o_col = FT_O0 + qb * 128;
          for (int t = 0; ok && t < I.nvis; ++t) {
            const int x = g + t;
            if (!mbar_wait_spin(bar(F_PF0 + (x & 1)), (x >> 1) & 1, st, kFwdTimeout - 12)) { ok = false; break; }
            // the first product overwrites this O buffer: the item two back must have read it
            if (t == 0 && on >= 2 &&
                !mbar_wait_spin(bar(F_OE0 + qb), ((on - 2) >> 1) & 1, st, kFwdTimeout - 16)) {
              ok = false;
              break;
            }
            const int vs = x % G::VST;
            if (!mbar_wait_spin(bar(F_VF0 + vs), (x / G::VST) & 1, st, kFwdTimeout - 13)) { ok = false; break; }
            tc_fence_after();
            const TileDescs dV_ = tile_descs<DP>(sbase + G::OFF_V + vs * G::TILE_BYTES);
            mma_dv<DP, F16>(tmem + o_col, tmem + FT_S0 + (x & 1) * 128, dV_, t > 0 ? 1u : 0u);
            mma_commit(bar(F_VE0 + vs));
            mma_commit(bar(F_PD0 + (x & 1)));
          }
          if (ok) mma_commit(bar(F_ACC0 + qb));  // every P V: O of this item is final
        }
      }
      g += I.nvis;
      ++on;
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0 && g > 0) {
      // every product this thread issued is complete before the CTA releases tensor memory
      const uint32_t drain = bar(s_side ? F_DRAIN2 : F_DRAIN);
      mma_commit(drain);
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      mbar_wait(drain, 0, dr, kFwdTimeout - 15);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - 4) >> 2;        // key half of the score tile (columns 64 wg ..)
    const int qd = warp & 3;               // TMEM lane quadrant
    const int r = qd * 32 + lane;          // query row inside the tile = TMEM lane
    const int col0 = wg * 64;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const SoftmaxConsts kc{p.scale_log2, p.cap_scale, p.cap_log2};
    float* s_max = reinterpret_cast<float*>(smem_raw + FSM_MAX);
    float* s_l = reinterpret_cast<float*>(smem_raw + FSM_L);
    // O columns this warpgroup rescales and stores: 16-column chunks [c_lo, c_hi)
    constexpr int NCH = DP / 16;
    constexpr int NCH0 = (NCH + 1) / 2;
    const int c_lo = wg ? NCH0 : 0, c_hi = wg ? NCH : NCH0;
    // The two warps of a lane quadrant (one per warpgroup) meet at named barrier 2 + qd
    // once per key tile, and all eight softmax warps at named barrier 1 once per item.
    // A pair leaves the key-tile loop only on a decision taken at its own barrier, and
    // every warp reaches the item barrier (bar.red.or of the abort flag), so no warp is
    // ever left waiting at a barrier alone.
    int g = 0, on = 0, items = 0;  // key tiles consumed, items with work, items
    // Q buffer (1 + index) whose staged O this warp's tensor stores may still read; it is
    // handed back (O-staged barrier) at the next item's first key tile or epilogue
    int os_pend = 0;
    auto flush_os = [&]() {
      if (os_pend) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(F_OS0 + os_pend - 1));
        os_pend = 0;
      }
    };
    for (int k = 0, idx = item_of(0); idx < num_items; idx = item_of(++k), ++items) {
      const FwdItem I = fwd_item(p, idx, lane);
      const int m0 = I.m * kTileQ;
      const int i = m0 + r;
      const int qb = on & 1;
      const uint32_t o_col = FT_O0 + qb * 128;
      float mrow = kNegInf;  // running maximum (log2 units); moved only by more than 8
      float lrow = 0.f;      // running sum of this warpgroup's P relative to mrow
      int ncur = I.n_begin - 1;
      bool aborted = false;
      for (int t = 0; t < I.nvis; ++t) {
        const int x = g + t;
        const int n = ncur = fwd_next_tile(I, ncur);
        const int kb = n * kTileK;  // key index of column 0
        const bool need_mask = !tile_full(I.gm, I.m, n);
        // visible columns: lo <= key - i <= hi and key < Sk  <=>  c in [cmin, cmax]
        const int cmin = max(i + I.lo - kb, -1);
        const int cmax = min(min(i + I.hi - kb, I.Sk - 1 - kb), 1 << 20);
        const uint32_t sbuf = t_lane + FT_S0 + (x & 1) * 128 + col0;
        const bool ok = warp_wait(bar(F_SF0 + (x & 1)), (x >> 1) & 1, st, kFwdTimeout - 30);
        float xs[64];
        float mx = kNegInf;
        if (ok) {
          tc_fence_after();
          mx = need_mask ? fwd_scores<true, SOFTCAP>(kc, sbuf, col0, cmin, cmax, xs)
                         : fwd_scores<false, SOFTCAP>(kc, sbuf, col0, cmin, cmax, xs);
        }
        // the row maximum over both halves: only the two warps that own the same rows (one
        // per warpgroup, barrier 2 + quadrant) meet here; both always reach it, and after
        // it both see the abort flag that a failed wait of either one has raised
        s_max[((x & 1) * 2 + wg) * 128 + r] = mx;
        if (named_bar_or(2 + qd, 64, *s_abort != 0)) {
          aborted = true;
          break;
        }
        mx = fmaxf(mx, s_max[((x & 1) * 2 + (wg ^ 1)) * 128 + r]);
        // move the reference maximum only when a score passes it by more than 8 (log2);
        // both warpgroups take the same decision for a row
        float alpha = 1.f;
        if (t == 0) {
          mrow = mx;
        } else if (mx > mrow + 8.f) {
          alpha = ex2_approx(mrow - mx);  // mrow finite here, or -inf: alpha = 0
          mrow = mx;
        }
        const float muse = mrow == kNegInf ? 0.f : mrow;  // all-masked so far: P = 0
        lrow = lrow * alpha + fwd_probs<F16>(sbuf, SOFTCAP ? 1.f : kc.scale_log2, muse, xs);
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds this item's products up to key tile x-1: wait for the last one, then
          // rescale this warpgroup's columns (a failed wait ends the loop at the next barrier)
          if (!warp_wait(bar(F_PD0 + ((x - 1) & 1)), ((x - 1) >> 1) & 1, st, kFwdTimeout - 31)) continue;
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < NCH0; ++cc) {
            if (c_lo + cc < c_hi) {
              uint32_t o[16];
              tmem_ld16(t_lane + o_col + (c_lo + cc) * 16, o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st16(t_lane + o_col + (c_lo + cc) * 16, o);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(F_PF0 + (x & 1)));
        if (t == 0) flush_os();
      }

      // O = acc / l and LSE = (m + log2 l) * ln 2 with l the sum of both halves; a row with
      // no visible key gives O = 0 and LSE = +inf.  The O buffer is released to the item
      // two ahead as soon as it is in registers.
      const bool have = I.nvis > 0;
      bool acc_ok = !aborted;
      if (have && acc_ok) {
        acc_ok = warp_wait(bar(F_ACC0 + qb), (on >> 1) & 1, st, kFwdTimeout - 32);
        if (acc_ok) tc_fence_after();
      }
      const int lb = items & 1;  // row-sum exchange slot: alternates item by item
      s_l[(lb * 2 + wg) * 128 + r] = lrow;
      const bool stop = named_bar_or(1, 256, aborted || !acc_ok || *s_abort != 0);
      const float lsum = lrow + s_l[(lb * 2 + (wg ^ 1)) * 128 + r];
      const bool row_ok = i < I.Sq;
      const bool store = !stop && row_ok;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + (int64_t)I.tb * p.o_sb +
                       (int64_t)(I.q_off + i) * p.o_ss + (int64_t)I.h * p.o_sh;
      flush_os();
      // Warpgroup 0 writes O columns [0, 64), warpgroup 1 columns [64, Dp): each a 64-column
      // panel or the 16 / 32-column tail panel.  Staged in the item's Q buffer (free once
      // the item's products are done) in the tensor map's swizzled layout, a warp's 32 rows
      // leave with one tensor store; the map clips rows past Sq and columns past D.  A
      // packed sequence's last rows (the next sequence follows) are stored row by row.
      const bool tma = p.tma_epilogue != 0 && have && !stop &&
                       (!p.varlen || m0 + qd * 32 + 32 <= I.Sq);
      auto out_unit = [&](auto wc) {
        constexpr int W = decltype(wc)::value;
        constexpr int ROWB = 2 * W;
        constexpr int NCW = ROWB / 16;
        const int c0 = wg == 0 ? 0 : 64;
        const uint32_t box =
            sbase + G::OFF_Q + qb * G::TILE_BYTES + (wg == 0 ? qd * 4096 : 16384 + qd * 32 * ROWB);
        const uint32_t srow = box + (uint32_t)(lane * ROWB);
        const uint32_t sw = (uint32_t)((lane * ROWB) >> 7) & (uint32_t)(NCW - 1);
#pragma unroll
        for (int gq = 0; gq < W / 16; ++gq) {
          uint32_t o[16];
          if (have && !stop) {
            tmem_ld16(t_lane + o_col + c0 + gq * 16, o);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = 0u;
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pk[e] = pack_h2<F16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          const int c = c0 + gq * 16;
          if (tma) {
            st_shared_v4(srow + (((uint32_t)(2 * gq) ^ sw) << 4), pk[0], pk[1], pk[2], pk[3]);
            st_shared_v4(srow + (((uint32_t)(2 * gq + 1) ^ sw) << 4), pk[4], pk[5], pk[6], pk[7]);
          } else if (store) {
            if (c < p.D)
              *reinterpret_cast<uint4*>(orow + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (c + 8 < p.D)
              *reinterpret_cast<uint4*>(orow + c + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
        if (tma) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(wg == 0 ? &to : &to_t, c0, I.h, I.q_off + m0 + qd * 32, I.tb, box);
            bulk_commit();
          }
        }
      };
      if (wg == 0) {
        out_unit(IntC<64>{});
      } else {
        if constexpr (DP > 64) out_unit(IntC<DP - 64>{});
      }
      if (have && !stop) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(F_OE0 + qb));
        os_pend = qb + 1;  // the Q buffer goes back to the producer once the stores read it
      }
      if (store && wg == 0) {
        const float lse = lsum > 0.f ? (mrow + log2f(lsum)) * 0.69314718055994531f
                                     : __int_as_float(0x7f800000);
        p.lse[(int64_t)I.tb * p.lse_sb + (int64_t)I.h * p.lse_sh + (int64_t)(I.q_off + i) * p.lse_ss] = lse;
      }
      if (stop) break;
      if (have) {
        g += I.nvis;
        ++on;
      }
    }
    flush_os();
    // the last tensor stores complete before the CTA (and its shared memory) ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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
                           const OperandMaps& v, const OperandMaps& o, cudaStream_t s) {
  auto kern = fwd_tc_kernel<DP, SC, F16>;
  // at least 116 KB, so that one CTA (which allocates all 512 TMEM columns) runs per SM
  const size_t smem = GeoF<DP>::TOTAL > 118784u ? GeoF<DP>::TOTAL : 118784u;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)p.Mb * p.B * p.H;
  if (items > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  // persistent: at most one CTA per SM, each walking items blockIdx.x, + gridDim.x, ...
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  kern<<<grid, kFwdThreads, smem, s>>>(p, q.full, q.tail, k.full, k.tail, v.full, v.tail, o.full,
                                       o.tail);
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
                          const OperandMaps& v, const OperandMaps& o, int Dp, bool softcap,
                          bool f16, cudaStream_t s) {
  if (p.Mb <= 0 || p.B <= 0 || p.H <= 0) return cudaSuccess;
#define FA_FWD_TC_CASE(DPV)                                                             \
  case DPV:                                                                             \
    if (f16)                                                                            \
      return softcap ? launch_fwd_one<DPV, true, true>(p, q, k, v, o, s)                   \
                     : launch_fwd_one<DPV, false, true>(p, q, k, v, o, s);                 \
    return softcap ? launch_fwd_one<DPV, true, false>(p, q, k, v, o, s)                    \
                   : launch_fwd_one<DPV, false, false>(p, q, k, v, o, s);
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
