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
// The grid is persistent (at most one CTA per SM): CTAs take key tiles from a ticket
// counter in key-tile-major order, so under causal masking the longest tiles go first
// (in the ordered mode the highest key tile goes first: see decode_tile).
//
// Warp roles (16 warps, 512 threads):
//   warp 0      TMA producer: K, V per tile (the next tile's V, and at Dp = 96 / 128 its
//               K, prefetched into L2 while the current one finishes; at Dp <= 80 K has
//               two stages and the next tile's K is loaded at once); Q+LSE2+D and dO per
//               step (2-stage Q ring, one dO buffer)
//   warp 1      TMEM allocator and MMA issue (one elected lane issues)
//   warp 2      tile scheduler: claims the next ticket when the current tile starts its
//               last step and publishes it in a 2-slot ring
//   warp 3      ordered (deterministic) mode only: waits, one step ahead of the drain,
//               for each dQ tile's turn and hands it to the drain
//   warps 4-7   dQ drain (160 registers each via setmaxnreg): TMEM -> registers, release
//               the TMEM columns, then two 32 KB halves through a staging buffer into
//               cp.reduce.async.bulk fp32 adds (ordered by key tile when deterministic)
//   warps 8-15  two compute warpgroups: warpgroup w handles queries [64w, 64w+64) of
//               the tile for every key row (thread = key = TMEM lane); at the end of
//               each tile they stage dK / dV in shared memory, each warpgroup Dp of the
//               2 Dp columns, and tensor stores write them out
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0, Dp)        dK accumulator          [128, 128+Dp)  dV accumulator
//   [256, 384)     S^T; P^T (bf16 pairs) is written back over the columns already read
//   [384, 512)     dP^T; reused for the dQ tile once dS has been formed
//
// Shared memory (1024-byte aligned tiles, 128B swizzle for 64-column panels, 32B/64B
// swizzle for a 16/32-column tail panel when Dp % 64 != 0):
//   K (two stages at Dp <= 80), V, Q[2], dO (128 rows x Dp bf16 each), dS^T (128 keys x
//   128 queries bf16), dQ staging (128 x 64 fp32), dV staging (Dp < 128)
#include "fa_bwd_common.cuh"

namespace fa {

namespace {

template <int DP>
struct Geo : Panels<DP> {
  using Panels<DP>::TILE_BYTES;
  // shared-memory layout (offsets from a 1024-aligned base)
  static constexpr uint32_t SMALL = 3072;
  // K has two stages where they fit beside the dV staging (Dp <= 80): the next tile's K
  // then lands while the current tile's last products still read the other stage
  static constexpr int KST = DP <= 80 ? 2 : 1;
  static constexpr uint32_t OFF_K = SMALL;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;            // 2 stages
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * TILE_BYTES;       // 1 stage
  static constexpr uint32_t OFF_DS = OFF_DO + TILE_BYTES;
  static constexpr uint32_t DS_BYTES = 128u * 128u * 2u;
  static constexpr uint32_t OFF_STG = OFF_DS + DS_BYTES;           // dQ reduction staging
  static constexpr uint32_t STG_BYTES = 128u * 64u * 4u;           // 64 fp32 columns
  // dV staging for the tensor-copy epilogue where it fits (Dp < 128); at Dp = 128 dV is
  // staged after dK's last reader, in the dS buffer
  static constexpr uint32_t OFF_EPI = OFF_STG + STG_BYTES;
  static constexpr uint32_t EPI_BYTES = DP < 128 ? TILE_BYTES : 0;
  static constexpr uint32_t TOTAL = OFF_EPI + EPI_BYTES;
  static_assert(TOTAL <= 232448, "fits the 227 KB opt-in shared memory");
};

// ---------------------------------------------------------------- dK / dV epilogue units
// The accumulators leave tensor memory in units of (accumulator, column range) per warp:
// warpgroup 0 writes dV columns [0, 64) and dK columns [64, Dp), warpgroup 1 dK columns
// [0, 64) and dV columns [64, Dp), so that every unit is one 64-column operand panel or
// the 16 / 32-column tail panel and both warpgroups move Dp columns.  A unit of a warp's
// 32 key rows is rounded to the 16-bit type, written into a shared-memory box laid out
// like the operand panels (rows of 2W bytes, 128B / 64B / 32B swizzle for W = 64 / 32 /
// 16) and stored by lane 0 with one tensor copy; the tensor map clips rows past the key
// length and columns past the head dim.  Without a tensor map (or for a packed sequence's
// last rows, which the next sequence follows) the lanes store their rows directly.

template <int N>
struct IntC {
  static constexpr int value = N;
};

// W columns from this warp's 32 TMEM lanes, times sc, as 16-bit pairs in pk[0, W / 2)
// (zeros when the tile has no visible query).
template <int W, bool F16>
__device__ __forceinline__ void epi_load(uint32_t taddr, float sc, bool valid, uint32_t (&pk)[32]) {
  if constexpr (W == 16) {
    uint32_t r[16];
    if (valid) {
      tmem_ld16(taddr, r);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) r[e] = 0u;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
      pk[e] = pack_h2<F16>(__uint_as_float(r[2 * e]) * sc, __uint_as_float(r[2 * e + 1]) * sc);
  } else {
#pragma unroll
    for (int h = 0; h < W / 32; ++h) {
      uint32_t r[32];
      if (valid) {
        tmem_ld32(taddr + h * 32, r);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[h * 16 + e] =
            pack_h2<F16>(__uint_as_float(r[2 * e]) * sc, __uint_as_float(r[2 * e + 1]) * sc);
    }
  }
}

// Row `lane` of a W-column box at sbox (1024-byte aligned): 16-byte chunk c sits at
// chunk c ^ (address bits 7.. of the row) within the row, the tensor map's swizzle.
template <int W>
__device__ __forceinline__ void epi_stage(uint32_t sbox, int lane, const uint32_t (&pk)[32]) {
  constexpr int ROWB = 2 * W;
  constexpr int NCH = ROWB / 16;
  const uint32_t row = sbox + (uint32_t)(lane * ROWB);
  const uint32_t sw = (uint32_t)((lane * ROWB) >> 7) & (uint32_t)(NCH - 1);
#pragma unroll
  for (int c = 0; c < NCH; ++c)
    st_shared_v4(row + (((uint32_t)c ^ sw) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                 pk[4 * c + 3]);
}

// The direct form: this lane's row from column col0 on, the first ncols columns of it.
template <int W>
__device__ __forceinline__ void epi_store_row(__nv_bfloat16* row, int ncols,
                                              const uint32_t (&pk)[32]) {
#pragma unroll
  for (int g = 0; g < W / 8; ++g)
    if (g * 8 < ncols)
      *reinterpret_cast<uint4*>(row + g * 8) =
          make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
}

// One unit of the calling warp (tma, store: warp-uniform).  The box is reused only once
// the issuing lane's earlier copies have read their sources.
template <int W>
__device__ __forceinline__ void epi_put(const uint32_t (&pk)[32], bool tma, bool store,
                                        uint32_t box, int lane, const CUtensorMap* map,
                                        int col, int h, int row, int b, __nv_bfloat16* grow,
                                        bool row_ok, int ncols) {
  if (!store) return;
  if (tma) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    epi_stage<W>(box, lane, pk);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_4d(map, col, h, row, b, box);
      bulk_commit();
    }
  } else if (row_ok) {
    epi_store_row<W>(grow, ncols, pk);
  }
}

// Releases the accumulator's columns (after the calling warp's tensor-memory reads) to the
// next tile.
__device__ __forceinline__ void epi_release(bool valid, int lane, uint32_t bar) {
  if (valid) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  }
}

// A whole unit: load, release, store.
template <int W, bool F16>
__device__ __forceinline__ void epi_unit(uint32_t taddr, float sc, bool valid, uint32_t release,
                                         bool tma, bool store, uint32_t box, int lane,
                                         const CUtensorMap* map, int col, int h, int row, int b,
                                         __nv_bfloat16* grow, bool row_ok, int ncols) {
  uint32_t pk[32];
  epi_load<W, F16>(taddr, sc, valid, pk);
  epi_release(valid, lane, release);
  epi_put<W>(pk, tma, store, box, lane, map, col, h, row, b, grow, row_ok, ncols);
}

// small-region layout
constexpr uint32_t SM_BAR = 0;          // 32 barriers x 8 B
constexpr uint32_t SM_TMEM = 256;       // TMEM base address slot
constexpr uint32_t SM_ABORT = 260;
constexpr uint32_t SM_TILE = 264;       // drain scratch words
constexpr uint32_t SM_RING = 512;       // 2 tile descriptors x 32 B
constexpr uint32_t SM_VRING = 576;      // packed sequences: 2 sequence descriptors x 32 B
constexpr uint32_t SM_BAR2 = 640;       // mbarriers 32.. x 8 B
constexpr uint32_t SM_LSE = 1024;       // 2 stages x 128 fp32
constexpr uint32_t SM_DSUM = 2048;      // 2 stages x 128 fp32

enum Bar : int {
  B_K = 0, B_V, B_QF0, B_QF1, B_QE0, B_QE1, B_DOF0, B_DOF1, B_DOE0, B_DOE1,
  B_SFULL, B_DPFULL, B_PFULL, B_DSFULL, B_DVDONE, B_DQFULL, B_DQEMPTY, B_DSEMPTY,
  B_ACC, B_DRAIN, B_TILEF0, B_TILEF1, B_TILEE0, B_TILEE1, B_KEMPTY, B_VEMPTY, B_DVEMPTY,
  B_DKEMPTY, B_NEXT, B_TURN, B_TURNE, B_K1, B_KEMPTY1, B_COUNT
};
static_assert(B_COUNT <= 40, "barrier areas hold 32 + 8 mbarriers");

// Consumers of a published tile descriptor: producer, MMA issuer, 4 drain warps and 8
// compute warps each arrive once on the slot's empty barrier (and, in the ordered mode,
// the ordering warp).
constexpr int kTileConsumers = 14;

// One key tile of work as the scheduler publishes it in shared memory.
struct TileDesc {
  int valid, n, b, hk, m_begin, m_count, total, pad;
};

// With packed sequences, the tile's sequence: its first query / key row in the packed
// tensors, its lengths, its mask bounds (clamped to +-2^30, which keeps the predicate for
// lengths up to 2^30) and the slot of its first query tile (fa_tiles.h).
struct SeqDesc {
  int q_off, k_off, Sq, Sk, lo, hi;
  long long slot0;
};

__device__ __forceinline__ MaskGeom seq_geom(const SeqDesc& v) {
  MaskGeom g;
  g.Sq = v.Sq;
  g.Sk = v.Sk;
  g.lo = v.lo;
  g.hi = v.hi;
  g.tm = kTileQ;
  g.tn = kTileK;
  g.Mb = (v.Sq + kTileQ - 1) / kTileQ;
  g.Nb = (v.Sk + kTileK - 1) / kTileK;
  return g;
}

__device__ __forceinline__ int clamp_pm30(long long x) {
  const long long lim = 1ll << 30;
  return (int)(x < -lim ? -lim : (x > lim ? lim : x));
}

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
// Completion times (clock64 relative to the CTA's start) of the MMA groups of the first
// FA_TRACE_ITERS steps of the first FA_TRACE_CTAS CTAs, observed by the otherwise idle
// warp 3: S, dP, dV, dK, dQ.
__device__ long long g_fa_mma_done[FA_TRACE_CTAS][FA_TRACE_ITERS][5];
// Whole-kernel tile timeline (global timer, ns): per CTA and per tile it ran.
constexpr int FA_TL_CTAS = 160, FA_TL_TILES = 24, FA_TL_EV = 12;
__device__ long long g_fa_tl[FA_TL_CTAS][FA_TL_TILES][FA_TL_EV];
__device__ __forceinline__ long long gtimer() {
  long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
#define FA_TL(t, ev, val)                                                          \
  do {                                                                             \
    if (blockIdx.x < FA_TL_CTAS && (t) < FA_TL_TILES)                              \
      g_fa_tl[blockIdx.x][(t)][(ev)] = (val);                                      \
  } while (0)
#else
#define FA_TL(t, ev, val) \
  do {                    \
  } while (0)
#define FA_TR(ev, it) \
  do {                \
  } while (0)
#endif

struct TileCoord {
  int n, b, hk;
};

__device__ __forceinline__ TileCoord decode_tile(const BwdMainParams& p, int t) {
  // Key-tile-major order.  Normally all (b, hk) of key tile 0 come first: under causal
  // masking the low key tiles see the most query tiles, so the longest work starts first.
  // In the ordered (deterministic) mode the last key tile comes first instead: the dQ
  // contributions to a query tile are added from the highest key tile down, which is the
  // order in which a key-tile-major sweep reaches them (key tile n + 1 reaches query tile
  // m one step before key tile n), and every tile a CTA waits for was claimed earlier,
  // by a CTA that is running or done.
  TileCoord c;
  const int per_n = p.B * p.Hk;
  const int n0 = t / per_n;
  const int r = t - n0 * per_n;
  c.n = p.deterministic ? p.Nb - 1 - n0 : n0;
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
template <bool MASK, bool SOFTCAP, bool F16>
__device__ __forceinline__ void phase_p(const SoftmaxConsts& kc, uint32_t taddr, const float* lse,
                                        const float (&lreg)[2], int qmin, int qmax, uint32_t (&pc)[32]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    uint32_t pk[16];
#pragma unroll
    for (int v4 = 0; v4 < 8; ++v4) {
      float lv[4];
      if (SOFTCAP) {
        const float4 l4 = reinterpret_cast<const float4*>(lse + c * 32)[v4];
        lv[0] = l4.x;
        lv[1] = l4.y;
        lv[2] = l4.z;
        lv[3] = l4.w;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) lv[u] = __shfl_sync(0xffffffffu, lreg[c], v4 * 4 + u);
      }
      float pv[4], pcv[4];
      if (SOFTCAP) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float fac;
          pv[u] = prob<SOFTCAP>(kc, __uint_as_float(r[v4 * 4 + u]), lv[u], &fac);
          pcv[u] = pv[u] * fac;
        }
      } else {
        // exp2(S * scale * log2e - LSE2), two columns per paired fused multiply-add
        const uint64_t sl2 = f2_pack(kc.scale_log2, kc.scale_log2);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
          const uint64_t t = f2_fma(f2_pack(__uint_as_float(r[v4 * 4 + u]), __uint_as_float(r[v4 * 4 + u + 1])),
                                    sl2, f2_pack(-lv[u], -lv[u + 1]));
          pv[u] = ex2_approx(f2_lo(t));
          pv[u + 1] = ex2_approx(f2_hi(t));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ql = c * 32 + v4 * 4 + u;
        if (MASK) {
          pv[u] = (ql >= qmin && ql <= qmax) ? pv[u] : 0.f;
          if (SOFTCAP) pcv[u] = (ql >= qmin && ql <= qmax) ? pcv[u] : 0.f;
        }
        if (!SOFTCAP) pcv[u] = pv[u];
      }
      pk[v4 * 2] = pack_h2<F16>(pv[0], pv[1]);
      pk[v4 * 2 + 1] = pack_h2<F16>(pv[2], pv[3]);
      pc[c * 16 + v4 * 2] = pack_f16(pcv[0], pcv[1]);
      pc[c * 16 + v4 * 2 + 1] = pack_f16(pcv[2], pcv[3]);
    }
    tmem_st16(taddr + c * 16, pk);
  }
}

// The five contractions as issued by the single MMA thread (S^T, dP^T and dV use the
// tile-descriptor helpers of fa_bwd_common.cuh).

// dK (+)= dS^T Q: A = dS^T (K-major, 128B swizzle, `ds` = its descriptor), B = Q (N = Dp,
// MN-major), K = 128 queries.
template <int DP, bool F16>
__device__ __forceinline__ void mma_dk(uint32_t d, DescWords ds, const TileDescs& B, uint32_t acc) {
  using P = Panels<DP>;
  constexpr uint32_t ID = idesc_h<F16>(128, P::NFULL * 64, false, true);
  constexpr uint32_t ID_T = idesc_h<F16>(128, P::TAIL ? P::TAIL : 16, false, true);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t a_off = (ks >> 2) * 1024 + (ks & 3) * 2;
    if (ks == 0) {
      mma_ss_wp(d, ds, a_off, B.mfull, 0, ID, acc);
      if (P::TAIL) mma_ss_wp(d + P::NFULL * 64, ds, a_off, B.mtail, 0, ID_T, acc);
    } else {
      mma_ss_w<1>(d, ds, a_off, B.mfull, ks * 128, ID);
      if (P::TAIL) mma_ss_w<1>(d + P::NFULL * 64, ds, a_off, B.mtail, ks * P::TAIL_ROWB, ID_T);
    }
  }
}

// dQ tile = dS K: A = dS (M = queries, MN-major view of the dS^T tile, `ds` = its
// descriptor), B = K (N = Dp, MN-major), K = 128 keys.
template <int DP, bool F16>
__device__ __forceinline__ void mma_dq(uint32_t d, DescWords ds, const TileDescs& B) {
  using P = Panels<DP>;
  constexpr uint32_t ID = idesc_h<F16>(128, P::NFULL * 64, true, true);
  constexpr uint32_t ID_T = idesc_h<F16>(128, P::TAIL ? P::TAIL : 16, true, true);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    if (ks == 0) {
      mma_ss_w<0>(d, ds, 0, B.mfull, 0, ID);
      if (P::TAIL) mma_ss_w<0>(d + P::NFULL * 64, ds, 0, B.mtail, 0, ID_T);
    } else {
      mma_ss_w<1>(d, ds, ks * 128, B.mfull, ks * 128, ID);
      if (P::TAIL) mma_ss_w<1>(d + P::NFULL * 64, ds, ks * 128, B.mtail, ks * P::TAIL_ROWB, ID_T);
    }
  }
}

// F16: the operands, P^T / dS and the dK / dV outputs are f16 (else bf16).
// MODE 1 (VARLEN): packed sequences (per-sequence offsets, lengths and mask bounds from
// cu_q / cu_k; tiles indexed by slot).  MODE 2 (SPARSE): block-sparse, a key tile's steps
// come from its precomputed list instead of the whole (q-head, query tile) range.  The
// batched dense instantiations (MODE 0) are unchanged by either.
template <int DP, bool SOFTCAP, bool F16, int MODE>
__global__ void __launch_bounds__(512, 1)
    bwd_main_kernel(const __grid_constant__ BwdMainParams p,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tq_t,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk_t,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tv_t,
                    const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdo_t,
                    const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdk_t,
                    const __grid_constant__ CUtensorMap tdv,
                    const __grid_constant__ CUtensorMap tdv_t) {
  using G = Geo<DP>;
  constexpr bool VARLEN = MODE == 1;
  constexpr bool SPARSE = MODE == 2;
#ifdef FA_TRACE
  const long long t_start = clock64();
#endif
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* small = smem_raw;
  volatile int* s_abort = reinterpret_cast<volatile int*>(small + SM_ABORT);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(small + SM_TMEM);
  const float* s_lse = reinterpret_cast<const float*>(small + SM_LSE);
  const float* s_dsum = reinterpret_cast<const float*>(small + SM_DSUM);
  auto bar = [&](int i) -> uint32_t {
    return sbase + (i < 32 ? SM_BAR + 8u * i : SM_BAR2 + 8u * (i - 32));
  };

#ifdef FA_TRACE
  if (threadIdx.x == 0) {
    FA_TL(FA_TL_TILES - 1, 0, gtimer());
    FA_TL(FA_TL_TILES - 1, 1, clock64());
  }
#endif
  if (threadIdx.x == 0) {
    *s_abort = 0;
    if ((sbase & 1023u) != 0) {
      // the tile layout assumes a 1024-byte aligned dynamic shared-memory base
      atomicExch(p.status, kTimeoutBase - 99);
      *s_abort = 1;
    }
    mbar_init(bar(B_K), 1);
    mbar_init(bar(B_K1), 1);
    mbar_init(bar(B_V), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QF0 + s), 1);
      mbar_init(bar(B_QE0 + s), 1);
      mbar_init(bar(B_DOF0 + s), 1);
      mbar_init(bar(B_DOE0 + s), 1);
      mbar_init(bar(B_TILEF0 + s), 1);
      mbar_init(bar(B_TILEE0 + s), kTileConsumers + (p.deterministic ? 1 : 0));
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
    mbar_init(bar(B_KEMPTY), 1);
    mbar_init(bar(B_KEMPTY1), 1);
    mbar_init(bar(B_VEMPTY), 1);
    mbar_init(bar(B_DVEMPTY), 8);
    mbar_init(bar(B_DKEMPTY), 8);
    mbar_init(bar(B_NEXT), 1);
    mbar_init(bar(B_TURN), 1);
    mbar_init(bar(B_TURNE), 1);
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
  SeqDesc* vring = reinterpret_cast<SeqDesc*>(small + SM_VRING);
  auto read_tile = [&](int t, TileDesc& d) -> bool {
    const bool ok = mbar_wait(bar(B_TILEF0 + (t & 1)), (t >> 1) & 1, st, kTimeoutBase - 40);
    if (ok) d = ring[t & 1];
    return ok && d.valid;
  };
  auto read_tile_ool = [&](int t, TileDesc& d) -> bool {
    const bool ok = mbar_wait_ool(bar(B_TILEF0 + (t & 1)), (t >> 1) & 1, st, kTimeoutBase - 40);
    if (ok) d = ring[t & 1];
    return ok && d.valid;
  };

  // Register split (launch: 512 threads x 128 = 65536): the producer / MMA warpgroup
  // gives registers to the dQ drain warpgroup, which keeps a whole dQ row in registers.
  // 128 * (96 + 160 + 128 + 128) = 65536; the host refuses to launch unless the kernel
  // was compiled to exactly 128 registers per thread, so the split always fits.
  if (warp < 4) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
#ifdef FA_TRACE
   if (warp == 3 && lane == 0 && blockIdx.x < FA_TRACE_CTAS && !p.deterministic) {
     // observer: poll the completion barriers in order of their phases
     const int bars[5] = {B_SFULL, B_DPFULL, B_DVDONE, -1, B_DQFULL};
     int k[5] = {0, 0, 0, 0, 0};
     const long long t_lim = clock64() + 400000000ll;
     while (clock64() < t_lim && !*s_abort) {
       bool all = true;
#pragma unroll
       for (int e = 0; e < 5; ++e) {
         if (k[e] >= FA_TRACE_ITERS) continue;
         all = false;
         const uint32_t b = e == 3 ? bar(B_QE0 + (k[e] & 1)) : bar(bars[e]);
         const uint32_t par = e == 3 ? ((k[e] >> 1) & 1) : (k[e] & 1);
         if (mbar_test_wait(b, par)) {
           g_fa_mma_done[blockIdx.x][k[e]][e] = clock64() - t_start;
           ++k[e];
         }
       }
       if (all) break;
     }
   }
#endif
   if (warp == 2) {
    // ------------------------------------------------------------------ tile scheduler
    if (lane == 0) {
      for (int t = 0;; ++t) {
        const int k = t & 1;
        // Claim the next tile only when the current one is about to run out of work (the
        // producer starts its last step), so that tiles stay in longest-first order across
        // CTAs instead of being claimed a whole tile ahead.
        const bool ready =
            (t == 0 || mbar_wait_ool(bar(B_NEXT), (t - 1) & 1, st, kTimeoutBase - 42)) &&
            (t < 2 || mbar_wait_ool(bar(B_TILEE0 + k), ((t - 2) >> 1) & 1, st, kTimeoutBase - 41));
        if (!ready) {
          ring[k].valid = 0;
          mbar_arrive(bar(B_TILEF0 + k));
          break;
        }
        // The first tile is blockIdx.x (the grid never exceeds the tile count); later ones
        // come from the ticket counter, which the preprocess clears, so the first claim
        // waits for that grid (a no-op unless this kernel was launched as its dependent).
        int ticket;
        if (*s_abort) {
          ticket = p.num_tiles;
        } else if (t == 0) {
          ticket = (int)blockIdx.x;
          if constexpr (SPARSE) pdl_wait_prior();  // the step lists come from the grid before
        } else {
          if (t == 1) pdl_wait_prior();
          ticket = (int)gridDim.x + atomicAdd(p.ticket, 1);
        }
        FA_TL(t, 0, ticket);
        FA_TL(t, 1, gtimer());
        TileDesc d{};
        d.valid = ticket < p.num_tiles;
        if (d.valid) {
          const TileCoord c = decode_tile(p, ticket);
          int64_t mb64, me64;
          if constexpr (VARLEN) {
            int64_t q0, sq, k0, sk;
            seq_rows(p.cu_q, p.used_q, c.b, p.total_q, &q0, &sq);
            seq_rows(p.cu_k, p.used_k, c.b, p.total_k, &k0, &sk);
            const MaskGeom g = make_geom(sq, sk, p.causal, p.window_left, p.window_right, kTileQ, kTileK);
            m_range(g, c.n, &mb64, &me64);
            SeqDesc v;
            v.q_off = (int)q0;
            v.k_off = (int)k0;
            v.Sq = (int)sq;
            v.Sk = (int)sk;
            v.lo = clamp_pm30(g.lo);
            v.hi = clamp_pm30(g.hi);
            v.slot0 = first_slot(p.cu_q, c.b, p.total_q);
            vring[k] = v;
          } else {
            m_range(gm, c.n, &mb64, &me64);
          }
          d.n = c.n;
          d.b = c.b;
          d.hk = c.hk;
          d.m_begin = (int)mb64;
          d.m_count = (int)(me64 - mb64);
          d.total = d.m_count * p.G;  // steps (g, m), m fastest
          if constexpr (SPARSE) {
            d.total = p.sp_counts[ticket];  // the kept steps, listed in the same order
            d.pad = ticket;
          }
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
      int git = 0, nk = 0, nv = 0, ndo = 0;
      bool alive = true;
      for (int t = 0; alive; ++t) {
        TileDesc d;
        if (!read_tile_ool(t, d)) break;
        // map coordinates: batch, first query row, first key row (packed: 0, offsets)
        int tb = d.b, q_off = 0, k_off = 0;
        long long slot0 = 0;
        if constexpr (VARLEN) {
          const SeqDesc v = vring[t & 1];
          tb = 0;
          q_off = v.q_off;
          k_off = v.k_off;
          slot0 = v.slot0;
        }
        mbar_arrive(bar(B_TILEE0 + (t & 1)));
        if (d.total == 0) {
          mbar_arrive(bar(B_NEXT));
          continue;
        }
        const int n0 = k_off + d.n * kTileK;
        auto load_k = [&]() {
          const int ks = G::KST == 2 ? (nk & 1) : 0;
          const uint32_t kb = bar(ks ? B_K1 : B_K);
          const uint32_t kdst = sbase + G::OFF_K + ks * G::TILE_BYTES;
          ++nk;
          mbar_arrive_expect_tx(kb, G::TILE_BYTES);
          _Pragma("unroll 1") for (int pnl = 0; pnl < G::NFULL; ++pnl)
            tma_load_4d(kdst + pnl * G::FULL_BYTES, &tk, pnl * 64, d.hk, n0, tb, kb);
          if (G::TAIL) tma_load_4d(kdst + G::TAIL_OFF, &tk_t, G::NFULL * 64, d.hk, n0, tb, kb);
        };
        auto load_v = [&]() {
          ++nv;
          mbar_arrive_expect_tx(bar(B_V), G::TILE_BYTES);
          _Pragma("unroll 1") for (int pnl = 0; pnl < G::NFULL; ++pnl)
            tma_load_4d(sbase + G::OFF_V + pnl * G::FULL_BYTES, &tv, pnl * 64, d.hk, n0, tb, bar(B_V));
          if (G::TAIL) tma_load_4d(sbase + G::OFF_V + G::TAIL_OFF, &tv_t, G::NFULL * 64, d.hk, n0, tb, bar(B_V));
        };
        const bool kv_busy = nk > 0;  // the previous tile may still be reading K and V
        if (G::KST == 2 && kv_busy) {
          // the stage this K goes to was last read two tiles back
          if (nk >= 2 && !mbar_wait_ool(bar((nk & 1) ? B_KEMPTY1 : B_KEMPTY), ((nk >> 1) - 1) & 1,
                                        st, kTimeoutBase - 5))
            break;
          load_k();
        }
        if (kv_busy) {
          // warm L2 with this tile's K and V so that the loads below, which must wait for
          // the previous tile's last MMAs, hit L2
          _Pragma("unroll 1") for (int pnl = 0; pnl < G::NFULL; ++pnl) {
            if (G::KST == 1) tma_prefetch_4d(&tk, pnl * 64, d.hk, n0, tb);
            tma_prefetch_4d(&tv, pnl * 64, d.hk, n0, tb);
          }
          if (G::TAIL) {
            if (G::KST == 1) tma_prefetch_4d(&tk_t, G::NFULL * 64, d.hk, n0, tb);
            tma_prefetch_4d(&tv_t, G::NFULL * 64, d.hk, n0, tb);
          }
        } else {
          load_k();
          load_v();
        }
        // After the first tile, the loads of a tile's first step go out in the order their
        // buffers are released by the previous tile: Q (its dK two steps back), V (its last
        // dP), dO (its last dV), K (its last dQ).
        for (int it = 0; it < d.total; ++it, ++git) {
          const int s = git & 1;
          int g = it / d.m_count;
          int m = d.m_begin + (it - g * d.m_count);
          if constexpr (SPARSE) {
            const int e = p.sp_lists[(size_t)d.pad * p.sp_stride + it];
            g = e >> 16;
            m = e & 0xffff;
          }
          const int h = d.hk * p.G + g;
          const int m0 = m * kTileQ;
          if (it == d.total - 1) mbar_arrive(bar(B_NEXT));  // time to claim the next tile
          if (git >= 2 && !mbar_wait_ool(bar(B_QE0 + s), ((git - 2) >> 1) & 1, st, kTimeoutBase - 1)) {
            alive = false;
            break;
          }
          const uint32_t qdst = sbase + G::OFF_Q + s * G::TILE_BYTES;
          mbar_arrive_expect_tx(bar(B_QF0 + s), G::TILE_BYTES + 2 * 512);
          _Pragma("unroll 1") for (int pnl = 0; pnl < G::NFULL; ++pnl)
            tma_load_4d(qdst + pnl * G::FULL_BYTES, &tq, pnl * 64, h, q_off + m0, tb, bar(B_QF0 + s));
          if (G::TAIL) tma_load_4d(qdst + G::TAIL_OFF, &tq_t, G::NFULL * 64, h, q_off + m0, tb, bar(B_QF0 + s));
          size_t row = ((size_t)d.b * p.H + h) * p.Sq_r + m0;
          if constexpr (VARLEN) row = ((size_t)h * p.T + slot0 + m) * kTileQ;
          if (git == 0) pdl_wait_prior();  // LSE2 and D come from the preprocess
          bulk_load(sbase + SM_LSE + s * 512, p.lse2 + row, 512, bar(B_QF0 + s));
          bulk_load(sbase + SM_DSUM + s * 512, p.dsum + row, 512, bar(B_QF0 + s));
          FA_TR(10, git);
          if (it == 0 && kv_busy) {
            if (!mbar_wait_ool(bar(B_VEMPTY), (nv - 1) & 1, st, kTimeoutBase - 4)) {
              ++git;
              alive = false;
              break;
            }
            load_v();
          }
          // dO has one buffer: dO_i+1 may land once dV_i (its last reader) is complete
          if (git >= 1 && !mbar_wait_ool(bar(B_DOE0), (git - 1) & 1, st, kTimeoutBase - 2)) {
            ++git;
            alive = false;
            break;
          }
          ++ndo;
          const uint32_t ddst = sbase + G::OFF_DO;
          mbar_arrive_expect_tx(bar(B_DOF0), G::TILE_BYTES);
          _Pragma("unroll 1") for (int pnl = 0; pnl < G::NFULL; ++pnl)
            tma_load_4d(ddst + pnl * G::FULL_BYTES, &tdo, pnl * 64, h, q_off + m0, tb, bar(B_DOF0));
          if (G::TAIL) tma_load_4d(ddst + G::TAIL_OFF, &tdo_t, G::NFULL * 64, h, q_off + m0, tb, bar(B_DOF0));
          if (G::KST == 1 && it == 0 && kv_busy) {
            if (!mbar_wait_ool(bar(B_KEMPTY), (nk - 1) & 1, st, kTimeoutBase - 5)) {
              ++git;
              alive = false;
              break;
            }
            FA_TL(t, 8, gtimer());
            load_k();
          }
        }
      }
      // Before the CTA may exit, every copy this thread started must have landed (on an
      // abort the consumers may not have waited for them).  Only the latest phase of each
      // barrier can still be pending.
      volatile int no_abort = 0;
      AbortState dr{&no_abort, p.status, p.wait_limit};
      if (G::KST == 1) {
        if (nk > 0) mbar_wait_ool(bar(B_K), (nk - 1) & 1, dr, kTimeoutBase - 3);
      } else {
        for (int ks = 0; ks < 2; ++ks) {
          const int nks = (nk - ks + 1) / 2;  // loads issued into K stage ks
          if (nks > 0) mbar_wait_ool(bar(ks ? B_K1 : B_K), (nks - 1) & 1, dr, kTimeoutBase - 3);
        }
      }
      if (nv > 0) mbar_wait_ool(bar(B_V), (nv - 1) & 1, dr, kTimeoutBase - 3);
      for (int s = 0; s < 2; ++s) {
        const int nq = (git - s + 1) / 2;  // loads issued into Q stage s
        if (nq > 0) mbar_wait_ool(bar(B_QF0 + s), (nq - 1) & 1, dr, kTimeoutBase - 3);
      }
      if (ndo > 0) mbar_wait_ool(bar(B_DOF0), (ndo - 1) & 1, dr, kTimeoutBase - 3);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Per tile: S_0, dP_0 (after the previous tile's last dV and drained dQ), then per step i:
    //   dV_i  (needs P^T_i; the first one of a tile also needs the previous tile's dK/dV
    //         read out)                                 -> frees the dO buffer, dv_done
    //   S_i+1 (needs dv_done_i: P^T_i aliases the S^T columns) -- overlaps phase B_i
    //   dK_i, dQ_i (need dS_i)                          -> dq_full
    //   dP_i+1 (needs the dQ_i columns drained)
    // The whole warp runs this code (its values are warp-uniform, so the descriptor
    // arithmetic stays on the uniform datapath); one elected lane issues the MMAs and
    // commits, and every wait is agreed on by the warp.
    {
      const bool leader = elect_one();
      auto wspin = [&](uint32_t b, uint32_t par, int code) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_spin(b, par, st, code));
      };
      const TileDescs dK0 = tile_descs<DP>(sbase + G::OFF_K), dV_ = tile_descs<DP>(sbase + G::OFF_V);
      const TileDescs dK1 = tile_descs<DP>(sbase + G::OFF_K + (G::KST - 1) * G::TILE_BYTES);
      int kst = 0;  // K stage of the current tile
      const TileDescs dDO = tile_descs<DP>(sbase + G::OFF_DO);
      const TileDescs dQ0 = tile_descs<DP>(sbase + G::OFF_Q), dQ1 = tile_descs<DP>(sbase + G::OFF_Q + G::TILE_BYTES);
      const DescWords dsK = desc_words(sbase + G::OFF_DS, 16, 1024, SWZ_128B);      // dS^T, K-major
      const DescWords dsM = desc_words(sbase + G::OFF_DS, 16384, 1024, SWZ_128B);   // dS, MN-major
      auto issue_S = [&](int g) -> bool {
        const int s = g & 1;
        if (!wspin(bar(B_QF0 + s), (g >> 1) & 1, kTimeoutBase - 11)) return false;
        tc_fence_after();
        if (leader) FA_TR(0, g);
        if (leader) mma_kmajor<DP, F16>(tmem + TM_S, kst ? dK1 : dK0, s ? dQ1 : dQ0);
        if (leader) mma_commit(bar(B_SFULL));
        return true;
      };
      auto issue_dP = [&](int g) -> bool {
        if (!wspin(bar(B_DOF0), g & 1, kTimeoutBase - 13)) return false;
        tc_fence_after();
        if (leader) FA_TR(1, g);
        if (leader) mma_kmajor<DP, F16>(tmem + TM_DP, dV_, dDO);
        if (leader) mma_commit(bar(B_DPFULL));
        return true;
      };
      int git = 0, kt = 0;
      bool ok = true;
      for (int t = 0; ok; ++t) {
        TileDesc d;
        if (!__all_sync(0xffffffffu, read_tile_ool(t, d))) break;
        if (leader) mbar_arrive(bar(B_TILEE0 + (t & 1)));
        if (d.total == 0) continue;
        // the previous tile's last P^T and dQ columns must be consumed before S_0 / dP_0
        if (git > 0 && !wspin(bar(B_DVDONE), (git - 1) & 1, kTimeoutBase - 12)) break;
        kst = G::KST == 2 ? (kt & 1) : 0;
        if (!wspin(bar(kst ? B_K1 : B_K), (G::KST == 2 ? kt >> 1 : kt) & 1, kTimeoutBase - 10)) break;
        if (leader) FA_TL(t, 2, gtimer());
        if (leader) FA_TL(t, 7, d.total);
        if (!issue_S(git)) break;
        if (git > 0 && !wspin(bar(B_DQEMPTY), (git - 1) & 1, kTimeoutBase - 14)) break;
        if (!wspin(bar(B_V), kt & 1, kTimeoutBase - 19)) break;
        if (!issue_dP(git)) break;
        if (d.total == 1) if (leader) mma_commit(bar(B_VEMPTY));  // V's last reader is the tile's last dP
        uint32_t acc = 0;
        for (int it = 0; it < d.total; ++it, ++git) {
          const int s = git & 1;
          // dV += P^T dO : A = P^T from TMEM (bf16 pairs), K = 128 queries in 8 steps
          if (!wspin(bar(B_PFULL), git & 1, kTimeoutBase - 15)) { ok = false; break; }
          // the accumulators are overwritten by this tile's first dV / dK: the previous
          // tile's epilogue must have read them
          if (it == 0 && kt > 0 &&
              !wspin(bar(B_DVEMPTY), (kt - 1) & 1, kTimeoutBase - 18)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) FA_TR(2, git);
          if (it == 0) if (leader) FA_TL(t, 3, gtimer());
          if (leader) mma_dv<DP, F16>(tmem + TM_DV, tmem + TM_S, dDO, acc);
          if (leader) mma_commit(bar(B_DOE0));
          if (leader) mma_commit(bar(B_DVDONE));
          if (it + 1 < d.total) {
            if (!wspin(bar(B_DVDONE), git & 1, kTimeoutBase - 12)) { ok = false; break; }
            if (!issue_S(git + 1)) { ok = false; break; }
          }
          // dK += dS^T Q : A = dS^T (K-major in shared memory), K = 128 queries
          if (!wspin(bar(B_DSFULL), git & 1, kTimeoutBase - 16)) { ok = false; break; }
          if (it == 0 && kt > 0 &&
              !wspin(bar(B_DKEMPTY), (kt - 1) & 1, kTimeoutBase - 18)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) FA_TR(3, git);
          if (leader) mma_dk<DP, F16>(tmem + TM_DK, dsK, s ? dQ1 : dQ0, acc);
          if (leader) mma_commit(bar(B_QE0 + s));
          if (leader) mma_dq<DP, F16>(tmem + TM_DP, dsM, kst ? dK1 : dK0);  // the dQ tile goes where dP^T was
          if (leader) mma_commit(bar(B_DQFULL));
          if (leader) mma_commit(bar(B_DSEMPTY));
          acc = 1;
          if (it + 1 < d.total) {
            if (!wspin(bar(B_DQEMPTY), git & 1, kTimeoutBase - 14)) { ok = false; break; }
            if (!issue_dP(git + 1)) { ok = false; break; }
            if (it + 2 == d.total) if (leader) mma_commit(bar(B_VEMPTY));
          }
        }
        if (!ok) break;
        if (leader) FA_TL(t, 4, gtimer());
        if (leader) mma_commit(bar(B_ACC));     // this tile's dK / dV are final
        if (leader) mma_commit(bar(kst ? B_KEMPTY1 : B_KEMPTY));  // and its K stage may be refilled
        ++kt;
      }
      if (git > 0 || kt > 0) {
        // every MMA must be complete before the CTA releases tensor memory
        if (leader) mma_commit(bar(B_DRAIN));
        volatile int no_abort = 0;
        AbortState dr{&no_abort, p.status, p.wait_limit};
        mbar_wait_ool(bar(B_DRAIN), 0, dr, kTimeoutBase - 17);
      }
    }
   } else if (warp == 3) {
    // ------------------------------------------------------------------ ordering warp
    // Ordered mode only.  One step ahead of the drain, lane 0 waits (bounded) until the
    // step's dQ tile holds the contributions of every higher key tile (its counter equals
    // this key tile's rank from the top), then hands the outcome to the drain (turn
    // barrier) and waits until the drain has taken it (turn-empty barrier) before the next
    // step.  The drain's TMEM read, which frees the dQ columns for the next dP product,
    // never waits on this global-memory round trip.
    if constexpr (!SPARSE) {
     if (p.deterministic) {
      if (lane == 0) pdl_wait_prior();  // the counters are cleared by the preprocess
      volatile int* s_turn = reinterpret_cast<volatile int*>(small + SM_TILE + 8);
      int git = 0;
      bool alive = true;
      for (int t = 0; alive; ++t) {
        TileDesc d;
        const bool have_tile = __all_sync(0xffffffffu, read_tile(t, d));
        SeqDesc vd{};
        if constexpr (VARLEN) {
          if (have_tile) vd = vring[t & 1];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_TILEE0 + (t & 1)));
        if (!have_tile) break;
        if (lane == 0) {
          for (int it = 0; it < d.total; ++it, ++git) {
            const int g = it / d.m_count;
            const int m = d.m_begin + (it - g * d.m_count);
            const int h = d.hk * p.G + g;
            size_t tile_id = ((size_t)d.b * p.H + h) * p.Mb + m;
            if constexpr (VARLEN) tile_id = (size_t)h * p.T + vd.slot0 + m;
            const int* sem = p.sems + tile_id;
            if (git > 0 &&
                !mbar_wait_ool(bar(B_TURNE), (git - 1) & 1, st, kTimeoutBase - 22)) {
              alive = false;
              break;
            }
            int64_t nb, ne;
            if constexpr (VARLEN)
              n_range(seq_geom(vd), m, &nb, &ne);
            else
              n_range(gm, m, &nb, &ne);
            const int want = (int)ne - 1 - d.n;  // rank from the highest key tile down
            int stop = 0;
            const long long t0 = clock64();
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
            s_turn[git & 1] = stop;
            mbar_arrive(bar(B_TURN));  // release: the drain that sees the phase sees s_turn
            if (stop) {
              alive = false;
              break;
            }
          }
        }
        alive = __shfl_sync(0xffffffffu, alive, 0);
      }
     }
    } else {
     // Block-sparse steps: the contributors of a query tile are the key tiles in its
     // element-mask range that the block mask keeps, and this key tile's rank is the
     // number of kept ones above it (counted by the whole warp with a ballot sum; the
     // list builder and the scheduler give key tiles out highest first, as above).
     if (p.deterministic) {
      if (lane == 0) pdl_wait_prior();  // the counters are cleared by the preprocess
      volatile int* s_turn = reinterpret_cast<volatile int*>(small + SM_TILE + 8);
      int git = 0;
      bool alive = true;
      for (int t = 0; alive; ++t) {
        TileDesc d;
        const bool have_tile = __all_sync(0xffffffffu, read_tile(t, d));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_TILEE0 + (t & 1)));
        if (!have_tile) break;
        for (int it = 0; alive && it < d.total; ++it, ++git) {
          const int e = p.sp_lists[(size_t)d.pad * p.sp_stride + it];
          const int g = e >> 16;
          const int m = e & 0xffff;
          const int h = d.hk * p.G + g;
          const size_t tile_id = ((size_t)d.b * p.H + h) * p.Mb + m;
          int64_t nb, ne;
          n_range(gm, m, &nb, &ne);
          const uint8_t* brow = p.block_mask + tile_id * (size_t)p.Nb;
          int cnt = 0;
          for (int n2 = d.n + 1 + lane; n2 < (int)ne; n2 += 32) cnt += brow[n2] != 0;
          const int want = __reduce_add_sync(0xffffffffu, cnt);
          int stop = 0;
          if (lane == 0) {
            const int* sem = p.sems + tile_id;
            if (git > 0 && !mbar_wait_ool(bar(B_TURNE), (git - 1) & 1, st, kTimeoutBase - 22)) {
              stop = 2;  // the drain is gone: no turn to hand over
            } else {
              const long long t0 = clock64();
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
              s_turn[git & 1] = stop;
              mbar_arrive(bar(B_TURN));  // release: the drain that sees the phase sees s_turn
            }
          }
          stop = __shfl_sync(0xffffffffu, stop, 0);
          if (stop) alive = false;
        }
      }
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
    // Ordered mode: the counter of the last tile added, incremented once its bulk adds
    // have completed.  The completion wait is deferred to the next step (or the end of
    // the key tile), so it overlaps the next dQ product.  A key tile only waits for higher
    // key tiles, a deferred increment only holds back lower ones, and the next key tile
    // this CTA takes starts after the release: no cycle.
    int* pend = nullptr;
    auto release_pending = [&]() {
      if (pend != nullptr) {
        bulk_wait_all();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(pend) : "memory");
        pend = nullptr;
      }
    };
    int git = 0;
    for (int t = 0;; ++t) {
      TileDesc d;
      const bool have_tile = __all_sync(0xffffffffu, read_tile(t, d));
      SeqDesc vd{};
      if constexpr (VARLEN) {
        if (have_tile) vd = vring[t & 1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TILEE0 + (t & 1)));
      if (!have_tile) break;
      for (int it = 0; it < d.total; ++it, ++git) {
        int g = it / d.m_count;
        int m = d.m_begin + (it - g * d.m_count);
        if constexpr (SPARSE) {
          const int e = p.sp_lists[(size_t)d.pad * p.sp_stride + it];
          g = e >> 16;
          m = e & 0xffff;
        }
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
        size_t tile_id = ((size_t)d.b * p.H + h) * p.Mb + m;
        if constexpr (VARLEN) tile_id = (size_t)h * p.T + vd.slot0 + m;
        float* dst = p.dq_accum + tile_id * (size_t)(128 * DP);
        int* sem = p.sems + tile_id;
        if (p.deterministic) {
          // Ordered mode: contributions to one dQ tile are added in descending key-tile
          // order; the ordering warp has waited for this step's turn.  No drain thread
          // leaves a step early, so the named barriers of a step are always reached by all
          // 128 drain threads.
          if (threadIdx.x == 128) {
            release_pending();
            volatile int* s_turn = reinterpret_cast<volatile int*>(small + SM_TILE + 8);
            int stop = !ok;
            if (!mbar_wait(bar(B_TURN), git & 1, st, kTimeoutBase - 23)) {
              stop = 1;
            } else {
              stop = stop || s_turn[git & 1];
              mbar_arrive(bar(B_TURNE));
              // the bulk adds below (async proxy) come after the counter acquire
              asm volatile("fence.proxy.async.global;" ::: "memory");
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
            if (git == 0 && hf == 0) pdl_wait_prior();  // the preprocess clears the accumulator
            bulk_reduce_add_f32(dst + (size_t)cg0 * 128 * 4, stg, (uint32_t)ncg * 128 * 16);
            bulk_commit();
          }
        }
        if (p.deterministic && threadIdx.x == 128 && *s_skip == 0) pend = sem;
        // no early exit: every drain thread reaches every named barrier of every step (on
        // an abort the waits return at once and the stores and bulk adds are skipped)
      }
      if (threadIdx.x == 128) release_pending();

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
      // the tile's mask geometry, mask bounds and first key row in dK / dV (packed
      // sequences: the sequence's own; else the call's)
      MaskGeom tg = gm;
      int t_lo = p.lo, t_hi = p.hi, t_sk = p.Sk, k_row0 = 0, tb = d.b;
      if constexpr (VARLEN) {
        if (have_tile) {
          const SeqDesc v = vring[t & 1];
          tg = seq_geom(v);
          t_lo = v.lo;
          t_hi = v.hi;
          t_sk = v.Sk;
          k_row0 = v.k_off;
          tb = 0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TILEE0 + (t & 1)));
      if (!have_tile) break;
      const int j = d.n * kTileK + jl;
      const bool row_ok = j < t_sk;

      for (int it = 0; it < d.total; ++it, ++git) {
        const int s = git & 1;
        int m = d.m_begin + (it - (it / d.m_count) * d.m_count);
        if constexpr (SPARSE) m = p.sp_lists[(size_t)d.pad * p.sp_stride + it] & 0xffff;
        const int m0 = m * kTileQ;
        const bool need_mask = !tile_full(tg, m, d.n);
        // visible columns: lo <= (j - i) <= hi with i = m0 + col0 + ql  <=>  ql in [qmin, qmax]
        const int base = j - m0 - col0;
        const int qmin = row_ok ? max(base - t_hi, -1) : 1 << 20;
        const int qmax = row_ok ? min(base - t_lo, 1 << 20) : -1;
        const float* lse = s_lse + s * 128 + col0;
        const float* dsum = s_dsum + s * 128 + col0;
        // Without softcap each lane holds the LSE2 / D of columns lane and 32 + lane of its
        // warpgroup's half, and the values reach the other lanes by shuffles: a broadcast
        // shared-memory read costs a shared-memory wavefront per 4 bytes, and the port is
        // what the step is bound by.  The ALU-heavier softcap step keeps the broadcast
        // reads, which cost fewer issue slots.

        if (!warp_wait(bar(B_SFULL), git & 1, st, kTimeoutBase - 30)) { alive = false; break; }
        tc_fence_after();
        if (threadIdx.x == 256) FA_TR(4, git);
        if (it == 0 && threadIdx.x == 256) FA_TL(t, 10, gtimer());
        float lreg[2] = {0.f, 0.f};
        if (!SOFTCAP) {
          lreg[0] = lse[lane];
          lreg[1] = lse[32 + lane];
        }
        uint32_t pc[32];  // P (times 1 - tanh^2 with softcap) as f16 pairs, reused for dS
        if (need_mask)
          phase_p<true, SOFTCAP, F16>(kc, t_lane + TM_S + col0, lse, lreg, qmin, qmax, pc);
        else
          phase_p<false, SOFTCAP, F16>(kc, t_lane + TM_S + col0, lse, lreg, qmin, qmax, pc);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL));
        if (threadIdx.x == 256) FA_TR(5, git);
        if (it == 0 && threadIdx.x == 256) FA_TL(t, 9, gtimer());
        if (threadIdx.x == 384) FA_TR(11, git);

        if (!warp_wait(bar(B_DPFULL), git & 1, st, kTimeoutBase - 31)) { alive = false; break; }
        if (git > 0 && !warp_wait(bar(B_DSEMPTY), (git - 1) & 1, st, kTimeoutBase - 32)) {
          alive = false;
          break;
        }
        tc_fence_after();
        if (threadIdx.x == 256) FA_TR(6, git);
        float dreg[2] = {0.f, 0.f};
        if (!SOFTCAP) {
          dreg[0] = dsum[lane];
          dreg[1] = dsum[32 + lane];
        }
        if (it == 0) {
          // the previous epilogue's tensor copies may still read this warp's dS rows
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(t_lane + TM_DP + col0 + c * 32, r);
          uint32_t pk[16];
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            float dv[4];
            if (SOFTCAP) {
              const float4 d4 = reinterpret_cast<const float4*>(dsum + c * 32)[v4];
              dv[0] = d4.x;
              dv[1] = d4.y;
              dv[2] = d4.z;
              dv[3] = d4.w;
            } else {
#pragma unroll
              for (int u = 0; u < 4; ++u) dv[u] = __shfl_sync(0xffffffffu, dreg[c], v4 * 4 + u);
            }
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              // dS = P * (dP - D), two columns per paired subtract and multiply
              const int e = v4 * 4 + e2 * 2;
              const float2 pcv = unpack_f16(pc[c * 16 + (e >> 1)]);
              const uint64_t d = f2_mul(f2_pack(pcv.x, pcv.y),
                                        f2_sub(f2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                               f2_pack(dv[2 * e2], dv[2 * e2 + 1])));
              pk[e >> 1] = pack_h2<F16>(f2_lo(d), f2_hi(d));
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
      // dV is final as soon as the tile's last dV is complete, so its unit is read out
      // (and, where it has its own staging buffer, stored) while the last dK / dQ still
      // run; dK follows once every MMA of the tile is complete and is staged in this
      // warp's own rows of the dS buffer, which no MMA reads any more.  Each
      // accumulator's columns are released to the next tile as soon as they are in
      // registers.
      const bool have = d.total > 0;
      constexpr int W1 = DP - 64;            // the second unit's width: 0, 16, 32 or 64
      const int krow = k_row0 + d.n * kTileK + qd * 32;
      const bool tma = p.tma_epilogue != 0 && (!VARLEN || d.n * kTileK + qd * 32 + 32 <= t_sk);
      const uint32_t slot = sbase + G::OFF_DS + wg * 16384 + qd * 4096;
      __nv_bfloat16* dv_row = p.dv + (int64_t)tb * p.dv_sb + (int64_t)(k_row0 + j) * p.dv_ss +
                              (int64_t)d.hk * p.dv_sh;
      __nv_bfloat16* dk_row = p.dk + (int64_t)tb * p.dk_sb + (int64_t)(k_row0 + j) * p.dk_ss +
                              (int64_t)d.hk * p.dk_sh;
      bool acc_ok = true;
      if (have) {
        acc_ok = warp_wait(bar(B_DVDONE), (git - 1) & 1, st, kTimeoutBase - 34);
        if (acc_ok) tc_fence_after();
      }
      const bool valid_v = have && acc_ok;
      if constexpr (G::EPI_BYTES == 0) {
        // dV waits in registers until dK's last reader is done with the dS buffer, then
        // both units of the warp go through its rows there, one after the other
        auto late = [&](auto wv, auto wk) {
          constexpr int WV = decltype(wv)::value, WK = decltype(wk)::value;
          const int cv = wg == 0 ? 0 : 64, ck = wg == 0 ? 64 : 0;
          uint32_t vpk[32];
          epi_load<WV, F16>(t_lane + TM_DV + cv, 1.f, valid_v, vpk);
          epi_release(valid_v, lane, bar(B_DVEMPTY));
          if (have) {
            acc_ok = acc_ok && warp_wait(bar(B_ACC), kt & 1, st, kTimeoutBase - 33);
            if (acc_ok) tc_fence_after();
            if (threadIdx.x == 256) FA_TL(t, 5, gtimer());
          }
          const bool store = acc_ok && __shfl_sync(0xffffffffu, *s_abort == 0, 0);
          epi_put<WV>(vpk, tma, store, slot, lane, WV == 64 ? &tdv : &tdv_t, cv, d.hk, krow, tb,
                      dv_row + cv, row_ok, p.D - cv);
          epi_unit<WK, F16>(t_lane + TM_DK + ck, p.dk_scale, have && acc_ok, bar(B_DKEMPTY), tma,
                            store, slot, lane, WK == 64 ? &tdk : &tdk_t, ck, d.hk, krow, tb,
                            dk_row + ck, row_ok, p.D - ck);
        };
        // warpgroup 0: dV columns [0, 64) and dK columns [64, Dp); warpgroup 1 the others
        if (wg == 0)
          late(IntC<64>{}, IntC<W1>{});
        else
          late(IntC<W1>{}, IntC<64>{});
      } else {
        // dV has a staging buffer of its own and leaves at once
        const bool store_v = acc_ok && __shfl_sync(0xffffffffu, *s_abort == 0, 0);
        const uint32_t vbox = sbase + G::OFF_EPI + (wg == 0 ? qd * 4096 : 16384 + qd * 64 * W1);
        if (wg == 0) {
          epi_unit<64, F16>(t_lane + TM_DV, 1.f, valid_v, bar(B_DVEMPTY), tma, store_v, vbox,
                            lane, &tdv, 0, d.hk, krow, tb, dv_row, row_ok, p.D);
        } else {
          if constexpr (W1 > 0)
            epi_unit<W1, F16>(t_lane + TM_DV + 64, 1.f, valid_v, bar(B_DVEMPTY), tma, store_v,
                              vbox, lane, &tdv_t, 64, d.hk, krow, tb, dv_row + 64, row_ok,
                              p.D - 64);
          else
            epi_release(valid_v, lane, bar(B_DVEMPTY));
        }
        if (have) {
          acc_ok = acc_ok && warp_wait(bar(B_ACC), kt & 1, st, kTimeoutBase - 33);
          if (acc_ok) tc_fence_after();
          if (threadIdx.x == 256) FA_TL(t, 5, gtimer());
        }
        const bool store = acc_ok && __shfl_sync(0xffffffffu, *s_abort == 0, 0);
        const bool valid_k = have && acc_ok;
        if (wg == 1) {
          epi_unit<64, F16>(t_lane + TM_DK, p.dk_scale, valid_k, bar(B_DKEMPTY), tma, store,
                            slot, lane, &tdk, 0, d.hk, krow, tb, dk_row, row_ok, p.D);
        } else {
          if constexpr (W1 > 0)
            epi_unit<W1, F16>(t_lane + TM_DK + 64, p.dk_scale, valid_k, bar(B_DKEMPTY), tma,
                              store, slot, lane, &tdk_t, 64, d.hk, krow, tb, dk_row + 64, row_ok,
                              p.D - 64);
          else
            epi_release(valid_k, lane, bar(B_DKEMPTY));
        }
      }
      if (have) ++kt;
      if (threadIdx.x == 256) FA_TL(t, 6, gtimer());
    }
    // the epilogue's last tensor copies complete before the CTA (and its shared memory) ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
#ifdef FA_TRACE
  if (threadIdx.x == 0) {
    FA_TL(FA_TL_TILES - 1, 2, gtimer());
    FA_TL(FA_TL_TILES - 1, 3, clock64());
  }
#endif
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

#ifdef FA_TRACE
cudaError_t bwd_trace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_fa_trace)) bytes = sizeof(g_fa_trace);
  cudaError_t e = cudaMemcpyFromSymbol(host, g_fa_trace, bytes);
  return e;
}
cudaError_t bwd_trace_mma_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_fa_mma_done)) bytes = sizeof(g_fa_mma_done);
  return cudaMemcpyFromSymbol(host, g_fa_mma_done, bytes);
}
cudaError_t bwd_timeline_copy(void* host, size_t bytes, bool clear) {
  if (clear) {
    static long long zero[FA_TL_CTAS][FA_TL_TILES][FA_TL_EV];
    return cudaMemcpyToSymbol(g_fa_tl, zero, sizeof(zero));
  }
  if (bytes > sizeof(g_fa_tl)) bytes = sizeof(g_fa_tl);
  return cudaMemcpyFromSymbol(host, g_fa_tl, bytes);
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

template <int DP, bool SC, bool F16, int MODE>
static cudaError_t launch_one(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                              const OperandMaps& v, const OperandMaps& d, const OperandMaps& dk,
                              const OperandMaps& dv, int num_ctas, bool pdl, cudaStream_t s) {
  auto kern = bwd_main_kernel<DP, SC, F16, MODE>;
  const size_t smem = Geo<DP>::TOTAL;
  // The in-kernel register split assumes exactly 128 registers per thread at launch.
  cudaFuncAttributes attr;
  cudaError_t ea = cudaFuncGetAttributes(&attr, kern);
  if (ea != cudaSuccess) return ea;
  if (attr.numRegs != 128) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // pdl: a programmatic dependent of the preprocess, whose results it waits for before
  // it reads them (its set-up and first input loads overlap the preprocess's last blocks)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_ctas);
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = la;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p, q.full, q.tail, k.full, k.tail, v.full, v.tail, d.full,
                         d.tail, dk.full, dk.tail, dv.full, dv.tail);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                            const OperandMaps& v, const OperandMaps& d, const OperandMaps& dk,
                            const OperandMaps& dv, int Dp, bool softcap, bool f16, int mode,
                            int num_ctas, bool pdl, cudaStream_t s) {
  if (num_ctas <= 0) return cudaSuccess;
#define FA_CASE_VL(DPV, MD)                                                             \
  if (f16)                                                                              \
    return softcap ? launch_one<DPV, true, true, MD>(p, q, k, v, d, dk, dv, num_ctas, pdl, s)        \
                   : launch_one<DPV, false, true, MD>(p, q, k, v, d, dk, dv, num_ctas, pdl, s);      \
  return softcap ? launch_one<DPV, true, false, MD>(p, q, k, v, d, dk, dv, num_ctas, pdl, s)         \
                 : launch_one<DPV, false, false, MD>(p, q, k, v, d, dk, dv, num_ctas, pdl, s);
#define FA_CASE(DPV)                                                                    \
  case DPV:                                                                             \
    if (mode == 1) {                                                                    \
      FA_CASE_VL(DPV, 1)                                                                \
    }                                                                                   \
    if (mode == 2) {                                                                    \
      FA_CASE_VL(DPV, 2)                                                                \
    }                                                                                   \
    FA_CASE_VL(DPV, 0)
  switch (Dp) {
    FA_CASE(64)
    FA_CASE(80)
    FA_CASE(96)
    FA_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef FA_CASE
#undef FA_CASE_VL
}

}  // namespace fa
