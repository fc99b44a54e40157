// fa_bwd_common.cuh — pieces shared by the backward kernels: the shared-memory geometry of
// a 128-row bf16 operand tile, the tcgen05 matrix descriptors that address it, a
// warp-uniform bounded wait, and the probability step (P = exp2(S*scale*log2e - LSE2)).
#pragma once

#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_tiles.h"

namespace fa {

// A 128-row tile of a Dp-wide bf16 operand in shared memory: 64-column panels with the
// 128-byte swizzle (what TMA writes for a 64-element box), plus a 16- or 32-column tail
// panel with the 32- or 64-byte swizzle when Dp % 64 != 0.
template <int DP>
struct Panels {
  static_assert(DP % 16 == 0 && DP >= 64 && DP <= 128, "Dp in [64, 128], multiple of 16");
  static constexpr int NFULL = DP / 64;                          // 64-column panels
  static constexpr int TAIL = DP % 64;                           // 0, 16 or 32 columns
  static_assert(TAIL == 0 || TAIL == 16 || TAIL == 32, "tail panel of 16 or 32 columns");
  static constexpr uint32_t FULL_BYTES = 128u * 128u;            // 128 rows x 128 B
  static constexpr uint32_t TAIL_ROWB = TAIL * 2;                // bytes per row in tail
  static constexpr uint32_t TAIL_OFF = NFULL * FULL_BYTES;
  static constexpr uint32_t TILE_BYTES = NFULL * FULL_BYTES + 128u * TAIL_ROWB;
  static constexpr uint32_t TAIL_SWZ = TAIL == 16 ? SWZ_32B : SWZ_64B;
  static constexpr int KSTEPS = DP / 16;
  static_assert(TILE_BYTES % 1024 == 0, "tiles stay 1024-byte aligned");
};

// K-major operand (rows = M or N, Dp contiguous columns = the contraction), K-step ks
// (16 columns).
template <int DP>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int ks) {
  using P = Panels<DP>;
  if (ks < P::NFULL * 4) {
    const uint32_t addr = tile + (ks >> 2) * P::FULL_BYTES + (ks & 3) * 32;
    return smem_desc(addr, 16, 1024, SWZ_128B);
  }
  const int kk = ks - P::NFULL * 4;
  return smem_desc(tile + P::TAIL_OFF + kk * 32, 16, 8 * P::TAIL_ROWB, P::TAIL_SWZ);
}

// MN-major operand whose 128 rows are the contraction index (16 rows per K-step) and whose
// Dp columns are N: descriptor of the 64-column panels (all of them; LBO = panel stride)
// or of the tail panel.
template <int DP>
__device__ __forceinline__ uint64_t desc_mn_full(uint32_t tile, int ks) {
  return smem_desc(tile + ks * 16 * 128, Panels<DP>::FULL_BYTES, 1024, SWZ_128B);
}
template <int DP>
__device__ __forceinline__ uint64_t desc_mn_tail(uint32_t tile, int ks) {
  using P = Panels<DP>;
  return smem_desc(tile + P::TAIL_OFF + ks * 16 * P::TAIL_ROWB, 128u * P::TAIL_ROWB,
                   8 * P::TAIL_ROWB, P::TAIL_SWZ);
}

// Every lane waits (each needs the barrier's acquire), then the warp agrees: a lane that
// saw the abort flag makes the whole warp stop, so .sync.aligned tcgen05 ops that follow
// are always executed by all 32 lanes or by none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const AbortState& st,
                                          int code) {
  const bool ok = mbar_wait(bar, parity, st, code);
  return __all_sync(0xffffffffu, ok);
}

struct SoftmaxConsts {
  float scale_log2;  // scale * log2(e)
  float cap_scale;   // scale / softcap
  float cap_log2;    // softcap * log2(e)
};

// P for one score: exp2(S*scale*log2e - LSE2) or, with softcap c,
// exp2(c*log2e*tanh(S*scale/c) - LSE2); *fac receives d z / d(scale*S) = 1 - tanh^2
// (1 without softcap), the factor the chain rule puts on dZ.
template <bool SOFTCAP>
__device__ __forceinline__ float prob(const SoftmaxConsts& k, float s, float lse2, float* fac) {
  if (SOFTCAP) {
    const float t = tanh_exp2(s * k.cap_scale);
    *fac = fmaf(-t, t, 1.f);
    return ex2_approx(fmaf(t, k.cap_log2, -lse2));
  }
  *fac = 1.f;
  return ex2_approx(fmaf(s, k.scale_log2, -lse2));
}

// Contractions issued by a single MMA thread.  Each operand tile's descriptors are built
// once; a K-step only adds a constant to the low descriptor word.  The K-step loops are
// fully unrolled, so consecutive MMAs reach the tensor pipe back to back.

// Descriptors of one 128-row operand tile: K-major (rows = M or N, Dp contiguous columns
// = the contraction) and MN-major (rows = the contraction, Dp columns = N) views of the
// 64-column panels and of the tail panel.
struct TileDescs {
  DescWords kfull, ktail, mfull, mtail;
};

template <int DP>
__device__ __forceinline__ TileDescs tile_descs(uint32_t tile) {
  using P = Panels<DP>;
  TileDescs o;
  o.kfull = desc_words(tile, 16, 1024, SWZ_128B);
  o.mfull = desc_words(tile, P::FULL_BYTES, 1024, SWZ_128B);
  o.ktail = desc_words(tile + P::TAIL_OFF, 16, 8 * P::TAIL_ROWB, P::TAIL_SWZ);
  o.mtail = desc_words(tile + P::TAIL_OFF, 128u * P::TAIL_ROWB, 8 * P::TAIL_ROWB, P::TAIL_SWZ);
  return o;
}

// D = A B^T with both operands K-major over Dp (backward: S^T = K Q^T, dP^T = V dO^T;
// forward: S = Q K^T).
template <int DP, bool F16>
__device__ __forceinline__ void mma_kmajor(uint32_t d, const TileDescs& A, const TileDescs& B) {
  using P = Panels<DP>;
  constexpr uint32_t ID = idesc_h<F16>(128, 128, false, false);
#pragma unroll
  for (int ks = 0; ks < P::NFULL * 4; ++ks) {
    const uint32_t off = (ks >> 2) * (P::FULL_BYTES >> 4) + (ks & 3) * 2;
    if (ks == 0)
      mma_ss_w<0>(d, A.kfull, off, B.kfull, off, ID);
    else
      mma_ss_w<1>(d, A.kfull, off, B.kfull, off, ID);
  }
#pragma unroll
  for (int kk = 0; kk < P::TAIL / 16; ++kk) mma_ss_w<1>(d, A.ktail, kk * 2, B.ktail, kk * 2, ID);
}

// D (+)= A B with A (128 x 128, 16-bit pairs) in tensor memory and B a 128-row tile read
// MN-major (N = Dp): backward dV += P^T dO (P^T written over the S^T columns), forward
// O += P V (P written over the S columns).  K-steps 0-3 read A's columns [0, 32), K-steps
// 4-7 its columns [64, 96): each half of the 128-column score tile holds its 64 values as
// pairs at the start of its own 64 columns.
template <int DP, bool F16>
__device__ __forceinline__ void mma_dv(uint32_t d, uint32_t a_tmem, const TileDescs& B, uint32_t acc) {
  using P = Panels<DP>;
  constexpr uint32_t ID = idesc_h<F16>(128, P::NFULL * 64, false, true);
  constexpr uint32_t ID_T = idesc_h<F16>(128, P::TAIL ? P::TAIL : 16, false, true);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t a_t = a_tmem + (ks >> 2) * 64 + (ks & 3) * 8;
    if (ks == 0) {
      mma_ts_wp(d, a_t, B.mfull, 0, ID, acc);
      if (P::TAIL) mma_ts_wp(d + P::NFULL * 64, a_t, B.mtail, 0, ID_T, acc);
    } else {
      mma_ts_w<1>(d, a_t, B.mfull, ks * 128, ID);
      if (P::TAIL) mma_ts_w<1>(d + P::NFULL * 64, a_t, B.mtail, ks * P::TAIL_ROWB, ID_T);
    }
  }
}

}  // namespace fa
