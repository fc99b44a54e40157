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

}  // namespace fa
