// fa_fwd.cu — forward attention producing O (bf16 or f16, the inputs' type) and the
// natural-log LSE (fp32).
//
// This is the prerequisite step of the backward (its O and LSE are the backward's
// inputs).  It follows the Triton page's `_attn_fwd_inner` online softmax: per 64-key
// tile, scores in log2 units, running row max m and row sum l, rescale of the output
// accumulator by exp2(m_old - m_new), acc += P V, and at the end O = acc / l and
// LSE = (m + log2 l) * ln 2 (natural log; +inf for a row with no visible key).
//
// The contractions use warp-level mma.sync (m16n8k16, bf16 or f16 -> fp32): one CTA of 4 warps
// owns 64 query rows (16 per warp) of one (batch, q-head).  Masking is the same
// bottom-right aligned band as the backward (lo <= j - i <= hi, j < Sk).
#include "fa_kernels.h"

#include <math.h>

namespace fa {

namespace {

constexpr int kFwdRows = 64;
constexpr int kFwdKeys = 64;

template <bool F16>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if (F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t ld_pair(const __nv_bfloat16* base, int64_t off, bool ok) {
  return ok ? *reinterpret_cast<const uint32_t*>(base + off) : 0u;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// tanh(x) = 1 - 2 / (exp(2x) + 1): the same formulation as the backward kernel, so both
// passes see the same softcapped logits.
__device__ __forceinline__ float tanh_exp2f(float x) {
  const float e = ex2f(x * 2.8853900817779268f);
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.f));
  return 1.f - 2.f * r;
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if (F16) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// F16: inputs and O are f16 (else bf16); the 16-bit pointers of FwdParams hold that type.
template <int DP, bool F16>
__global__ void __launch_bounds__(128) fwd_kernel(const FwdParams p) {
  constexpr int LDS = DP + 8;  // padded smem row (elements): conflict-free fragment loads
  constexpr int KT = DP / 16;  // k-steps of the S contraction
  constexpr int NT = DP / 8;   // n8 tiles of the output
  __shared__ __align__(16) __nv_bfloat16 sK[kFwdKeys * LDS];
  __shared__ __align__(16) __nv_bfloat16 sV[kFwdKeys * LDS];

  const int mblk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = mblk * kFwdRows + warp * 16;
  const int r0 = row0 + g, r1 = row0 + g + 8;

  const __nv_bfloat16* qb = p.q + (int64_t)b * p.q_sb + (int64_t)h * p.q_sh;
  uint32_t qf[KT][4];
#pragma unroll
  for (int kk = 0; kk < KT; ++kk) {
    const int c0 = kk * 16 + 2 * t, c1 = c0 + 8;
    qf[kk][0] = ld_pair(qb, (int64_t)r0 * p.q_ss + c0, r0 < p.Sq && c0 < p.D);
    qf[kk][1] = ld_pair(qb, (int64_t)r1 * p.q_ss + c0, r1 < p.Sq && c0 < p.D);
    qf[kk][2] = ld_pair(qb, (int64_t)r0 * p.q_ss + c1, r0 < p.Sq && c1 < p.D);
    qf[kk][3] = ld_pair(qb, (int64_t)r1 * p.q_ss + c1, r1 < p.Sq && c1 < p.D);
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};

  // keys any row of this block can see
  const int qlo = mblk * kFwdRows;
  const int qhi = min(qlo + kFwdRows - 1, p.Sq - 1);
  long long jmin = (long long)qlo + p.lo, jmax = (long long)qhi + p.hi;
  if (jmin < 0) jmin = 0;
  if (jmax > p.Sk - 1) jmax = p.Sk - 1;

  const __nv_bfloat16* kb = p.k + (int64_t)b * p.k_sb + (int64_t)hk * p.k_sh;
  const __nv_bfloat16* vb = p.v + (int64_t)b * p.v_sb + (int64_t)hk * p.v_sh;
  const uint32_t sV_addr = static_cast<uint32_t>(__cvta_generic_to_shared(sV));

  for (long long n0 = (jmin / kFwdKeys) * kFwdKeys; n0 <= jmax; n0 += kFwdKeys) {
    __syncthreads();
    for (int c = threadIdx.x; c < kFwdKeys * (DP / 8); c += 128) {
      const int r = c / (DP / 8), col = (c % (DP / 8)) * 8;
      const long long j = n0 + r;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (j < p.Sk && col < p.D) {
        kv = *reinterpret_cast<const uint4*>(kb + j * p.k_ss + col);
        vv = *reinterpret_cast<const uint4*>(vb + j * p.v_ss + col);
      }
      *reinterpret_cast<uint4*>(sK + r * LDS + col) = kv;
      *reinterpret_cast<uint4*>(sV + r * LDS + col) = vv;
    }
    __syncthreads();

    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const __nv_bfloat16* kr = sK + (nt * 8 + g) * LDS + kk * 16 + 2 * t;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 8);
        mma_16816<F16>(s[nt], qf[kk], b0, b1);
      }
    }
    // scores in log2 units, masked entries -> -inf
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const long long j = n0 + nt * 8 + 2 * t + (e & 1);
        const int i = (e < 2) ? r0 : r1;
        float z;
        if (p.softcap_on) {
          z = tanh_exp2f(s[nt][e] * p.cap_scale) * p.cap_log2;
        } else {
          z = s[nt][e] * p.scale_log2;
        }
        const long long d = j - i;
        const bool vis = j < p.Sk && d >= p.lo && d <= p.hi;
        z = vis ? z : -INFINITY;
        s[nt][e] = z;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], z);
      }
    }
    float alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      tmax[rr] = fmaxf(tmax[rr], __shfl_xor_sync(0xffffffffu, tmax[rr], 1));
      tmax[rr] = fmaxf(tmax[rr], __shfl_xor_sync(0xffffffffu, tmax[rr], 2));
      const float mnew = fmaxf(mrow[rr], tmax[rr]);
      alpha[rr] = (mnew == -INFINITY) ? 1.f : ex2f(mrow[rr] - mnew);
      mrow[rr] = mnew;
      lrow[rr] *= alpha[rr];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    uint32_t pa[4][4];  // P as A fragments, 4 k16 steps over the 64 keys
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = mrow[e >> 1];
        pv[e] = (m == -INFINITY) ? 0.f : ex2f(s[nt][e] - m);
        lrow[e >> 1] += pv[e];
      }
      const int kk = nt >> 1;
      if ((nt & 1) == 0) {
        pa[kk][0] = pack2<F16>(pv[0], pv[1]);
        pa[kk][1] = pack2<F16>(pv[2], pv[3]);
      } else {
        pa[kk][2] = pack2<F16>(pv[0], pv[1]);
        pa[kk][3] = pack2<F16>(pv[2], pv[3]);
      }
    }
    // O += P V : B fragments from V [key][d] with ldmatrix.trans, two n8 tiles per call
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        const int rowk = kk * 16 + (lane & 15);
        const int colv = n * 8 + ((lane >> 4) << 3);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(sV_addr + (uint32_t)(rowk * LDS + colv) * 2u, b0, b1, b2, b3);
        mma_16816<F16>(o[n], pa[kk], b0, b1);
        mma_16816<F16>(o[n + 1], pa[kk], b2, b3);
      }
    }
  }

  float inv[2], lse[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    float l = lrow[rr];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const bool empty = !(l > 0.f);
    inv[rr] = empty ? 0.f : 1.f / l;
    lse[rr] = empty ? INFINITY : (mrow[rr] + log2f(l)) * 0.69314718055994531f;
  }
  __nv_bfloat16* ob = p.o + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int col = n * 8 + 2 * t;
    if (col < p.D) {
      if (r0 < p.Sq)
        *reinterpret_cast<uint32_t*>(ob + (int64_t)r0 * p.o_ss + col) = pack2<F16>(o[n][0] * inv[0], o[n][1] * inv[0]);
      if (r1 < p.Sq)
        *reinterpret_cast<uint32_t*>(ob + (int64_t)r1 * p.o_ss + col) = pack2<F16>(o[n][2] * inv[1], o[n][3] * inv[1]);
    }
  }
  if (t == 0) {
    float* lb = p.lse + (int64_t)b * p.lse_sb + (int64_t)h * p.lse_sh;
    if (r0 < p.Sq) lb[(int64_t)r0 * p.lse_ss] = lse[0];
    if (r1 < p.Sq) lb[(int64_t)r1 * p.lse_ss] = lse[1];
  }
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int Dp, bool f16, cudaStream_t s) {
  dim3 grid((p.Sq + kFwdRows - 1) / kFwdRows, p.H, p.B);
#define FA_FWD_CASE(DPV)                                   \
  case DPV:                                                \
    if (f16)                                               \
      fwd_kernel<DPV, true><<<grid, 128, 0, s>>>(p);       \
    else                                                   \
      fwd_kernel<DPV, false><<<grid, 128, 0, s>>>(p);      \
    break;
  switch (Dp) {
    FA_FWD_CASE(64)
    FA_FWD_CASE(80)
    FA_FWD_CASE(96)
    FA_FWD_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef FA_FWD_CASE
  return cudaGetLastError();
}

}  // namespace fa
