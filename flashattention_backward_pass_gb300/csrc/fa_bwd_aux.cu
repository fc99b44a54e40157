// fa_bwd_aux.cu — the two memory-bound kernels around the backward main kernel.
//
// preprocess (call-trace page: `softmax_d` holds the row sums of dout*out; `dq_accum` is
// the fp32 dQ accumulator):
//   D_i   = sum_d dO_id * O_id   (fp32; 0 on the padded rows of the last query tile)
//   LSE2  = LSE * log2(e)        (the sm90 page's P = exp2(S*scale*log2e - LSE_log2); +inf
//                                 on padded rows, which makes P = 0 there)
//   zero the dQ accumulator, the deterministic-mode counters and the status/ticket words.
// convert (call-trace page: the "reduction kernel" after the dq_accum stores):
//   dQ = bf16(scale * accumulator), cropped to Sq rows and D columns.
#include "fa_kernels.h"

#include <math.h>

namespace fa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Two rows per warp, 16 lanes per row, 8 bf16 per lane (D <= 128).
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdPreParams p) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int l16 = lane & 15;
  const int64_t nrows = (int64_t)p.B * p.H * p.Sq_r;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);

  if (blockIdx.x == 0 && threadIdx.x < 4) p.header[threadIdx.x] = 0;

  for (int64_t r2 = wid; 2 * r2 < nrows; r2 += warps_total) {
    const int64_t r = 2 * r2 + half;
    float acc = 0.f;
    int64_t bh = 0, i = 0;
    const bool valid_row = r < nrows;
    if (valid_row) {
      bh = r / p.Sq_r;
      i = r - bh * p.Sq_r;
      if (i < p.Sq && l16 * 8 < p.D) {
        const int64_t b = bh / p.H, h = bh - (bh / p.H) * p.H;
        const uint4 a = *reinterpret_cast<const uint4*>(p.dout + b * p.do_sb + i * p.do_ss +
                                                         h * p.do_sh + l16 * 8);
        const uint4 o = *reinterpret_cast<const uint4*>(p.out + b * p.o_sb + i * p.o_ss +
                                                         h * p.o_sh + l16 * 8);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 af = __bfloat1622float2(a2[e]);
          const float2 of = __bfloat1622float2(o2[e]);
          acc = fmaf(af.x, of.x, acc);
          acc = fmaf(af.y, of.y, acc);
        }
      }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid_row && l16 == 0) {
      float l2 = INFINITY;
      if (i < p.Sq) {
        const int64_t b = bh / p.H, h = bh - (bh / p.H) * p.H;
        const float l = p.lse[b * p.lse_sb + h * p.lse_sh + i * p.lse_ss];
        l2 = l * kLog2e;
      }
      p.dsum[r] = acc;
      p.lse2[r] = l2;
    }
  }

  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < p.zero_count; k += nthreads)
    p.zero_ptr[k] = z;
}

// Block (16, 16): threadIdx.x = 8-column group, threadIdx.y = query row.  A warp covers two
// rows: its reads are whole 32-byte sectors of the accumulator tile layout and its writes
// are two contiguous 256-byte row segments of dQ.
__global__ void __launch_bounds__(256) bwd_convert_kernel(const BwdConvParams p) {
  const int o = threadIdx.x;                    // 8-column group
  const int i = blockIdx.x * 16 + threadIdx.y;  // query row
  const int bh = blockIdx.y;
  if (i >= p.Sq || o * 8 >= p.D) return;
  const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
  const int m = i >> 7, q = i & 127;
  const float* tile = p.dq_accum + ((size_t)bh * p.Mb + m) * (size_t)(128 * p.Dp);
  const float4 lo = *reinterpret_cast<const float4*>(tile + ((size_t)(2 * o) * 128 + q) * 4);
  const float4 hi = *reinterpret_cast<const float4*>(tile + ((size_t)(2 * o + 1) * 128 + q) * 4);
  const float s = p.scale;
  __nv_bfloat162 r[4];
  r[0] = __floats2bfloat162_rn(lo.x * s, lo.y * s);
  r[1] = __floats2bfloat162_rn(lo.z * s, lo.w * s);
  r[2] = __floats2bfloat162_rn(hi.x * s, hi.y * s);
  r[3] = __floats2bfloat162_rn(hi.z * s, hi.w * s);
  *reinterpret_cast<uint4*>(p.dq + (int64_t)b * p.dq_sb + (int64_t)i * p.dq_ss +
                            (int64_t)h * p.dq_sh + o * 8) = *reinterpret_cast<uint4*>(r);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdPreParams& p, cudaStream_t s) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t row_pairs = ((int64_t)p.B * p.H * p.Sq_r + 1) / 2;
  const int64_t need = (row_pairs + 7) / 8;            // 8 warps per block
  const int64_t need_zero = (p.zero_count + 255) / 256;
  int64_t blocks = need > need_zero ? need : need_zero;
  const int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  bwd_preprocess_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_convert(const BwdConvParams& p, cudaStream_t s) {
  if (p.Sq == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  dim3 grid((p.Sq + 15) / 16, p.B * p.H);
  bwd_convert_kernel<<<grid, dim3(16, 16), 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
