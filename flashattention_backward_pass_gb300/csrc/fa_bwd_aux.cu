// fa_bwd_aux.cu — the two memory-bound kernels around the backward main kernel.
//
// preprocess (call-trace page: `softmax_d` holds the row sums of dout*out; `dq_accum` is
// the fp32 dQ accumulator):
//   D_i   = sum_d dO_id * O_id   (fp32; 0 on the padded rows of the last query tile)
//   LSE2  = LSE * log2(e)        (the sm90 page's P = exp2(S*scale*log2e - LSE_log2); +inf
//                                 on padded rows, which makes P = 0 there)
//   zero the fp32 dQ accumulator, the deterministic-mode counters and the status/ticket
//   words.
// convert (call-trace page: the "reduction kernel" after the dq_accum stores):
//   dQ = bf16(scale * accumulator), cropped to Sq rows and D columns.
#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_tiles.h"

#include <math.h>

namespace fa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Blocks [0, row_blocks) compute D and LSE2: each warp takes 4 rows per pass (8 lanes per
// row, 16 bf16 per lane as two 16-byte loads each of dO and O), so a warp keeps 8 loads per
// lane in flight.  Blocks [row_blocks, gridDim.x) clear the accumulator and the counters
// with 16-byte stores.  The two kinds of blocks run side by side, so the latency-bound row
// reductions overlap the bandwidth-bound clearing.
// F16: dO and O are f16 (else bf16).  VARLEN: packed sequences (rows by slot).  WIDE:
// rows of up to 256 columns (two 128-column passes).
template <bool F16, bool VARLEN, bool WIDE = false>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdPreParams p, int row_blocks) {
  if (blockIdx.x == 0 && threadIdx.x < 4) p.header[threadIdx.x] = 0;
  if ((int)blockIdx.x >= row_blocks) {
    const int64_t nthreads = (int64_t)(gridDim.x - row_blocks) * blockDim.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t k = (int64_t)(blockIdx.x - row_blocks) * blockDim.x + threadIdx.x;
         k < p.zero_count; k += nthreads)
      p.zero_ptr[k] = z;
    // A clearing block that is done lets the main kernel (launched as this grid's
    // programmatic dependent) start once every block has finished or signalled; the main
    // kernel waits for this grid's results before it reads them.  Signalling at the start
    // instead let the main kernel's CTAs take SMs that this grid still needed (slower).
    pdl_launch_dependents();
    return;
  }
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;  // row within the warp's group of 4
  const int l8 = lane & 7;    // 16-column slice of the row
  const int64_t nrows = VARLEN ? (int64_t)p.H * p.T * 128 : (int64_t)p.B * p.H * p.Sq_r;
  const int64_t warps_total = (int64_t)row_blocks * (blockDim.x >> 5);
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);

  for (int64_t r4 = wid; 4 * r4 < nrows; r4 += warps_total) {
    const int64_t r = 4 * r4 + sub;
    float acc = 0.f;
    // the row's (batch coordinate, row coordinate, head) in dO / O / LSE, and whether it
    // is a query row at all (rather than padding of its last tile)
    int64_t b = 0, i = 0, h = 0;
    bool real = false;
    const bool valid_row = r < nrows;
    if (valid_row) {
      if constexpr (VARLEN) {
        // per head T slots of 128 rows; slot t belongs to sequence slot_owner(t)
        const int64_t tile = r >> 7;
        h = tile / p.T;
        const int64_t t = tile - h * p.T;
        const int sb = slot_owner(p.cu_q, p.B, p.total_q, t);
        int64_t q0, sq;
        seq_rows(p.cu_q, p.used_q, sb, p.total_q, &q0, &sq);
        const int64_t il = (t - first_slot(p.cu_q, sb, p.total_q)) * 128 + (r & 127);
        real = il >= 0 && il < sq;  // (il < 0 only for malformed offsets)
        i = q0 + il;
      } else {
        const int64_t bh = r / p.Sq_r;
        const int64_t il = r - bh * p.Sq_r;
        real = il < p.Sq;
        b = bh / p.H;
        h = bh - b * p.H;
        i = il;
      }
      if (real) {
        const __nv_bfloat16* a = p.dout + b * p.do_sb + i * p.do_ss + h * p.do_sh;
        const __nv_bfloat16* o = p.out + b * p.o_sb + i * p.o_ss + h * p.o_sh;
#pragma unroll
        for (int ch = 0; ch < (WIDE ? 2 : 1); ++ch) {
          uint4 av[2], ov[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = ch * 128 + l8 * 16 + u * 8;
            av[u] = c < p.D ? *reinterpret_cast<const uint4*>(a + c) : make_uint4(0, 0, 0, 0);
            ov[u] = c < p.D ? *reinterpret_cast<const uint4*>(o + c) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t aw[4] = {av[u].x, av[u].y, av[u].z, av[u].w};
            const uint32_t ow[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 af = unpack_h2<F16>(aw[e]);
              const float2 of = unpack_h2<F16>(ow[e]);
              acc = fmaf(af.x, of.x, acc);
              acc = fmaf(af.y, of.y, acc);
            }
          }
        }
      }
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid_row && l8 == 0) {
      float l2 = INFINITY;
      if (real) {
        const float l = p.lse[b * p.lse_sb + h * p.lse_sh + i * p.lse_ss];
        l2 = l * kLog2e;
      }
      p.dsum[r] = acc;
      p.lse2[r] = l2;
    }
  }
}

// Block (16, 16) covers 64 query rows of one (b, h): threadIdx.x = 8-column group,
// threadIdx.y = row within each of 4 groups of 16 rows.  A thread issues its 8 loads (two
// per row) before any store, so a warp keeps 8 x 32 bytes per lane in flight.  Per row
// group a warp covers two rows: its reads are whole 32-byte sectors of the accumulator
// tile layout and its writes two contiguous 256-byte row segments of dQ.
// F16: dQ is written as f16 (else bf16).
constexpr int kConvRows = 4;
template <bool F16>
__global__ void __launch_bounds__(256) bwd_convert_kernel(const BwdConvParams p) {
  const int o = threadIdx.x;  // 8-column group
  bool active = o * 8 < p.D;
  // this block's 64 rows: tile (its index in the accumulator), first local row inside the
  // tile, and the (batch coordinate, first row coordinate, head, rows that exist) in dQ
  size_t tile_id;
  int row0, b, h, nvalid;
  int64_t i0;
  if (p.varlen) {
    // per head T slots of 128 rows, two blocks per slot
    tile_id = blockIdx.x >> 1;
    row0 = (blockIdx.x & 1) * (16 * kConvRows);
    h = (int)(tile_id / (size_t)p.T);
    const int64_t t = (int64_t)tile_id - (int64_t)h * p.T;
    const int sb = slot_owner(p.cu_q, p.B, p.total_q, t);
    int64_t q0, sq;
    seq_rows(p.cu_q, p.used_q, sb, p.total_q, &q0, &sq);
    const int64_t il = (t - first_slot(p.cu_q, sb, p.total_q)) * 128 + row0;
    b = 0;
    i0 = q0 + il;
    // (il < 0 only for malformed offsets: write nothing then)
    nvalid = (int)(il < 0 || sq - il < 0 ? 0 : (sq - il > 16 * kConvRows ? 16 * kConvRows : sq - il));
  } else {
    const int nrb = (p.Sq + 16 * kConvRows - 1) / (16 * kConvRows);   // row blocks per (b, h)
    const int bh = (int)(blockIdx.x / (unsigned)nrb);
    const int rb = (int)(blockIdx.x - (unsigned)bh * (unsigned)nrb);
    b = bh / p.H;
    h = bh - b * p.H;
    const int r0 = rb * (16 * kConvRows);
    row0 = r0 & 127;
    tile_id = (size_t)bh * p.Mb + (r0 >> 7);
    i0 = r0;
    nvalid = p.Sq - r0 < 16 * kConvRows ? p.Sq - r0 : 16 * kConvRows;
  }
  const float* tile = p.dq_accum + tile_id * (size_t)(128 * p.Dp);
  float4 lo[kConvRows], hi[kConvRows];
#pragma unroll
  for (int r = 0; r < kConvRows; ++r) {
    const int rl = r * 16 + threadIdx.y;  // row within the block
    const int q = row0 + rl;              // row within the tile
    lo[r] = hi[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && rl < nvalid) {
      lo[r] = __ldcs(reinterpret_cast<const float4*>(tile + ((size_t)(2 * o) * 128 + q) * 4));
      hi[r] = __ldcs(reinterpret_cast<const float4*>(tile + ((size_t)(2 * o + 1) * 128 + q) * 4));
    }
  }
  const float s = p.scale;
#pragma unroll
  for (int r = 0; r < kConvRows; ++r) {
    const int rl = r * 16 + threadIdx.y;
    if (!active || rl >= nvalid) break;
    const uint4 v = make_uint4(pack_h2<F16>(lo[r].x * s, lo[r].y * s), pack_h2<F16>(lo[r].z * s, lo[r].w * s),
                               pack_h2<F16>(hi[r].x * s, hi[r].y * s), pack_h2<F16>(hi[r].z * s, hi[r].w * s));
    *reinterpret_cast<uint4*>(p.dq + (int64_t)b * p.dq_sb + (i0 + rl) * p.dq_ss +
                              (int64_t)h * p.dq_sh + o * 8) = v;
  }
  // The block's 64 accumulator rows are dead now (every load above has been consumed by
  // a store).  Their L2 lines are still dirty from the main kernel's adds: drop them
  // without a write-back to DRAM.  A 128-byte line holds 8 rows of one 4-column group.
  __syncthreads();
  const int nlines = (p.Dp / 4) * (16 * kConvRows / 8);
  const int tid = threadIdx.y * 16 + threadIdx.x;
  for (int l = tid; l < nlines; l += 256) {
    const int cg = l >> 3, ro = l & 7;
    const float* line = tile + ((size_t)cg * 128 + row0 + ro * 8) * 4;
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
  }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdPreParams& p, bool f16, cudaStream_t s) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nrows = p.varlen ? (int64_t)p.H * p.T * 128 : (int64_t)p.B * p.H * p.Sq_r;
  const int64_t row_quads = (nrows + 3) / 4;
  int64_t row_blocks = (row_quads + 7) / 8;                 // 8 warps per block
  const int64_t row_cap = (int64_t)sms * 8;
  if (row_blocks > row_cap) row_blocks = row_cap;
  if (row_blocks < 1) row_blocks = 1;
  int64_t zero_blocks = (p.zero_count + 255) / 256;
  const int64_t zero_cap = (int64_t)sms * 8;
  if (zero_blocks > zero_cap) zero_blocks = zero_cap;
  const unsigned grid = (unsigned)(row_blocks + zero_blocks);
  if (p.D > 128) {
    // head dims above 128 (batched calls only)
    if (f16)
      bwd_preprocess_kernel<true, false, true><<<grid, 256, 0, s>>>(p, (int)row_blocks);
    else
      bwd_preprocess_kernel<false, false, true><<<grid, 256, 0, s>>>(p, (int)row_blocks);
  } else if (p.varlen) {
    if (f16)
      bwd_preprocess_kernel<true, true><<<grid, 256, 0, s>>>(p, (int)row_blocks);
    else
      bwd_preprocess_kernel<false, true><<<grid, 256, 0, s>>>(p, (int)row_blocks);
  } else {
    if (f16)
      bwd_preprocess_kernel<true, false><<<grid, 256, 0, s>>>(p, (int)row_blocks);
    else
      bwd_preprocess_kernel<false, false><<<grid, 256, 0, s>>>(p, (int)row_blocks);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_convert(const BwdConvParams& p, bool f16, cudaStream_t s) {
  if (p.Sq == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
  const int64_t blocks = p.varlen ? (int64_t)p.H * p.T * (128 / (16 * kConvRows))
                                  : (int64_t)((p.Sq + 16 * kConvRows - 1) / (16 * kConvRows)) * p.B * p.H;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)blocks);
  if (f16)
    bwd_convert_kernel<true><<<grid, dim3(16, 16), 0, s>>>(p);
  else
    bwd_convert_kernel<false><<<grid, dim3(16, 16), 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fa

namespace fa {

namespace {

// Block-sparse step lists: warp t handles key-tile ticket t (the main kernel's
// key-tile-major order: n = t / (B Hk), or Nb - 1 - t / (B Hk) in the ordered mode, then
// b, then hk).  Its candidate steps are the
// main kernel's dense sequence — q-head g of the group outer, query tile m in the
// element mask's range inner — and it keeps those whose block-mask byte
// block_mask[b, hk*G + g, m, n] is set, compacted in order with warp ballots.
__global__ void __launch_bounds__(256) bwd_sparse_lists_kernel(const BwdSparseParams p) {
  const int t = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
  const int lane = threadIdx.x & 31;
  if (t >= p.num_tiles) return;
  const int per_n = p.B * p.Hk;
  const int n0 = t / per_n;
  const int n = p.deterministic ? p.Nb - 1 - n0 : n0;
  const int r = t - n0 * per_n;
  const int b = r / p.Hk;
  const int hk = r - b * p.Hk;
  MaskGeom gm;
  gm.Sq = p.Sq;
  gm.Sk = p.Sk;
  gm.lo = p.lo64;
  gm.hi = p.hi64;
  gm.tm = kTileQ;
  gm.tn = kTileK;
  gm.Mb = p.Mb;
  gm.Nb = p.Nb;
  int64_t mb, me;
  m_range(gm, n, &mb, &me);
  const int mc = (int)(me - mb);
  const int total = mc * p.G;
  int* out = p.lists + (size_t)t * p.stride;
  int kept = 0;
  for (int c0 = 0; c0 < total; c0 += 32) {
    const int c = c0 + lane;
    int g = 0, m = 0;
    bool keep = false;
    if (c < total) {
      g = c / mc;
      m = (int)mb + (c - g * mc);
      const int h = hk * p.G + g;
      keep = p.block_mask[(((size_t)b * p.H + h) * p.Mb + m) * (size_t)p.Nb + n] != 0;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (keep) out[kept + __popc(bal & ((1u << lane) - 1u))] = (g << 16) | m;
    kept += __popc(bal);
  }
  if (lane == 0) p.counts[t] = kept;
}

}  // namespace

cudaError_t launch_bwd_sparse_lists(const BwdSparseParams& p, cudaStream_t s) {
  if (p.num_tiles <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((p.num_tiles + 7) / 8);  // 8 warps per block
  bwd_sparse_lists_kernel<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
