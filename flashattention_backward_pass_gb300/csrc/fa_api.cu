// fa_api.cu — host side of the C ABI declared in include/fa.h: argument validation,
// workspace carving, TMA tensor-map encoding and the kernel launches.
//
// Validation rules follow the pages: non-null inputs, matching dims, K/V shape match,
// equal dtypes, head dim bounds and H % Hk == 0 (Triton page, `validate_inputs`); fp32
// LSE (`flash_bwd_sm90.py` page, `_check_type`); head dim a multiple of 8
// (`can_implement`); 16-byte-divisible strides for the TMA copies (the sm90 page's
// `__call__` assumes 128-bit-divisible strides); Sq == 0 launches nothing (call-trace
// page, `mha_bwd` launches only when seqlen_q > 0).
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_kernels.h"
#include "fa_tiles.h"

using namespace fa;

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Test hooks (process-wide): a shorter bounded-wait limit and, for the deterministic
// path, an ordering counter that no contributor will ever match (so the ordered wait
// must run out and report FA_ERR_DEVICE_TIMEOUT).
long long g_wait_limit = 2000000000ll;
int g_poison_first_counter = 0;
int g_bwd_algorithm = FA_BWD_ALGO_AUTO;

// Optional timing of the three backward kernels: events recorded on the caller's stream
// before the preprocess, before and after the main kernel and after the convert.  The
// events belong to the device that was current when profiling was enabled; a call on
// another device records nothing (and fa_profile_read then reports the last call made on
// the profiled device).
bool g_profile = false;
int g_profile_dev = -1;
cudaEvent_t g_ev[4] = {nullptr, nullptr, nullptr, nullptr};

void prof_record(int i, cudaStream_t s) {
  if (!g_profile) return;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != g_profile_dev) return;
  cudaEventRecord(g_ev[i], s);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int pad64(int d) { return (d + 63) / 64 * 64; }

int padded_dim(int D) {
  if (D <= 64) return 64;
  if (D <= 80) return 80;
  if (D <= 96) return 96;
  return 128;
}

struct BwdLayout {
  int Mb, Sq_r, Dp;
  size_t off_lse2, off_dsum, off_accum, off_sems, total, accum_bytes, sems_bytes;
};

bool bwd_layout(int B, int H, int Sq, int D, BwdLayout* L) {
  if (B < 0 || H <= 0 || Sq < 0 || D <= 0) return false;
  L->Dp = padded_dim(D);
  L->Mb = (Sq + kTileQ - 1) / kTileQ;
  L->Sq_r = L->Mb * kTileQ;
  const size_t rows = (size_t)B * H * L->Sq_r;
  size_t off = WS_HEADER_BYTES;
  L->off_lse2 = off;
  off = align_up(off + rows * 4, 256);
  L->off_dsum = off;
  off = align_up(off + rows * 4, 256);
  L->off_accum = off;
  const size_t accum = (size_t)B * H * L->Mb * kTileQ * L->Dp * 4;
  off += accum;
  L->off_sems = off;
  const size_t sems = align_up((size_t)B * H * L->Mb * 4, 16);
  off += sems;
  L->accum_bytes = accum;
  L->sems_bytes = sems;
  L->total = align_up(off, 256);
  return true;
}

// Head dims above 128 or Dv != D (fa_wide.cu): the same header, LSE2 and D regions, and a
// dQ accumulator of (B, H, ceil(Sq / 64), ceil(pad64(D) / 128)) blocks of 128 x 64 fp32.
bool bwd_layout_wide(int B, int H, int Sq, int D, BwdLayout* L) {
  if (B < 0 || H <= 0 || Sq < 0 || D <= 0) return false;
  L->Dp = pad64(D);
  L->Mb = (Sq + kTileQ - 1) / kTileQ;
  L->Sq_r = L->Mb * kTileQ;
  const size_t rows = (size_t)B * H * L->Sq_r;
  size_t off = WS_HEADER_BYTES;
  L->off_lse2 = off;
  off = align_up(off + rows * 4, 256);
  L->off_dsum = off;
  off = align_up(off + rows * 4, 256);
  L->off_accum = off;
  const size_t blocks = (size_t)B * H * (size_t)((Sq + 63) / 64) * (size_t)((L->Dp + 127) / 128);
  const size_t accum = blocks * 32768u;
  off += accum;
  L->off_sems = off;
  const size_t sems = align_up(blocks * 4, 16);  // ordering counters (deterministic mode)
  off += sems;
  L->accum_bytes = accum;
  L->sems_bytes = sems;
  L->total = align_up(off, 256);
  return true;
}

// Packed sequences: per head T = total_q / 128 + batch slots of 128 query rows (each
// sequence's query tiles take consecutive slots; fa_tiles.h), with the same regions as
// the batched layout.
bool bwd_layout_varlen(int batch, int H, int total_q, int D, BwdLayout* L) {
  if (batch < 0 || H <= 0 || total_q < 0 || D <= 0) return false;
  L->Dp = padded_dim(D);
  const size_t T = (size_t)slot_count(total_q, batch);
  L->Mb = 0;
  L->Sq_r = 0;
  const size_t rows = (size_t)H * T * kTileQ;
  size_t off = WS_HEADER_BYTES;
  L->off_lse2 = off;
  off = align_up(off + rows * 4, 256);
  L->off_dsum = off;
  off = align_up(off + rows * 4, 256);
  L->off_accum = off;
  const size_t accum = rows * L->Dp * 4;
  off += accum;
  L->off_sems = off;
  const size_t sems = align_up((size_t)H * T * 4, 16);
  off += sems;
  L->accum_bytes = accum;
  L->sems_bytes = sems;
  L->total = align_up(off, 256);
  return true;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Packed-sequence arguments of the varlen entry points.
struct VarlenArgs {
  const int* cu_q;
  const int* cu_k;
  const int* used_q;  // optional per-sequence used lengths (null: the whole range)
  const int* used_k;
  int batch, max_q, max_k;
};

// A (B, S, H, D) view of 16-bit elements of type `dtype` (FA_DTYPE_BF16 or FA_DTYPE_F16).
int check_h16_4d(const fa_tensor* t, int dtype, int64_t d0, int64_t d1, int64_t d2, int64_t d3) {
  if (!t) return FA_ERR_NULL;
  if (t->ndim != 4) return FA_ERR_SHAPE;
  if (t->dtype != dtype) return FA_ERR_DTYPE;
  if (t->shape[0] != d0 || t->shape[1] != d1 || t->shape[2] != d2 || t->shape[3] != d3)
    return FA_ERR_SHAPE;
  if (t->stride[3] != 1) return FA_ERR_LAYOUT;
  const int64_t numel = d0 * d1 * d2 * d3;
  if (numel > 0 && !t->data) return FA_ERR_NULL;
  if (numel > 0) {
    if (!is_aligned16(t->data)) return FA_ERR_ALIGNMENT;
    for (int i = 0; i < 3; ++i)
      if (t->shape[i] > 1 && (t->stride[i] % 8 != 0 || t->stride[i] <= 0)) return FA_ERR_ALIGNMENT;
  }
  return FA_OK;
}

int check_lse(const fa_tensor* t, int64_t B, int64_t H, int64_t Sq) {
  if (!t) return FA_ERR_NULL;
  if (t->ndim != 3) return FA_ERR_SHAPE;
  if (t->dtype != FA_DTYPE_FP32) return FA_ERR_DTYPE;
  if (t->shape[0] != B || t->shape[1] != H || t->shape[2] != Sq) return FA_ERR_SHAPE;
  if (B * H * Sq > 0 && !t->data) return FA_ERR_NULL;
  return FA_OK;
}

// Shapes shared by fa_fwd and fa_bwd.  Returns a status; fills the problem sizes: D is
// the head dim of q and k, Dv the one of v (the `flash_bwd_sm90.py` page's `head_dim` and
// `head_dim_v`).  Also returns the shared 16-bit element type of q, k and v in *dtype.
int check_qkv(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, int* B, int* Sq,
              int* Sk, int* H, int* Hk, int* D, int* Dv, int* dtype) {
  if (!q || !k || !v) return FA_ERR_NULL;
  if (q->ndim != 4 || k->ndim != 4 || v->ndim != 4) return FA_ERR_SHAPE;
  if (q->dtype != FA_DTYPE_BF16 && q->dtype != FA_DTYPE_F16) return FA_ERR_DTYPE;
  if (k->dtype != q->dtype || v->dtype != q->dtype) return FA_ERR_DTYPE;
  const int64_t b = q->shape[0], sq = q->shape[1], h = q->shape[2], d = q->shape[3];
  const int64_t sk = k->shape[1], hk = k->shape[2], dv = v->shape[3];
  if (b < 0 || sq < 0 || sk < 0 || h <= 0 || hk <= 0 || d <= 0 || dv <= 0) return FA_ERR_SHAPE;
  if (k->shape[0] != b || k->shape[3] != d) return FA_ERR_SHAPE;
  for (int i = 0; i < 3; ++i)
    if (v->shape[i] != k->shape[i]) return FA_ERR_SHAPE;
  if (h % hk != 0) return FA_ERR_SHAPE;
  if (d % 8 != 0 || d > 256 || dv % 8 != 0 || dv > 256) return FA_ERR_HEADDIM;
  // launch-grid limits: the forward's grid has B in z and H in y (each at most 65535)
  if (b > 65535 || sq > (1 << 30) || sk > (1 << 30) || h > 65535) return FA_ERR_UNSUPPORTED;
  int st = check_h16_4d(q, q->dtype, b, sq, h, d);
  if (st) return st;
  st = check_h16_4d(k, q->dtype, b, sk, hk, d);
  if (st) return st;
  st = check_h16_4d(v, q->dtype, b, sk, hk, dv);
  if (st) return st;
  *dtype = q->dtype;
  *B = (int)b;
  *Sq = (int)sq;
  *Sk = (int)sk;
  *H = (int)h;
  *Hk = (int)hk;
  *D = (int)d;
  *Dv = (int)dv;
  return FA_OK;
}

// Head dims the 128-wide kernels take (one dim for q, k and v, at most 128); every other
// valid pair goes to the wide kernels of fa_wide.cu.
bool is_wide(int D, int Dv) { return D != Dv || D > 128; }

int check_scalars(float scale, float softcap) {
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_ARG;
  if (!(softcap >= 0.f) || !isfinite(softcap)) return FA_ERR_ARG;
  return FA_OK;
}

void mask_bounds(int Sq, int Sk, int causal, int wl, int wr, long long* lo, long long* hi) {
  MaskGeom g = make_geom(Sq, Sk, causal, wl, wr, kTileQ, kTileK);
  *lo = g.lo;
  *hi = g.hi;
}

int clamp30(long long x) {
  const long long lim = 1ll << 30;
  return (int)(x < -lim ? -lim : (x > lim ? lim : x));
}

// A packed (total, H, D) tensor of a variable-length call as a (1, total, H, D) view, and
// a (H, total) LSE as (1, H, total): the batched validation and tensor-map code then
// apply unchanged, with the sequence offsets added to the row coordinate.
int packed_view(const fa_tensor* t, int want_ndim, fa_tensor* out) {
  if (!t) return FA_ERR_NULL;
  if (t->ndim != want_ndim) return FA_ERR_SHAPE;
  memset(out, 0, sizeof(*out));
  out->data = t->data;
  out->dtype = t->dtype;
  out->ndim = want_ndim + 1;
  out->shape[0] = 1;
  out->stride[0] = t->shape[0] * t->stride[0];
  for (int d = 0; d < want_ndim; ++d) {
    out->shape[d + 1] = t->shape[d];
    out->stride[d + 1] = t->stride[d];
  }
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Tensor map over a bf16 or f16 (B, S, H, D) operand, box = (width, 1, rows, 1) at
// 128B/64B/32B swizzle.  Out-of-range rows and columns (S tail, D padding) read as zero.
bool encode_operand(CUtensorMap* map, const fa_tensor* t, int width, int rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)t->shape[3], (cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1],
                        (cuuint64_t)t->shape[0]};
  cuuint64_t strides[3] = {(cuuint64_t)(t->shape[2] > 1 ? t->stride[2] : t->shape[3]) * 2,
                           (cuuint64_t)(t->shape[1] > 1 ? t->stride[1] : t->shape[3]) * 2,
                           (cuuint64_t)(t->shape[0] > 1 ? t->stride[0] : t->shape[3]) * 2};
  cuuint32_t box[4] = {(cuuint32_t)width, 1, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMapSwizzle swz = width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                       : (width == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_32B);
  const CUtensorMapDataType ty =
      t->dtype == FA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(map, ty, 4, t->data, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_pair(OperandMaps* m, const fa_tensor* t, int Dp, int rows = 128) {
  memset(m, 0, sizeof(*m));
  if (!encode_operand(&m->full, t, 64, rows)) return false;
  const int tail = Dp % 64;
  if (tail) return encode_operand(&m->tail, t, tail, rows);
  m->tail = m->full;
  return true;
}

}  // namespace

extern "C" {

int fa_abi_version(void) { return FA_ABI_VERSION; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_NULL: return "FA_ERR_NULL: a required pointer is NULL";
    case FA_ERR_SHAPE: return "FA_ERR_SHAPE: tensor shapes do not match";
    case FA_ERR_DTYPE: return "FA_ERR_DTYPE: unsupported dtype";
    case FA_ERR_HEADDIM: return "FA_ERR_HEADDIM: head dims must be multiples of 8 and <= 256";
    case FA_ERR_LAYOUT: return "FA_ERR_LAYOUT: last dimension must be contiguous";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT: base or stride not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: outside what this build implements";
    case FA_ERR_ARG: return "FA_ERR_ARG: invalid scalar argument";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call or launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    default: return "unknown fa status";
  }
}

size_t fa_fwd_workspace_size(int B, int H, int Hk, int Sq, int Sk, int D) {
  (void)B; (void)H; (void)Hk; (void)Sq; (void)Sk; (void)D;
  return 0;
}

// The batched forward; block_mask (null = dense) is the (B, H, Mb, Nb) tile mask.
static int fwd_common(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, fa_tensor* out,
                      fa_tensor* lse, float softmax_scale, int causal, int window_left,
                      int window_right, float softcap, void* workspace, size_t workspace_bytes,
                      void* stream, const uint8_t* block_mask) {
  int B, Sq, Sk, H, Hk, D, Dv, dt;
  int st = check_qkv(q, k, v, &B, &Sq, &Sk, &H, &Hk, &D, &Dv, &dt);
  if (st) return st;
  if ((st = check_h16_4d(out, dt, B, Sq, H, Dv))) return st;
  if ((st = check_lse(lse, B, H, Sq))) return st;
  if ((st = check_scalars(softmax_scale, softcap))) return st;
  const bool wide = is_wide(D, Dv);
  if (wide && block_mask) return FA_ERR_UNSUPPORTED;  // block sparsity: 128-wide kernels only
  if (B == 0 || Sq == 0) return FA_OK;
  long long lo, hi;
  mask_bounds(Sq, Sk, causal, window_left, window_right, &lo, &hi);
  const int* status = (workspace && workspace_bytes >= WS_HEADER_BYTES && is_aligned16(workspace))
                          ? (int*)workspace + WS_STATUS
                          : nullptr;
  const cudaStream_t s = (cudaStream_t)stream;
  if (wide && Sk > 0) {
    WideParams w;
    memset(&w, 0, sizeof(w));
    w.B = B; w.H = H; w.Hk = Hk; w.G = H / Hk; w.Sq = Sq; w.Sk = Sk;
    w.Dk = D; w.Dv = Dv; w.DPK = pad64(D); w.DPV = pad64(Dv);
    w.Mb = (Sq + kTileQ - 1) / kTileQ;
    w.Nb = (Sk + kTileK - 1) / kTileK;
    w.lo64 = lo; w.hi64 = hi; w.lo = clamp30(lo); w.hi = clamp30(hi);
    w.scale_log2 = softmax_scale * kLog2e;
    w.cap_scale = softcap > 0.f ? softmax_scale / softcap : 0.f;
    w.cap_log2 = softcap * kLog2e;
    w.o = out->data;
    w.o_sb = out->stride[0]; w.o_ss = out->stride[1]; w.o_sh = out->stride[2];
    w.lse = (float*)lse->data;
    w.lse_sb = lse->stride[0]; w.lse_sh = lse->stride[1]; w.lse_ss = lse->stride[2];
    w.status = const_cast<int*>(status);
    w.wait_limit = g_wait_limit;
    CUtensorMap mq, mk, mv;
    if (!encode_operand(&mq, q, 64) || !encode_operand(&mk, k, 64) || !encode_operand(&mv, v, 64))
      return FA_ERR_CUDA;
    return launch_fwd_wide(w, mq, mk, mv, softcap > 0.f, dt == FA_DTYPE_F16, s) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
  }
  FwdTcParams p;
  memset(&p, 0, sizeof(p));
  p.B = B; p.H = H; p.Hk = Hk; p.G = H / Hk; p.Sq = Sq; p.Sk = Sk; p.D = Dv;
  p.Mb = (Sq + kTileQ - 1) / kTileQ;
  p.Nb = (Sk + kTileK - 1) / kTileK;
  p.lo64 = lo;
  p.hi64 = hi;
  p.lo = clamp30(lo);
  p.hi = clamp30(hi);
  p.scale_log2 = softmax_scale * kLog2e;
  p.cap_scale = softcap > 0.f ? softmax_scale / softcap : 0.f;
  p.cap_log2 = softcap * kLog2e;
  p.o = out->data;
  p.o_sb = out->stride[0]; p.o_ss = out->stride[1]; p.o_sh = out->stride[2];
  p.lse = (float*)lse->data;
  p.lse_sb = lse->stride[0]; p.lse_sh = lse->stride[1]; p.lse_ss = lse->stride[2];
  // optional workspace: its status word receives a device timeout (read with fa_bwd_status)
  p.status = const_cast<int*>(status);
  p.wait_limit = g_wait_limit;
  p.block_mask = block_mask;
  if (Sk == 0)  // no key: O = 0 and LSE = +inf (tensor maps need a non-empty key extent)
    return launch_fwd_empty(p, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  // tcgen05 kernel: one CTA per (128-query tile, batch, q-head)
  const int Dp = padded_dim(D);
  OperandMaps mq, mk, mv, mo;
  if (!encode_pair(&mq, q, Dp) || !encode_pair(&mk, k, Dp) || !encode_pair(&mv, v, Dp))
    return FA_ERR_CUDA;
  // O leaves through tensor copies where its layout has tensor maps; else row stores
  p.tma_epilogue = encode_pair(&mo, out, Dp, 32) ? 1 : 0;
  if (launch_fwd_tc(p, mq, mk, mv, mo, Dp, softcap > 0.f, dt == FA_DTYPE_F16, s) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

int fa_fwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, fa_tensor* out,
           fa_tensor* lse, float softmax_scale, int causal, int window_left, int window_right,
           float softcap, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_common(q, k, v, out, lse, softmax_scale, causal, window_left, window_right, softcap,
                    workspace, workspace_bytes, stream, nullptr);
}

int fa_fwd_blocksparse(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                       fa_tensor* out, fa_tensor* lse, const uint8_t* block_mask,
                       float softmax_scale, int causal, int window_left, int window_right,
                       float softcap, void* workspace, size_t workspace_bytes, void* stream) {
  if (!block_mask) return FA_ERR_NULL;
  return fwd_common(q, k, v, out, lse, softmax_scale, causal, window_left, window_right, softcap,
                    workspace, workspace_bytes, stream, block_mask);
}

int fa_fwd_varlen(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, fa_tensor* out,
                  fa_tensor* lse, const int* cu_seqlens_q, const int* cu_seqlens_k,
                  const int* seqused_q, const int* seqused_k, int batch,
                  int max_seqlen_q, int max_seqlen_k, float softmax_scale, int causal,
                  int window_left, int window_right, float softcap, void* workspace,
                  size_t workspace_bytes, void* stream) {
  fa_tensor q4, k4, v4, o4, l3;
  int st;
  if ((st = packed_view(q, 3, &q4)) || (st = packed_view(k, 3, &k4)) || (st = packed_view(v, 3, &v4)) ||
      (st = packed_view(out, 3, &o4)) || (st = packed_view(lse, 2, &l3)))
    return st;
  int B1, Tq, Tk, H, Hk, D, Dv, dt;
  if ((st = check_qkv(&q4, &k4, &v4, &B1, &Tq, &Tk, &H, &Hk, &D, &Dv, &dt))) return st;
  if (is_wide(D, Dv)) return FA_ERR_UNSUPPORTED;  // packed sequences: 128-wide kernels only
  if ((st = check_h16_4d(&o4, dt, 1, Tq, H, D))) return st;
  if ((st = check_lse(&l3, 1, H, Tq))) return st;
  if ((st = check_scalars(softmax_scale, softcap))) return st;
  if (batch < 0 || batch > 65535) return batch < 0 ? FA_ERR_ARG : FA_ERR_UNSUPPORTED;
  if (max_seqlen_q < 0 || max_seqlen_k < 0 || max_seqlen_q > Tq || max_seqlen_k > Tk)
    return FA_ERR_ARG;
  if (batch == 0 || Tq == 0 || max_seqlen_q == 0) return FA_OK;
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULL;
  FwdTcParams p;
  memset(&p, 0, sizeof(p));
  p.B = batch; p.H = H; p.Hk = Hk; p.G = H / Hk; p.D = D;
  p.Sq = max_seqlen_q; p.Sk = max_seqlen_k;
  p.Mb = (max_seqlen_q + kTileQ - 1) / kTileQ;
  p.Nb = (max_seqlen_k + kTileK - 1) / kTileK;
  p.scale_log2 = softmax_scale * kLog2e;
  p.cap_scale = softcap > 0.f ? softmax_scale / softcap : 0.f;
  p.cap_log2 = softcap * kLog2e;
  p.o = o4.data;
  p.o_sb = o4.stride[0]; p.o_ss = o4.stride[1]; p.o_sh = o4.stride[2];
  p.lse = (float*)l3.data;
  p.lse_sb = l3.stride[0]; p.lse_sh = l3.stride[1]; p.lse_ss = l3.stride[2];
  p.status = (workspace && workspace_bytes >= WS_HEADER_BYTES && is_aligned16(workspace))
                 ? (int*)workspace + WS_STATUS
                 : nullptr;
  p.wait_limit = g_wait_limit;
  p.varlen = 1;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.used_q = seqused_q;
  p.used_k = seqused_k;
  p.total_q = Tq;
  p.total_k = Tk;
  p.causal = causal ? 1 : 0;
  p.window_left = window_left;
  p.window_right = window_right;
  const cudaStream_t s = (cudaStream_t)stream;
  if (Tk == 0 || max_seqlen_k == 0) {  // no sequence has a key: O = 0, LSE = +inf
    FwdTcParams e = p;
    e.B = 1; e.Sq = Tq;
    e.o_sb = 0; e.lse_sb = 0;
    return launch_fwd_empty(e, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  const int Dp = padded_dim(D);
  OperandMaps mq, mk, mv, mo;
  if (!encode_pair(&mq, &q4, Dp) || !encode_pair(&mk, &k4, Dp) || !encode_pair(&mv, &v4, Dp))
    return FA_ERR_CUDA;
  p.tma_epilogue = encode_pair(&mo, &o4, Dp, 32) ? 1 : 0;
  if (launch_fwd_tc(p, mq, mk, mv, mo, Dp, softcap > 0.f, dt == FA_DTYPE_F16, s) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

size_t fa_bwd_workspace_size(int B, int H, int Hk, int Sq, int Sk, int D, int deterministic) {
  return fa_bwd_workspace_size_dv(B, H, Hk, Sq, Sk, D, D, deterministic);
}

size_t fa_bwd_workspace_size_dv(int B, int H, int Hk, int Sq, int Sk, int D, int Dv,
                                int deterministic) {
  (void)Hk; (void)Sk; (void)deterministic;
  BwdLayout L;
  if (Dv <= 0) return 0;
  if (is_wide(D, Dv) ? !bwd_layout_wide(B, H, Sq, D, &L) : !bwd_layout(B, H, Sq, D, &L)) return 0;
  return L.total;
}

// The backward for head dims above 128 or Dv != D: preprocess (D over Dv columns), the
// wide main kernel, and the convert of its transposed dQ blocks.  Batched, dense calls
// (the caller has checked that).
static int bwd_wide(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                    const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse, fa_tensor* dq,
                    fa_tensor* dk, fa_tensor* dv, int B, int H, int Hk, int Sq, int Sk, int D,
                    int Dv, bool f16, float softmax_scale, int causal, int window_left,
                    int window_right, float softcap, int deterministic, void* workspace,
                    size_t workspace_bytes, cudaStream_t s) {
  BwdLayout L;
  if (!bwd_layout_wide(B, H, Sq, D, &L)) return FA_ERR_SHAPE;
  if (!workspace || workspace_bytes < L.total) return FA_ERR_WORKSPACE;
  if (!is_aligned16(workspace)) return FA_ERR_ALIGNMENT;
  uint8_t* ws = (uint8_t*)workspace;
  long long lo, hi;
  mask_bounds(Sq, Sk, causal, window_left, window_right, &lo, &hi);

  BwdPreParams pre;
  memset(&pre, 0, sizeof(pre));
  pre.dout = (const __nv_bfloat16*)dout->data;
  pre.out = (const __nv_bfloat16*)out->data;
  pre.lse = (const float*)lse->data;
  pre.do_sb = dout->stride[0]; pre.do_ss = dout->stride[1]; pre.do_sh = dout->stride[2];
  pre.o_sb = out->stride[0]; pre.o_ss = out->stride[1]; pre.o_sh = out->stride[2];
  pre.lse_sb = lse->stride[0]; pre.lse_sh = lse->stride[1]; pre.lse_ss = lse->stride[2];
  pre.B = B; pre.H = H; pre.Sq = Sq; pre.Sq_r = L.Sq_r; pre.D = Dv;
  pre.lse2 = (float*)(ws + L.off_lse2);
  pre.dsum = (float*)(ws + L.off_dsum);
  // the accumulator and the counters are adjacent and cleared together
  pre.zero_ptr = (float4*)(ws + L.off_accum);
  pre.zero_count = (int64_t)((L.accum_bytes + L.sems_bytes) / 16);
  pre.header = (int*)ws;
  prof_record(0, s);
  if (launch_bwd_preprocess(pre, f16, s) != cudaSuccess) return FA_ERR_CUDA;
  if (g_poison_first_counter && deterministic) {
    const int poison = -1000000;
    if (cudaMemcpyAsync(ws + L.off_sems, &poison, sizeof(int), cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return FA_ERR_CUDA;
  }

  WideParams w;
  memset(&w, 0, sizeof(w));
  w.B = B; w.H = H; w.Hk = Hk; w.G = H / Hk; w.Sq = Sq; w.Sk = Sk;
  w.Dk = D; w.Dv = Dv; w.DPK = pad64(D); w.DPV = pad64(Dv);
  w.Mb = (Sq + 63) / 64;
  w.Nb = (Sk + kTileK - 1) / kTileK;
  w.nks = (w.DPK + 127) / 128;
  const int nvs = (w.DPV + 127) / 128;
  w.nslice = w.nks > nvs ? w.nks : nvs;
  w.lo64 = lo; w.hi64 = hi; w.lo = clamp30(lo); w.hi = clamp30(hi);
  w.scale_log2 = softmax_scale * kLog2e;
  w.cap_scale = softcap > 0.f ? softmax_scale / softcap : 0.f;
  w.cap_log2 = softcap * kLog2e;
  w.dk_scale = softmax_scale;
  w.scale = softmax_scale;
  w.lse2 = (const float*)(ws + L.off_lse2);
  w.dsum = (const float*)(ws + L.off_dsum);
  w.Sq_r = L.Sq_r;
  w.dq_accum = (float*)(ws + L.off_accum);
  w.dk = dk->data; w.dv = dv->data; w.dq = dq->data;
  w.dk_sb = dk->stride[0]; w.dk_ss = dk->stride[1]; w.dk_sh = dk->stride[2];
  w.dv_sb = dv->stride[0]; w.dv_ss = dv->stride[1]; w.dv_sh = dv->stride[2];
  w.dq_sb = dq->stride[0]; w.dq_ss = dq->stride[1]; w.dq_sh = dq->stride[2];
  w.status = (int*)ws + WS_STATUS;
  w.wait_limit = g_wait_limit;
  w.deterministic = deterministic ? 1 : 0;
  w.ticket = (int*)ws + WS_TICKET;
  w.sems = (int*)(ws + L.off_sems);
  prof_record(1, s);
  if (Sk > 0) {
    CUtensorMap mq, mk, mv, mdo;
    if (!encode_operand(&mq, q, 64, 64) || !encode_operand(&mk, k, 64) ||
        !encode_operand(&mv, v, 64) || !encode_operand(&mdo, dout, 64, 64))
      return FA_ERR_CUDA;
    if (launch_bwd_wide(w, mq, mk, mv, mdo, softcap > 0.f, f16, s) != cudaSuccess) return FA_ERR_CUDA;
  }
  prof_record(2, s);
  if (launch_convert_wide(w, f16, s) != cudaSuccess) return FA_ERR_CUDA;
  prof_record(3, s);
  return FA_OK;
}

// The backward for a batch (vl == nullptr) or for packed sequences (vl: the tensors are
// (1, total, H, D) views and LSE a (1, H, total_q) view).
static int bwd_common(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                      const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse,
                      fa_tensor* dq, fa_tensor* dk, fa_tensor* dv, float softmax_scale, int causal,
                      int window_left, int window_right, float softcap, int deterministic,
                      void* workspace, size_t workspace_bytes, void* stream,
                      const VarlenArgs* vl, const uint8_t* block_mask) {
  int B, Sq, Sk, H, Hk, D, Dv, dt;
  int st = check_qkv(q, k, v, &B, &Sq, &Sk, &H, &Hk, &D, &Dv, &dt);
  if (st) return st;
  if ((st = check_h16_4d(dout, dt, B, Sq, H, Dv))) return st;
  if ((st = check_h16_4d(out, dt, B, Sq, H, Dv))) return st;
  if ((st = check_h16_4d(dq, dt, B, Sq, H, D))) return st;
  if ((st = check_h16_4d(dk, dt, B, Sk, Hk, D))) return st;
  if ((st = check_h16_4d(dv, dt, B, Sk, Hk, Dv))) return st;
  const bool f16 = dt == FA_DTYPE_F16;
  // The algorithm of this call.  AUTO: the split algorithm for deterministic batched bf16
  // calls on a square shape (its two kernels never wait; on square causal and windowed
  // shapes the fused ordered mode is slower, since deadlock freedom makes it claim the
  // short key tiles first), the fused one otherwise (rectangular shapes, whose few query
  // tiles per key tile make the split algorithm's recomputation costly).
  int algo = g_bwd_algorithm;
  if (algo == FA_BWD_ALGO_AUTO) {
    algo = (deterministic && !f16 && !vl && !block_mask && Sq == Sk) ? FA_BWD_ALGO_SPLIT
                                                                   : FA_BWD_ALGO_FUSED;
  }
  if (is_wide(D, Dv)) {
    // the wide kernels: batched and dense calls only, whichever algorithm is selected
    if (vl || block_mask) return FA_ERR_UNSUPPORTED;
    if ((st = check_lse(lse, B, H, Sq))) return st;
    if ((st = check_scalars(softmax_scale, softcap))) return st;
    if (B == 0 || Sq == 0) return FA_OK;
    return bwd_wide(dout, q, k, v, out, lse, dq, dk, dv, B, H, Hk, Sq, Sk, D, Dv, f16,
                    softmax_scale, causal, window_left, window_right, softcap, deterministic,
                    workspace, workspace_bytes, (cudaStream_t)stream);
  }
  // the split algorithm is built for batched dense bf16 only; block sparsity has no ordered
  // (deterministic) mode
  if ((f16 || vl || block_mask) && algo == FA_BWD_ALGO_SPLIT) return FA_ERR_UNSUPPORTED;
  if ((st = check_lse(lse, B, H, Sq))) return st;
  if ((st = check_scalars(softmax_scale, softcap))) return st;
  const int total_q = Sq, total_k = Sk;  // packed: the row extents of the views
  if (vl) {
    if (vl->batch < 0 || vl->max_q < 0 || vl->max_k < 0 || vl->max_q > total_q ||
        vl->max_k > total_k)
      return FA_ERR_ARG;
    if (vl->batch > 65535) return FA_ERR_UNSUPPORTED;
    if (vl->batch == 0 || total_q == 0 || vl->max_q == 0) return FA_OK;
    if (!vl->cu_q || !vl->cu_k) return FA_ERR_NULL;
    B = vl->batch;
    Sq = vl->max_q;
    Sk = vl->max_k;
  }
  if (B == 0 || Sq == 0) return FA_OK;
  BwdLayout L;
  if (vl ? !bwd_layout_varlen(B, H, total_q, D, &L) : !bwd_layout(B, H, Sq, D, &L))
    return FA_ERR_SHAPE;
  if (vl) L.Mb = (Sq + kTileQ - 1) / kTileQ;  // query tiles of the longest sequence
  const long long T = vl ? slot_count(total_q, B) : 0;
  // block sparsity: per key-tile ticket a step count and a list of G * Mb entries after
  // the regular regions
  const int Nb_all = (Sk + kTileK - 1) / kTileK;
  size_t off_sp_counts = 0, off_sp_lists = 0;
  if (block_mask) {
    if (L.Mb > 65535) return FA_ERR_UNSUPPORTED;  // list entries hold the query tile in 16 bits
    const size_t tiles = (size_t)Nb_all * B * Hk;
    off_sp_counts = L.total;
    off_sp_lists = align_up(off_sp_counts + tiles * 4, 256);
    L.total = align_up(off_sp_lists + tiles * (size_t)(H / Hk) * L.Mb * 4, 256);
  }
  if (!workspace || workspace_bytes < L.total) return FA_ERR_WORKSPACE;
  if (!is_aligned16(workspace)) return FA_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;

  long long lo, hi;
  mask_bounds(Sq, Sk, causal, window_left, window_right, &lo, &hi);
  const int Dp = L.Dp;
  // The split algorithm needs key tiles to build its tensor maps; with Sk == 0 (every dQ
  // row is zero, dK/dV are empty) the fused path's convert writes the zero dQ.
  const bool split = algo == FA_BWD_ALGO_SPLIT && Sk > 0;

  BwdPreParams pre;
  memset(&pre, 0, sizeof(pre));
  pre.dout = (const __nv_bfloat16*)dout->data;
  pre.out = (const __nv_bfloat16*)out->data;
  pre.lse = (const float*)lse->data;
  pre.do_sb = dout->stride[0]; pre.do_ss = dout->stride[1]; pre.do_sh = dout->stride[2];
  pre.o_sb = out->stride[0]; pre.o_ss = out->stride[1]; pre.o_sh = out->stride[2];
  pre.lse_sb = lse->stride[0]; pre.lse_sh = lse->stride[1]; pre.lse_ss = lse->stride[2];
  pre.B = B; pre.H = H; pre.Sq = Sq; pre.Sq_r = L.Sq_r; pre.D = D;
  if (vl) {
    pre.varlen = 1;
    pre.cu_q = vl->cu_q;
    pre.used_q = vl->used_q;
    pre.total_q = total_q;
    pre.T = T;
  }
  pre.lse2 = (float*)(ws + L.off_lse2);
  pre.dsum = (float*)(ws + L.off_dsum);
  // the accumulator and the counters are adjacent and cleared together
  pre.zero_ptr = (float4*)(ws + L.off_accum);
  pre.zero_count = split ? 0 : (int64_t)((L.accum_bytes + L.sems_bytes) / 16);
  pre.header = (int*)ws;
  prof_record(0, s);
  if (launch_bwd_preprocess(pre, f16, s) != cudaSuccess) return FA_ERR_CUDA;
  if (g_poison_first_counter && deterministic) {
    const int poison = -1000000;
    if (cudaMemcpyAsync(ws + L.off_sems, &poison, sizeof(int), cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return FA_ERR_CUDA;
  }

  const int Nb = (Sk + kTileK - 1) / kTileK;
  const int num_ctas = Nb * B * Hk;
  prof_record(1, s);
  if (num_ctas > 0) {
    OperandMaps mq, mk, mv, mdo;
    if (!encode_pair(&mq, q, Dp) || !encode_pair(&mk, k, Dp) || !encode_pair(&mv, v, Dp) ||
        !encode_pair(&mdo, dout, Dp))
      return FA_ERR_CUDA;
    BwdMainParams p;
    memset(&p, 0, sizeof(p));
    p.B = B; p.H = H; p.Hk = Hk; p.G = H / Hk; p.Sq = Sq; p.Sk = Sk; p.D = D;
    p.Mb = L.Mb; p.Nb = Nb; p.Sq_r = L.Sq_r;
    p.num_tiles = num_ctas;
    p.lo = clamp30(lo);
    p.hi = clamp30(hi);
    p.lo64 = lo;
    p.hi64 = hi;
    p.scale_log2 = softmax_scale * kLog2e;
    p.cap_scale = softcap > 0.f ? softmax_scale / softcap : 0.f;
    p.cap_log2 = softcap * kLog2e;
    p.dk_scale = softmax_scale;
    p.deterministic = deterministic ? 1 : 0;
    p.lse2 = (const float*)(ws + L.off_lse2);
    p.dsum = (const float*)(ws + L.off_dsum);
    p.dq_accum = (float*)(ws + L.off_accum);
    p.sems = (int*)(ws + L.off_sems);
    p.status = (int*)ws + WS_STATUS;
    p.ticket = (int*)ws + WS_TICKET;
    p.dk = (__nv_bfloat16*)dk->data;
    p.dv = (__nv_bfloat16*)dv->data;
    p.dk_sb = dk->stride[0]; p.dk_ss = dk->stride[1]; p.dk_sh = dk->stride[2];
    p.dv_sb = dv->stride[0]; p.dv_ss = dv->stride[1]; p.dv_sh = dv->stride[2];
    p.ticket_dq = (int*)ws + WS_TICKET_DQ;
    p.dq = (__nv_bfloat16*)dq->data;
    p.dq_sb = dq->stride[0]; p.dq_ss = dq->stride[1]; p.dq_sh = dq->stride[2];
    p.wait_limit = g_wait_limit;
    if (vl) {
      p.cu_q = vl->cu_q;
      p.cu_k = vl->cu_k;
      p.used_q = vl->used_q;
      p.used_k = vl->used_k;
      p.total_q = total_q;
      p.total_k = total_k;
      p.T = T;
      p.causal = causal ? 1 : 0;
      p.window_left = window_left;
      p.window_right = window_right;
    }
    if (split) {
      if (launch_bwd_split(p, mq, mk, mv, mdo, Dp, softcap > 0.f, num_ctas, 0, s) != cudaSuccess)
        return FA_ERR_CUDA;
      prof_record(2, s);
      if (launch_bwd_split(p, mq, mk, mv, mdo, Dp, softcap > 0.f, 0, B * H * L.Mb, s) !=
          cudaSuccess)
        return FA_ERR_CUDA;
      prof_record(3, s);
      return FA_OK;
    }
    // persistent: one CTA per SM at most, each looping over key tiles
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    const int grid = num_ctas < sms ? num_ctas : sms;
    if (block_mask) {
      BwdSparseParams sp;
      memset(&sp, 0, sizeof(sp));
      sp.block_mask = block_mask;
      sp.B = B; sp.H = H; sp.Hk = Hk; sp.G = H / Hk; sp.Sq = Sq; sp.Sk = Sk;
      sp.Mb = L.Mb; sp.Nb = Nb;
      sp.lo64 = lo;
      sp.hi64 = hi;
      sp.counts = (int*)(ws + off_sp_counts);
      sp.lists = (int*)(ws + off_sp_lists);
      sp.stride = (long long)(H / Hk) * L.Mb;
      sp.num_tiles = num_ctas;
      sp.deterministic = deterministic ? 1 : 0;
      if (launch_bwd_sparse_lists(sp, s) != cudaSuccess) return FA_ERR_CUDA;
      p.sp_counts = sp.counts;
      p.sp_lists = sp.lists;
      p.block_mask = block_mask;
      p.sp_stride = sp.stride;
    }
    const int mode = vl ? 1 : (block_mask ? 2 : 0);
    // dK / dV leave through tensor copies where the outputs' layout has tensor maps (the
    // alignment checks above make that the rule); otherwise each thread stores its row
    OperandMaps mdk, mdv;
    p.tma_epilogue = encode_pair(&mdk, dk, Dp, 32) && encode_pair(&mdv, dv, Dp, 32) ? 1 : 0;
    // the main kernel overlaps the preprocess's tail when nothing else was enqueued between
    // them (block-sparse calls build their step lists in between; the counter-poisoning
    // test hook writes a counter)
    const bool pdl = !block_mask && !(g_poison_first_counter && deterministic);
    if (launch_bwd_main(p, mq, mk, mv, mdo, mdk, mdv, Dp, softcap > 0.f, f16, mode, grid, pdl,
                        s) != cudaSuccess)
      return FA_ERR_CUDA;
  }

  prof_record(2, s);
  BwdConvParams cp;
  memset(&cp, 0, sizeof(cp));
  cp.dq_accum = (const float*)(ws + L.off_accum);
  cp.dq = (__nv_bfloat16*)dq->data;
  cp.dq_sb = dq->stride[0]; cp.dq_ss = dq->stride[1]; cp.dq_sh = dq->stride[2];
  cp.B = B; cp.H = H; cp.Sq = Sq; cp.D = D; cp.Dp = Dp; cp.Mb = L.Mb;
  cp.scale = softmax_scale;
  if (vl) {
    cp.varlen = 1;
    cp.cu_q = vl->cu_q;
    cp.used_q = vl->used_q;
    cp.total_q = total_q;
    cp.T = T;
  }
  if (launch_bwd_convert(cp, f16, s) != cudaSuccess) return FA_ERR_CUDA;
  prof_record(3, s);
  return FA_OK;
}

int fa_bwd(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
           const fa_tensor* out, const fa_tensor* lse, fa_tensor* dq, fa_tensor* dk,
           fa_tensor* dv, float softmax_scale, int causal, int window_left, int window_right,
           float softcap, int deterministic, void* workspace, size_t workspace_bytes,
           void* stream) {
  return bwd_common(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, causal, window_left,
                    window_right, softcap, deterministic, workspace, workspace_bytes, stream,
                    nullptr, nullptr);
}

size_t fa_bwd_blocksparse_workspace_size(int B, int H, int Hk, int Sq, int Sk, int D) {
  BwdLayout L;
  if (Hk <= 0 || Sk < 0 || !bwd_layout(B, H, Sq, D, &L)) return 0;
  const size_t tiles = (size_t)((Sk + kTileK - 1) / kTileK) * B * Hk;
  const size_t lists = align_up(L.total + tiles * 4, 256);
  return align_up(lists + tiles * (size_t)(H / Hk) * L.Mb * 4, 256);
}

int fa_bwd_blocksparse(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                       const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse,
                       fa_tensor* dq, fa_tensor* dk, fa_tensor* dv, const uint8_t* block_mask,
                       float softmax_scale, int causal, int window_left, int window_right,
                       float softcap, int deterministic, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!block_mask) return FA_ERR_NULL;
  return bwd_common(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, causal, window_left,
                    window_right, softcap, deterministic, workspace, workspace_bytes, stream,
                    nullptr, block_mask);
}

size_t fa_bwd_varlen_workspace_size(int batch, int H, int total_q, int D, int deterministic) {
  (void)deterministic;
  BwdLayout L;
  if (!bwd_layout_varlen(batch, H, total_q, D, &L)) return 0;
  return L.total;
}

int fa_bwd_varlen(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                  const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse, fa_tensor* dq,
                  fa_tensor* dk, fa_tensor* dv, const int* cu_seqlens_q, const int* cu_seqlens_k,
                  const int* seqused_q, const int* seqused_k, int batch, int max_seqlen_q,
                  int max_seqlen_k, float softmax_scale, int causal,
                  int window_left, int window_right, float softcap, int deterministic,
                  void* workspace, size_t workspace_bytes, void* stream) {
  fa_tensor d4, q4, k4, v4, o4, l3, dq4, dk4, dv4;
  int st;
  if ((st = packed_view(dout, 3, &d4)) || (st = packed_view(q, 3, &q4)) ||
      (st = packed_view(k, 3, &k4)) || (st = packed_view(v, 3, &v4)) ||
      (st = packed_view(out, 3, &o4)) || (st = packed_view(lse, 2, &l3)) ||
      (st = packed_view(dq, 3, &dq4)) || (st = packed_view(dk, 3, &dk4)) ||
      (st = packed_view(dv, 3, &dv4)))
    return st;
  VarlenArgs vl{cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k, batch, max_seqlen_q,
                max_seqlen_k};
  return bwd_common(&d4, &q4, &k4, &v4, &o4, &l3, &dq4, &dk4, &dv4, softmax_scale, causal,
                    window_left, window_right, softcap, deterministic, workspace,
                    workspace_bytes, stream, &vl, nullptr);
}

int fa_bwd_status(void* workspace, void* stream, int* device_status) {
  if (!workspace || !device_status) return FA_ERR_NULL;
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  if (cudaMemcpyAsync(&v, (int*)workspace + WS_STATUS, sizeof(int), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyAsync((int*)workspace + WS_STATUS, &zero, sizeof(int), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  *device_status = v;
  return FA_OK;
}

int fa_bwd_set_algorithm(int algorithm) {
  if (algorithm != FA_BWD_ALGO_SPLIT && algorithm != FA_BWD_ALGO_FUSED &&
      algorithm != FA_BWD_ALGO_AUTO)
    return FA_ERR_ARG;
  g_bwd_algorithm = algorithm;
  return FA_OK;
}

int fa_bwd_get_algorithm(void) { return g_bwd_algorithm; }

int fa_debug_set_wait_limit(long long cycles) {
  if (cycles <= 0) return FA_ERR_ARG;
  g_wait_limit = cycles;
  return FA_OK;
}

int fa_debug_poison_ordering(int enable) {
  g_poison_first_counter = enable ? 1 : 0;
  return FA_OK;
}

#ifdef FA_TRACE
// Tracing builds only: copies the per-phase timestamps of the main kernel to the host.
int fa_trace_read(void* host, size_t bytes) {
  return bwd_trace_copy(host, bytes) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
int fa_trace_read_split(void* host, size_t bytes) {
  return split_trace_copy(host, bytes) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
int fa_trace_mma(void* host, size_t bytes) {
  return bwd_trace_mma_copy(host, bytes) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
int fa_trace_timeline(void* host, size_t bytes, int clear) {
  return bwd_timeline_copy(host, bytes, clear != 0) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
#endif

int fa_profile_enable(int enable) {
  if (enable) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (g_ev[0] && dev != g_profile_dev) {
      // events of another device: make new ones on this device
      int cur = dev;
      if (cudaSetDevice(g_profile_dev) == cudaSuccess) {
        for (int i = 0; i < 4; ++i) cudaEventDestroy(g_ev[i]);
      }
      cudaSetDevice(cur);
      for (int i = 0; i < 4; ++i) g_ev[i] = nullptr;
    }
    if (!g_ev[0]) {
      for (int i = 0; i < 4; ++i)
        if (cudaEventCreate(&g_ev[i]) != cudaSuccess) return FA_ERR_CUDA;
      g_profile_dev = dev;
    }
  }
  g_profile = enable != 0;
  return FA_OK;
}

int fa_profile_read(float* ms3) {
  if (!ms3) return FA_ERR_NULL;
  if (!g_ev[0]) return FA_ERR_ARG;
  if (cudaEventSynchronize(g_ev[3]) != cudaSuccess) return FA_ERR_CUDA;
  for (int i = 0; i < 3; ++i)
    if (cudaEventElapsedTime(&ms3[i], g_ev[i], g_ev[i + 1]) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
