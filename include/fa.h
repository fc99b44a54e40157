/*
 * fa.h — C ABI of the GB300 (sm_103a) FlashAttention forward/backward library.
 *
 * The operation is softmax attention and its gradient as traced on the
 * "FlashAttention backward call trace" page (`mha_bwd` signature, `softmax_d`,
 * in-place `dq, dk, dv`, GQA `sum_out`), the "Fused Attention (Flash Attention v2)"
 * Triton page (`_attn_fwd_inner`, `_bwd_kernel_dk/dv/dq`), the "GQA/MQA" page
 * (kv-head map, bottom-right causal block range) and the `flash_bwd_sm90.py` page
 * (`mma_one_m_block`: P = exp2(S*scale*log2e - LSE2), dS = P*(dP - dPsum)).
 *
 *   forward : O = softmax(mask(z)) V,  z = softcap>0 ? c*tanh(scale*QK^T/c) : scale*QK^T
 *             LSE_i = ln sum_j exp(z_ij)           (natural log; +inf for a row with no key)
 *   backward: D_i = sum_d dO_id O_id,  dZ = P*(dO V^T - D),  dA = dZ*(1 - tanh^2) (softcap),
 *             dV = P^T dO,  dK = scale dA^T Q,  dQ = scale dA K,
 *             dK/dV of kv-head hk summed over its H/Hk q-heads.
 *
 * Masking (bottom-right aligned, offset Sk - Sq): key j visible to query i iff
 *   j <= i + (Sk-Sq) + window_right  (window_right >= 0; causal forces window_right = 0) and
 *   j >= i + (Sk-Sq) - window_left   (window_left  >= 0).  Negative bounds are unbounded.
 *
 * Conventions shared by every entry point
 *   - Tensors are described by fa_tensor (element strides; the last dimension must
 *     have stride 1).  Q, O, dO, dQ: (B, Sq, H, D).  K, V, dK, dV: (B, Sk, Hk, D).
 *     LSE: (B, H, Sq) fp32.  Data type: bf16 for Q/K/V/O/dO/dQ/dK/dV.
 *   - Every pointer is device memory owned by the caller.  The library allocates
 *     nothing and frees nothing; scratch comes from the caller's workspace buffer.
 *   - Calls are asynchronous on `stream` (cudaStream_t passed as void*; NULL = the
 *     legacy default stream).  A return of FA_OK means "validated and enqueued".
 *   - All argument errors are detected on the host before any launch and leave the
 *     outputs untouched.  A device-side wait that runs out of time records
 *     FA_ERR_DEVICE_TIMEOUT in the workspace status word (see fa_bwd_status).
 *   - Head dims: q and k share D, v may have its own Dv (the `flash_bwd_sm90.py` page's
 *     `head_dim` / `head_dim_v`); O, dO and dV then have Dv columns.  D % 8 == 0,
 *     Dv % 8 == 0, both <= 256.  D == Dv <= 128 runs on the 128-wide kernels (padded
 *     inside to a multiple of 16); every other pair runs on the wide kernels (padded to
 *     a multiple of 64), which take batched, dense calls only (packed sequences and block
 *     masks return FA_ERR_UNSUPPORTED there).
 *   - Other limits: H % Hk == 0; base pointers 16-byte aligned; every non-unit stride a
 *     multiple of 8 elements (16 bytes).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 3

/* Element types.  Q, K, V, O, dO, dQ, dK and dV of one call share one 16-bit type:
 * bf16, or f16 (the call-trace page's dispatch covers both, `run_mha_bwd_constexpr`);
 * LSE is fp32. */
typedef enum {
    FA_DTYPE_BF16 = 0,
    FA_DTYPE_FP32 = 1,
    FA_DTYPE_F16 = 2
} fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = -1,          /* a required pointer is NULL                          */
    FA_ERR_SHAPE = -2,         /* mismatched dims, K/V mismatch, H % Hk != 0, ndim    */
    FA_ERR_DTYPE = -3,         /* tensors not all bf16 or all f16 / LSE not fp32      */
    FA_ERR_HEADDIM = -4,       /* D or Dv not a multiple of 8, or above 256           */
    FA_ERR_LAYOUT = -5,        /* last dimension not contiguous                       */
    FA_ERR_ALIGNMENT = -6,     /* base not 16-byte aligned or stride not 16-byte mult */
    FA_ERR_WORKSPACE = -7,     /* workspace NULL or smaller than the size query       */
    FA_ERR_UNSUPPORTED = -8,   /* outside what this build implements (B or H > 65535, */
                               /* S > 2^30, the split algorithm with f16)             */
    FA_ERR_ARG = -9,           /* invalid scalar (scale <= 0, softcap < 0, ...)       */
    FA_ERR_CUDA = -10,         /* a CUDA runtime/driver call or launch failed         */
    FA_ERR_DEVICE_TIMEOUT = -11 /* a bounded device-side wait gave up (status word)   */
} fa_status;

/* Strided view of a tensor.  `ndim` is 4 (B,S,H,D) or 3 (LSE: B,H,S).  shape and
 * stride are in elements; unused trailing entries are ignored. */
typedef struct {
    void* data;
    int64_t shape[4];
    int64_t stride[4];
    int32_t ndim;
    int32_t dtype; /* fa_dtype */
} fa_tensor;

/* Library/ABI version (FA_ABI_VERSION). */
int fa_abi_version(void);

/* Human-readable name of a status code (static storage; never NULL).  The library's own
 * helper: the pages raise Python / C++ exceptions instead of returning codes. */
const char* fa_status_string(int status);

/*
 * Workspace the forward needs, in bytes (0 for this build: the forward keeps its
 * statistics in registers and tensor memory and writes O and LSE directly).  A caller
 * may still pass a workspace of at least 256 bytes (16-byte aligned): a device-side wait
 * of the forward that runs out of time then records FA_ERR_DEVICE_TIMEOUT in its status
 * word, which fa_bwd_status reads and clears.  Without one, such a timeout only stops
 * the affected CTAs.
 */
size_t fa_fwd_workspace_size(int B, int H, int Hk, int Sq, int Sk, int D);

/*
 * fa_fwd — O (bf16, (B,Sq,H,D)) and natural-log LSE (fp32, (B,H,Sq)) from Q, K, V.
 * Defined by the Triton page's `_attn_fwd_inner`/`_attn_fwd_kernel` (online softmax,
 * LSE saved per row) with the mask/softcap conventions above.  `out` and `lse` are
 * written in place.  softmax_scale > 0 (callers normally pass 1/sqrt(D)).
 * Returns a fa_status.
 */
int fa_fwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
           fa_tensor* out, fa_tensor* lse,
           float softmax_scale, int causal, int window_left, int window_right,
           float softcap, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_varlen — the forward over a batch of packed sequences of different lengths
 * (the Triton page's `flash_attn_varlen_func` / `set_varlen_params`: cu_seqlens_q,
 * cu_seqlens_k, max_seqlen_q, max_seqlen_k).  Sequence b owns rows
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q / out and [cu_seqlens_k[b], cu_seqlens_k[b+1])
 * of k / v, and is computed exactly as a batch of one of that length (the mask is
 * bottom-right aligned per sequence).
 *   q, out (total_q, H, D) and k, v (total_k, Hk, D): ndim 3, same 16-bit type;
 *   lse (H, total_q) fp32, natural log (+inf for a row with no visible key);
 *   cu_seqlens_q / cu_seqlens_k: DEVICE int32 arrays of batch + 1 non-decreasing offsets
 *     starting at 0 (caller-owned; read by the kernels, not by the host);
 *   seqused_q / seqused_k: NULL, or DEVICE int32 arrays of batch used lengths (the
 *     optional `mSeqUsedQ` / `mSeqUsedK` kernel arguments of the `flash_bwd_sm90.py`
 *     page, whose meaning it leaves unstated): sequence b then computes only
 *     the first seqused_q[b] query rows and seqused_k[b] key rows of its range (each
 *     clamped into [0, the range's length]), as a batch of one of those lengths; the rows
 *     after them are padding.  Padding rows of out and lse are not written.  They are
 *     read as part of a sequence's last 128-row tile, where their contribution is exactly
 *     zero, so they must hold finite values (zeros, for instance);
 *   max_seqlen_q / max_seqlen_k: at least the longest sequence (rows of a longer one are
 *     not computed) and at most total_q / total_k.
 * Offsets outside [0, total] are clamped into the tensors, so malformed offsets cannot
 * make the kernels access memory outside them (their results are then undefined).  With
 * no key at all (total_k == 0 or max_seqlen_k == 0) every row of out is 0 and every lse
 * row +inf, padding included.
 * batch == 0, total_q == 0 or max_seqlen_q == 0 returns FA_OK without a launch.  Errors
 * as fa_fwd, plus FA_ERR_ARG for batch < 0 or max lengths outside [0, total] and
 * FA_ERR_UNSUPPORTED for batch > 65535.
 */
int fa_fwd_varlen(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                  fa_tensor* out, fa_tensor* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k,
                  const int* seqused_q, const int* seqused_k, int batch,
                  int max_seqlen_q, int max_seqlen_k,
                  float softmax_scale, int causal, int window_left, int window_right,
                  float softcap, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace the backward needs, in bytes, for the given problem.  It holds what the
 * call-trace page's `mha_bwd` allocates for itself before `run_mha_bwd` (the fp32
 * `dq_accum` and `softmax_d` = rowsum(dO*O)), plus the LSE in log2 units that the
 * `flash_bwd_sm90.py` page's kernel consumes, the deterministic-mode ordering counters
 * (its `mdQ_semaphore`) and a status word.  Here the caller allocates it and passes it to
 * fa_bwd.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int Hk, int Sq, int Sk, int D, int deterministic);

/*
 * The same for a call whose v has its own head dim Dv (q / k: D); equal to
 * fa_bwd_workspace_size when Dv == D.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size_dv(int B, int H, int Hk, int Sq, int Sk, int D, int Dv,
                                int deterministic);

/*
 * fa_bwd — dQ (B,Sq,H,D), dK (B,Sk,Hk,D) and dV (B,Sk,Hk,Dv), written in place (the call-trace
 * page's `_flash_attn_backward` mutates dq, dk, dv).  Inputs: dout, q, k, v, out and the
 * forward's natural-log lse.  dropout is not supported (p = 0).
 *
 * Two algorithms (see fa_bwd_set_algorithm), both hand-written tcgen05/TMEM/TMA kernels on
 * `stream`, after a preprocess kernel (D = rowsum(dO*O), LSE*log2e):
 *   FA_BWD_ALGO_SPLIT: a dK/dV kernel (one CTA per 128-key tile of one kv-head;
 *     recomputes P per 128-query tile; dK/dV accumulate in tensor memory over all q-heads
 *     of the kv-head, so the GQA reduction happens in-kernel) and a dQ kernel (persistent
 *     CTAs, at most one per SM, each claiming 128-query tiles of one q-head; recomputes P
 *     and dS over the tile's key tiles; dQ accumulates in tensor memory and is written once).  No atomics: every output is summed in a
 *     fixed order, so results are bitwise reproducible whatever `deterministic` says.
 *   FA_BWD_ALGO_FUSED (default): one kernel computes all five products per (key tile, query tile)
 *     and adds fp32 dQ partials into an accumulator in the workspace (bulk reductions),
 *     then a convert kernel writes dQ = bf16(scale * accumulator).  deterministic != 0
 *     orders the dQ additions by key tile through per-tile counters (bitwise
 *     reproducible); deterministic == 0 lets them land in any order.
 *
 * B == 0 or Sq == 0 returns FA_OK without launching (and, when Sk > 0 and Sq == 0,
 * without touching dK/dV).  Returns a fa_status.
 */
int fa_bwd(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
           const fa_tensor* out, const fa_tensor* lse,
           fa_tensor* dq, fa_tensor* dk, fa_tensor* dv,
           float softmax_scale, int causal, int window_left, int window_right, float softcap,
           int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-sparse attention (the `flash_bwd_sm90.py` page's `blocksparse_tensors`: each key
 * block visits only its listed query blocks).  block_mask: DEVICE bytes, contiguous
 * (B, H, ceil(Sq/128), ceil(Sk/128)); entry [b, h, m, n] != 0 keeps the pair (query rows
 * [128m, 128m+128), key rows [128n, 128n+128)) for q-head h, 0 removes it entirely, on
 * top of the causal / window mask.  A row left with no visible key gives O = 0, LSE =
 * +inf and dQ = 0, as elsewhere.  Forward and backward must get the same mask.
 *
 * fa_fwd_blocksparse: fa_fwd's arguments plus block_mask (NULL: FA_ERR_NULL).
 * fa_bwd_blocksparse: fa_bwd's arguments plus block_mask; the workspace must hold
 *   fa_bwd_blocksparse_workspace_size bytes (fa_bwd's regions plus, per key tile, a list
 *   of its kept (q-head, query tile) steps); the fused algorithm only
 *   (FA_ERR_UNSUPPORTED while the split one is selected or for more than 65535 query
 *   tiles).  deterministic != 0 adds the dQ contributions of the kept key tiles of a
 *   query tile in descending key-tile order, as fa_bwd's ordered mode does (bitwise
 *   reproducible).
 */
int fa_fwd_blocksparse(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                       fa_tensor* out, fa_tensor* lse, const uint8_t* block_mask,
                       float softmax_scale, int causal, int window_left, int window_right,
                       float softcap, void* workspace, size_t workspace_bytes, void* stream);
size_t fa_bwd_blocksparse_workspace_size(int B, int H, int Hk, int Sq, int Sk, int D);
int fa_bwd_blocksparse(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                       const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse,
                       fa_tensor* dq, fa_tensor* dk, fa_tensor* dv, const uint8_t* block_mask,
                       float softmax_scale, int causal, int window_left, int window_right,
                       float softcap, int deterministic, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Workspace of fa_bwd_varlen, in bytes: per q-head, total_q / 128 + batch tiles of 128
 * query rows (each sequence's query tiles are consecutive; the slack is at most one
 * partial tile per sequence) for the fp32 dQ accumulator, D and LSE2, plus counters and
 * the status word.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_varlen_workspace_size(int batch, int H, int total_q, int D, int deterministic);

/*
 * fa_bwd_varlen — the backward over packed sequences (the layouts and sequence offsets of
 * fa_fwd_varlen): dout, out, dq (total_q, H, D); k, v, dk, dv (total_k, Hk, D); lse
 * (H, total_q) fp32 natural log as fa_fwd_varlen writes it.  Every sequence is computed
 * exactly as a batch of one of its length (bottom-right aligned mask per sequence).  The
 * fused algorithm only (FA_ERR_UNSUPPORTED while the split one is selected); the
 * workspace must hold fa_bwd_varlen_workspace_size bytes.  Offset clamping, argument
 * errors and the status word as in fa_fwd_varlen and fa_bwd.  dK / dV rows of key rows
 * that no sequence owns are left untouched.  seqused_q / seqused_k as in fa_fwd_varlen
 * (the same arrays the forward got): padding rows of dq, dk and dv are not written, and
 * padding rows of dout, q, k, v must hold finite values.
 */
int fa_bwd_varlen(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                  const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse,
                  fa_tensor* dq, fa_tensor* dk, fa_tensor* dv,
                  const int* cu_seqlens_q, const int* cu_seqlens_k,
                  const int* seqused_q, const int* seqused_k, int batch,
                  int max_seqlen_q, int max_seqlen_k,
                  float softmax_scale, int causal, int window_left, int window_right,
                  float softcap, int deterministic, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * fa_bwd_status — waits for `stream`, then reads the device status word that the last
 * fa_bwd (or fa_fwd given this workspace) left in `workspace` (0 when every bounded wait
 * completed, else FA_ERR_DEVICE_TIMEOUT's device-side code) into *device_status, and
 * clears it.  The pages have no counterpart: it is this library's way of reporting a
 * device-side wait that ran out, which the pages' kernels do not bound.  `workspace` must
 * be a buffer that a backward call accepted (the status word sits in its first 256 bytes).
 * Returns FA_OK, FA_ERR_NULL for a NULL pointer, or FA_ERR_CUDA if a copy failed.
 */
int fa_bwd_status(void* workspace, void* stream, int* device_status);

/*
 * fa_bwd_noalloc — the same backward as fa_bwd (same arguments, layouts, results and
 * argument errors; a device-side timeout is read with fa_bwd_noalloc_status) for callers that cannot allocate device memory: code running where a
 * cudaMalloc is not allowed (a serving or real-time loop that must not synchronize the
 * device, a region recorded into a CUDA graph) or an embedding with a fixed memory
 * budget that has no allocator to provide fa_bwd's workspace.  The source pages have no
 * counterpart to this entry point.
 *
 * It allocates nothing.  Its scratch is one library-owned device array of
 * FA_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading the library keeps until the
 * process exits.  A problem whose fa_bwd_workspace_size exceeds that is rejected with
 * FA_ERR_WORKSPACE before any launch.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current) and caches it; make
 * that first call outside any stream capture.  All calls on a device share the array:
 * each call clears what must start at zero, but calls that overlap on the GPU race, so
 * order them on one stream.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)
int fa_bwd_noalloc(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                   const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse,
                   fa_tensor* dq, fa_tensor* dk, fa_tensor* dv,
                   float softmax_scale, int causal, int window_left, int window_right,
                   float softcap, int deterministic, void* stream);

/*
 * fa_bwd_noalloc_status — fa_bwd_status for fa_bwd_noalloc: waits for `stream`, then reads
 * the status word in the current device's library-owned scratch array into
 * *device_status (0 when every bounded wait of the last fa_bwd_noalloc on this device
 * completed, non-zero when one ran out and the outputs are incomplete) and clears it.
 * Allocates nothing.  Call it before the next fa_bwd_noalloc on the device, whose first
 * kernel clears the word.  No counterpart on the pages.  Returns FA_OK, FA_ERR_NULL, or
 * FA_ERR_CUDA if the address lookup or a copy failed.
 */
int fa_bwd_noalloc_status(void* stream, int* device_status);

/*
 * Backward algorithm for later fa_bwd calls in this process (not thread-safe).
 * fa_bwd_set_algorithm returns FA_ERR_ARG for an unknown value; fa_bwd_get_algorithm
 * returns the current one.
 *   FA_BWD_ALGO_AUTO (default): the fused algorithm, except for deterministic batched
 *     bf16 calls without a block mask on a square shape (Sq == Sk), which run the split
 *     algorithm: there it needs no waits, while the fused ordered mode must claim the
 *     shortest key tiles first.  Both results are bitwise reproducible, but they are not
 *     the same bits, so on those shapes a deterministic batched call no longer matches the
 *     fused ordered mode (which fa_bwd_varlen always uses) bit for bit; select
 *     FA_BWD_ALGO_FUSED for that.
 *   FA_BWD_ALGO_FUSED / FA_BWD_ALGO_SPLIT: always that algorithm (the split one refuses
 *     f16, packed sequences and block masks with FA_ERR_UNSUPPORTED).
 * Wide head dims (D > 128 or Dv != D) have a kernel of their own whatever is selected.
 */
#define FA_BWD_ALGO_SPLIT 0
#define FA_BWD_ALGO_FUSED 1
#define FA_BWD_ALGO_AUTO 2
int fa_bwd_set_algorithm(int algorithm);
int fa_bwd_get_algorithm(void);

/*
 * Test hooks for failure detection (process-wide, not thread-safe; not for production).
 *
 * fa_debug_set_wait_limit — cycles a bounded device-side wait (mbarrier phase, ordered
 *   dQ counter) may spin before it gives up and records FA_ERR_DEVICE_TIMEOUT in the
 *   workspace status word.  Default 2e9 (about one second).  cycles <= 0: FA_ERR_ARG.
 * fa_debug_poison_ordering — when enable != 0, every later deterministic fa_bwd sets the
 *   ordering counter of the first dQ tile to a value no contributor will match, so the
 *   ordered wait must run out: the kernels end, the status word reads the timeout, and
 *   the context stays usable.  No effect on non-deterministic calls.
 */
int fa_debug_set_wait_limit(long long cycles);
int fa_debug_poison_ordering(int enable);

/*
 * Kernel timing (process-wide).  fa_profile_enable(1) creates four CUDA events on the
 * current device; every later fa_bwd records them on its stream before the preprocess,
 * before and after the main kernel, and after the convert.  fa_profile_read waits for
 * the last event and writes the three durations of the most recent fa_bwd, in ms, to
 * ms3[0] (preprocess), ms3[1] (main) and ms3[2] (convert).  Returns FA_ERR_ARG if
 * profiling was never enabled.
 */
int fa_profile_enable(int enable);
int fa_profile_read(float* ms3);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
