// fa_kernels.h — parameter blocks and launchers shared by the host API and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kTileQ = 128;   // queries per tile (M of dQ, N of S^T / dP^T)
constexpr int kTileK = 128;   // keys per CTA (M of S^T, dP^T, dK, dV)

// Status-word slots at the start of the backward workspace.
enum : int { WS_STATUS = 0, WS_TICKET = 1, WS_TICKET_DQ = 2, WS_HEADER_BYTES = 256 };

struct BwdPreParams {
  const __nv_bfloat16* dout;
  const __nv_bfloat16* out;
  const float* lse;
  int64_t do_sb, do_ss, do_sh;   // element strides of dO (B, S, H)
  int64_t o_sb, o_ss, o_sh;      // element strides of O
  int64_t lse_sb, lse_sh, lse_ss;
  int B, H, Sq, Sq_r, D;
  float* lse2;                   // (B*H, Sq_r) LSE * log2(e); +inf on padded rows
  float* dsum;                   // (B*H, Sq_r) rowsum(dO*O); 0 on padded rows
  float4* zero_ptr;              // dQ accumulator + counters, zeroed here
  int64_t zero_count;            // in float4 units
  int* header;                   // status word + tile ticket, zeroed here
  // packed sequences (varlen != 0): dout / out / lse are (1, total_q, H, D) / (1, H,
  // total_q) views, B sequences, rows laid out per head in T slots of 128 (fa_tiles.h)
  int varlen;
  const int* cu_q;
  const int* used_q;             // per-sequence used query rows, or null
  int total_q;
  int64_t T;
};

struct BwdMainParams {
  int B, H, Hk, G, Sq, Sk, D;
  int Mb, Nb, Sq_r;
  int num_tiles;                 // key tiles x batch x kv-heads (persistent CTAs loop over them)
  int lo, hi;                    // visible iff lo <= j - i <= hi (clamped to +-2^30)
  long long lo64, hi64;          // the same bounds, unclamped (tile ranges)
  float scale_log2;              // scale * log2(e)
  float cap_scale;               // scale / softcap
  float cap_log2;                // softcap * log2(e)
  float dk_scale;                // scale (dK = scale * dA^T Q)
  int deterministic;
  const float* lse2;
  const float* dsum;
  float* dq_accum;               // tiles of (Dp/4, 128, 4) fp32 per (b, h, m-tile)
  int* sems;                     // (B*H*Mb) ordering counters (deterministic mode)
  int* status;
  int* ticket;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t dk_sb, dk_ss, dk_sh;
  int64_t dv_sb, dv_ss, dv_sh;
  // split algorithm: the dQ kernel's tile ticket and its bf16 output
  int* ticket_dq;
  __nv_bfloat16* dq;
  int64_t dq_sb, dq_ss, dq_sh;
  long long wait_limit;
  // packed sequences (the VARLEN kernel): q, k, v, dout, dk, dv are (1, total, H, D)
  // views; B sequences; Nb / Mb count the tiles of the longest one; dQ tiles, LSE2 / D
  // rows and counters are indexed per head by slot (fa_tiles.h: first_slot, T slots)
  const int* cu_q;
  const int* cu_k;
  const int* used_q;   // per-sequence used query / key rows, or null (fa_tiles.h seq_rows)
  const int* used_k;
  int total_q, total_k;
  long long T;
  int causal, window_left, window_right;
  // block sparsity (the SPARSE kernel): per key-tile ticket, the number of kept steps and
  // their (q-head in group << 16 | query tile) entries at sp_lists[ticket * sp_stride + i]
  const int* sp_counts;
  const int* sp_lists;
  long long sp_stride;
  // and the (B, H, Mb, Nb) block mask itself: the ordered mode counts, for a step's query
  // tile, the kept key tiles above this one
  const uint8_t* block_mask;  // dK / dV leave through tensor copies of 32-row boxes (tensor maps of dk and dv passed
  // to the main kernel); 0: every row is stored by its thread
  int tma_epilogue;
};

// Builds the block-sparse step lists of the main kernel from a (B, H, Mb, Nb) block mask:
// one warp per key-tile ticket (the main kernel's ticket order).
struct BwdSparseParams {
  const uint8_t* block_mask;
  int B, H, Hk, G, Sq, Sk, Mb, Nb;
  long long lo64, hi64;
  int* counts;
  int* lists;
  long long stride;    // G * Mb
  int num_tiles;
  int deterministic;   // the main kernel's ticket order: highest key tile first
};

struct BwdConvParams {
  const float* dq_accum;
  __nv_bfloat16* dq;
  int64_t dq_sb, dq_ss, dq_sh;
  int B, H, Sq, D, Dp, Mb;
  float scale;
  // packed sequences (varlen != 0): dq is a (1, total_q, H, D) view; tiles by slot
  int varlen;
  const int* cu_q;
  const int* used_q;   // per-sequence used query rows, or null
  int total_q;
  int64_t T;
};


// The tcgen05 forward: one CTA per (128-query tile, batch, q-head); q, k, v reach it
// through tensor maps, O and LSE are written with plain stores.
struct FwdTcParams {
  int B, H, Hk, G, Sq, Sk, D, Mb, Nb;
  long long lo64, hi64;          // visible iff lo <= j - i <= hi (unclamped; tile ranges)
  int lo, hi;                    // the same bounds clamped to +-2^30 (per-element mask)
  float scale_log2;              // scale * log2(e)
  float cap_scale;               // scale / softcap
  float cap_log2;                // softcap * log2(e)
  void* o;                       // (B, Sq, H, D) of the inputs' 16-bit type
  int64_t o_sb, o_ss, o_sh;
  float* lse;                    // (B, H, Sq) natural log
  int64_t lse_sb, lse_sh, lse_ss;
  int* status;                   // timeout status word, or null
  long long wait_limit;
  // Packed variable-length sequences (varlen != 0): q, k, v and o are (1, total, H, D)
  // views, B is the number of sequences and sequence b owns rows [cu_q[b], cu_q[b+1]) of
  // q / o and [cu_k[b], cu_k[b+1]) of k / v; Mb counts the query tiles of the longest
  // sequence.  The mask is bottom-right aligned per sequence, so lo / hi are derived per
  // sequence from causal and the window sizes.
  int varlen;
  const int* cu_q;
  const int* cu_k;
  // Optional per-sequence used lengths: sequence b computes only the first used_q[b]
  // query rows and used_k[b] key rows of its range (clamped to the range); null: all.
  const int* used_q;
  const int* used_k;
  int total_q, total_k;
  int causal, window_left, window_right;
  // Block sparsity (batched calls): (B, H, Mb, Nb) bytes, contiguous; a zero entry
  // removes the (query tile, key tile) pair.  Null: every pair the mask allows is kept.
  const uint8_t* block_mask;
  // O leaves through tensor copies of 32-row boxes staged in the item's Q buffer (tensor
  // maps of o passed to the kernel); 0: every row is stored by its thread
  int tma_epilogue;
};

// Head dims above 128, or a V head dim different from the Q/K one (fa_wide.cu).  Both
// padded dims are multiples of 64 and at most 256; the tensor maps use 64-column
// 128B-swizzled boxes (128 rows for K / V and the forward's Q, 64 rows for the
// backward's Q / dO steps).
struct WideParams {
  int B, H, Hk, G, Sq, Sk;
  int Dk, Dv;                    // logical head dims of q / k and of v
  int DPK, DPV;                  // padded to multiples of 64
  int Mb, Nb;                    // forward: 128-query tiles; backward: 64-query blocks; 128-key tiles
  int nslice;                    // backward: 128-column output slices (max over dK and dV)
  int nks;                       // backward: slices that carry dK / dQ columns
  long long lo64, hi64;          // visible iff lo <= j - i <= hi (unclamped)
  int lo, hi;                    // clamped to +-2^30
  float scale_log2, cap_scale, cap_log2, dk_scale;
  void* o;                       // forward output (B, Sq, H, Dv)
  int64_t o_sb, o_ss, o_sh;
  float* lse;
  int64_t lse_sb, lse_sh, lse_ss;
  const float* lse2;             // backward: (B*H, Sq_r) from the preprocess
  const float* dsum;
  int Sq_r;
  float* dq_accum;               // (B, H, Mb, nks) blocks of 128 x 64 fp32 (see fa_wide.cu)
  void* dk;                      // (B, Sk, Hk, Dk)
  void* dv;                      // (B, Sk, Hk, Dv)
  int64_t dk_sb, dk_ss, dk_sh, dv_sb, dv_ss, dv_sh;
  void* dq;                      // convert: (B, Sq, H, Dk)
  int64_t dq_sb, dq_ss, dq_sh;
  float scale;
  int* status;
  long long wait_limit;
  // deterministic mode: tiles are claimed from *ticket highest key tile first, and the dQ
  // partials of a block are added in descending key-tile order through sems (one counter
  // per accumulator block)
  int deterministic;
  int* ticket;
  int* sems;
};

// Tensor maps for one bf16 (B, S, H, D) operand: a 64-column 128B-swizzled box and,
// when Dp % 64 != 0, a narrower box for the remaining 16 or 32 columns.
struct OperandMaps {
  CUtensorMap full;
  CUtensorMap tail;
};

size_t bwd_main_smem_bytes(int Dp);
cudaError_t launch_bwd_preprocess(const BwdPreParams& p, bool f16, cudaStream_t s);
// f16: the 16-bit operands and outputs are f16 (else bf16); mode: 0 batched, 1 packed
// sequences, 2 block-sparse (step lists from launch_bwd_sparse_lists)
// dk, dv: tensor maps of the outputs with 32-row boxes (used when p.tma_epilogue is set)
// pdl: launched as a programmatic dependent of the kernel before it on the stream (the
// preprocess), which must then be the last operation enqueued before it
cudaError_t launch_bwd_main(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                            const OperandMaps& v, const OperandMaps& dout, const OperandMaps& dk,
                            const OperandMaps& dv, int Dp, bool softcap, bool f16, int mode,
                            int num_ctas, bool pdl, cudaStream_t s);
cudaError_t launch_bwd_sparse_lists(const BwdSparseParams& p, cudaStream_t s);
cudaError_t launch_bwd_convert(const BwdConvParams& p, bool f16, cudaStream_t s);
// dK/dV kernel (num_kv_ctas = key tiles x batch x kv-heads) then dQ kernel (num_q_ctas =
// query tiles x batch x q-heads, claimed by at most one persistent CTA per SM), both on
// stream s.
cudaError_t launch_bwd_split(const BwdMainParams& p, const OperandMaps& q, const OperandMaps& k,
                             const OperandMaps& v, const OperandMaps& dout, int Dp, bool softcap,
                             int num_kv_ctas, int num_q_ctas, cudaStream_t s);
cudaError_t launch_fwd_empty(const FwdTcParams& p, cudaStream_t s);
// o: tensor maps of the output with 32-row boxes (used when p.tma_epilogue is set)
cudaError_t launch_fwd_tc(const FwdTcParams& p, const OperandMaps& q, const OperandMaps& k,
                          const OperandMaps& v, const OperandMaps& o, int Dp, bool softcap,
                          bool f16, cudaStream_t s);
size_t wide_fwd_smem_bytes(int DPK, int DPV);
size_t wide_bwd_smem_bytes(int DPK, int DPV);
cudaError_t launch_fwd_wide(const WideParams& p, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, bool softcap, bool f16, cudaStream_t s);
cudaError_t launch_bwd_wide(const WideParams& p, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const CUtensorMap& dout, bool softcap,
                            bool f16, cudaStream_t s);
cudaError_t launch_convert_wide(const WideParams& p, bool f16, cudaStream_t s);
#ifdef FA_TRACE
cudaError_t bwd_trace_copy(void* host, size_t bytes);
cudaError_t split_trace_copy(void* host, size_t bytes);
cudaError_t bwd_timeline_copy(void* host, size_t bytes, bool clear);
cudaError_t bwd_trace_mma_copy(void* host, size_t bytes);
#endif

}  // namespace fa
