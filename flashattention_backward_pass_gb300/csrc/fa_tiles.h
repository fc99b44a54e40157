// fa_tiles.h — which (query tile, key tile) pairs the mask leaves any visible entry in.
//
// Masking is bottom-right aligned (GQA/MQA page, causal block range: the key index
// limit is the query index plus seqlen_k - seqlen_q).  Key j is visible to query i iff
// lo <= j - i <= hi with lo = (Sk-Sq) - window_left (or -inf) and hi = (Sk-Sq) +
// window_right (or +inf; causal forces window_right = 0), 0 <= i < Sq, 0 <= j < Sk.
//
// The backward kernel gives each CTA one key tile n and walks the query tiles m with a
// visible entry; the deterministic dQ order needs, for a query tile m, the first key tile
// that touches it.  Both ranges come from the same predicate, so they agree exactly.
// Plain C++ (no CUDA types) so the host, the device and a CPU test all use this file.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int64_t kUnbounded = (int64_t)1 << 40;

struct MaskGeom {
  int64_t Sq, Sk;
  int64_t lo, hi;  // visible iff lo <= j - i <= hi
  int64_t tm, tn;  // query / key tile sizes
  int64_t Mb, Nb;  // number of query / key tiles
};

FA_HD int64_t floor_div(int64_t a, int64_t b) {  // b > 0
  int64_t q = a / b;
  return (a % b != 0 && a < 0) ? q - 1 : q;
}
FA_HD int64_t ceil_div_s(int64_t a, int64_t b) { return -floor_div(-a, b); }
FA_HD int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }
FA_HD int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

FA_HD MaskGeom make_geom(int64_t Sq, int64_t Sk, int causal, int64_t window_left,
                         int64_t window_right, int64_t tm, int64_t tn) {
  MaskGeom g;
  g.Sq = Sq;
  g.Sk = Sk;
  if (causal) window_right = 0;
  g.lo = window_left >= 0 ? (Sk - Sq) - window_left : -kUnbounded;
  g.hi = window_right >= 0 ? (Sk - Sq) + window_right : kUnbounded;
  g.tm = tm;
  g.tn = tn;
  g.Mb = (Sq + tm - 1) / tm;
  g.Nb = (Sk + tn - 1) / tn;
  return g;
}

// Does query tile m / key tile n contain a visible (i, j) with i < Sq, j < Sk?
FA_HD bool tile_active(const MaskGeom& g, int64_t m, int64_t n) {
  int64_t i_lo = m * g.tm, i_hi = min64(m * g.tm + g.tm - 1, g.Sq - 1);
  int64_t j_lo = n * g.tn, j_hi = min64(n * g.tn + g.tn - 1, g.Sk - 1);
  if (i_lo > i_hi || j_lo > j_hi) return false;
  return (j_lo - i_hi) <= g.hi && (j_hi - i_lo) >= g.lo;
}

// Query-tile range [*m_begin, *m_end) with a visible entry for key tile n (may be empty).
FA_HD void m_range(const MaskGeom& g, int64_t n, int64_t* m_begin, int64_t* m_end) {
  int64_t j_lo = n * g.tn, j_hi = min64(n * g.tn + g.tn - 1, g.Sk - 1);
  int64_t b = 0, e = g.Mb;
  if (j_lo > j_hi || g.Mb == 0) { *m_begin = 0; *m_end = 0; return; }
  // j_lo - i_hi <= hi  <=>  min(m*tm + tm - 1, Sq - 1) >= j_lo - hi
  int64_t need = j_lo - g.hi;
  if (g.Sq - 1 < need) { *m_begin = 0; *m_end = 0; return; }
  b = max64(b, ceil_div_s(need - (g.tm - 1), g.tm));
  // j_hi - i_lo >= lo  <=>  m*tm <= j_hi - lo
  int64_t lim = j_hi - g.lo;
  if (lim < 0) { *m_begin = 0; *m_end = 0; return; }
  e = min64(e, floor_div(lim, g.tm) + 1);
  if (b >= e) { b = 0; e = 0; }
  *m_begin = b;
  *m_end = e;
}

// Key-tile range [*n_begin, *n_end) with a visible entry for query tile m (may be empty).
FA_HD void n_range(const MaskGeom& g, int64_t m, int64_t* n_begin, int64_t* n_end) {
  int64_t i_lo = m * g.tm, i_hi = min64(m * g.tm + g.tm - 1, g.Sq - 1);
  int64_t b = 0, e = g.Nb;
  if (i_lo > i_hi || g.Nb == 0) { *n_begin = 0; *n_end = 0; return; }
  // j_lo - i_hi <= hi  <=>  n*tn <= i_hi + hi
  int64_t lim = i_hi + g.hi;
  if (lim < 0) { *n_begin = 0; *n_end = 0; return; }
  e = min64(e, floor_div(lim, g.tn) + 1);
  // j_hi - i_lo >= lo  <=>  min(n*tn + tn - 1, Sk - 1) >= i_lo + lo
  int64_t need = i_lo + g.lo;
  if (g.Sk - 1 < need) { *n_begin = 0; *n_end = 0; return; }
  b = max64(b, ceil_div_s(need - (g.tn - 1), g.tn));
  if (b >= e) { b = 0; e = 0; }
  *n_begin = b;
  *n_end = e;
}

// True when every (i, j) of the tile with i < m*tm + tm, j < n*tn + tn is visible and
// the key tile lies inside Sk, so the kernel can skip the per-element mask.  Query rows
// past Sq need no mask: their LSE is +inf, which makes P = 0 there.
FA_HD bool tile_full(const MaskGeom& g, int64_t m, int64_t n) {
  int64_t dmin = n * g.tn - (m * g.tm + g.tm - 1);
  int64_t dmax = n * g.tn + g.tn - 1 - m * g.tm;
  return dmin >= g.lo && dmax <= g.hi && (n * g.tn + g.tn) <= g.Sk;
}

// ------------------------------------------------------------------ packed sequences
//
// A variable-length batch packs B sequences along the row axis: sequence b owns query
// rows [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]).  Offsets are clamped into
// [0, total] before use, so malformed offsets cannot address rows outside the tensors.
FA_HD int64_t clamp_row(int64_t x, int64_t total) { return x < 0 ? 0 : (x > total ? total : x); }

FA_HD void seq_rows(const int* cu, int b, int64_t total, int64_t* start, int64_t* len) {
  const int64_t a = clamp_row(cu[b], total), e = clamp_row(cu[b + 1], total);
  *start = a;
  *len = e > a ? e - a : 0;
}

// With per-sequence used lengths (`used` non-null): sequence b keeps its rows from cu but
// computes only the first used[b] of them (clamped into [0, its row count]); the rest are
// padding.  Null `used`: every row of the sequence is used.
FA_HD void seq_rows(const int* cu, const int* used, int b, int64_t total, int64_t* start,
                    int64_t* len) {
  seq_rows(cu, b, total, start, len);
  if (used != nullptr) {
    const int64_t u = used[b];
    *len = u < 0 ? 0 : (u < *len ? u : *len);
  }
}

// The backward's per-head tile layout for packed sequences: the 128-row query tiles of
// sequence b take the slots [first_slot(b), first_slot(b) + ceil(Sq_b / 128)), with
// first_slot(b) = floor(cu_q[b] / 128) + b.  For non-decreasing offsets the ranges of
// different sequences never overlap (floor((a + s) / 128) >= floor(a / 128) +
// floor(s / 128) and ceil(s / 128) <= floor(s / 128) + 1), and slot_count slots cover
// all of them; with clamped offsets every slot index stays below slot_count even when
// the offsets are malformed.
FA_HD int64_t first_slot(const int* cu_q, int b, int64_t total_q) {
  return clamp_row(cu_q[b], total_q) / 128 + b;
}
FA_HD int64_t slot_count(int64_t total_q, int64_t B) { return total_q / 128 + B; }

// The sequence whose slot range starts at or before slot t (the largest such b).
FA_HD int slot_owner(const int* cu_q, int B, int64_t total_q, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (first_slot(cu_q, mid, total_q) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

}  // namespace fa
