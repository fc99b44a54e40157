"""The tile-range header (which query tiles a key tile visits, and the first key tile
of a query tile, used to order deterministic dQ additions) against brute force over
every element of every tile.  Compiled with g++; no GPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

HARNESS = r'''
#include <cstdio>
#include "fa_tiles.h"
using namespace fa;
static bool vis(const MaskGeom& g, long i, long j) {
  return i < g.Sq && j < g.Sk && (j - i) >= g.lo && (j - i) <= g.hi;
}
int main() {
  long bad = 0, cases = 0;
  const int sizes[] = {1, 5, 64, 127, 128, 129, 200, 256, 300, 513};
  const int wins[] = {-1, 0, 1, 100, 128, 300};
  for (int Sq : sizes) for (int Sk : sizes) for (int causal = 0; causal < 2; ++causal)
  for (int wl : wins) for (int wr : wins) {
    MaskGeom g = make_geom(Sq, Sk, causal, wl, wr, 128, 128);
    for (long n = 0; n < g.Nb; ++n) {
      long mb, me; m_range(g, n, &mb, &me);
      for (long m = 0; m < g.Mb; ++m) {
        bool any = false, all = true;
        for (long i = m * 128; i < m * 128 + 128; ++i)
          for (long j = n * 128; j < n * 128 + 128; ++j) {
            bool v = vis(g, i, j);
            any = any || v;
            // tile_full promises every (i, j) with j < Sk is visible (rows past Sq may be
            // anything: their P is forced to zero by LSE = +inf)
            if (i < g.Sq && !v) all = false;
            if (i >= g.Sq && j < g.Sk && !((j - i) >= g.lo && (j - i) <= g.hi)) all = false;
          }
        bool act = tile_active(g, m, n);
        bool in_range = m >= mb && m < me;
        if (act != any || in_range != any) { ++bad; if (bad < 5) printf("range Sq=%d Sk=%d c=%d wl=%d wr=%d m=%ld n=%ld any=%d act=%d in=%d\n", Sq, Sk, causal, wl, wr, m, n, any, act, in_range); }
        if (tile_full(g, m, n) && !all) { ++bad; if (bad < 5) printf("full Sq=%d Sk=%d m=%ld n=%ld\n", Sq, Sk, m, n); }
        if (tile_full(g, m, n) && (n * 128 + 128 > g.Sk)) ++bad;
        ++cases;
      }
    }
    for (long m = 0; m < g.Mb; ++m) {
      long nb, ne; n_range(g, m, &nb, &ne);
      for (long n = 0; n < g.Nb; ++n) {
        bool in = n >= nb && n < ne;
        if (in != tile_active(g, m, n)) { ++bad; if (bad < 5) printf("nrange Sq=%d Sk=%d m=%ld n=%ld\n", Sq, Sk, m, n); }
      }
    }
  }
  printf("cases=%ld bad=%ld\n", cases, bad);
  return bad != 0;
}
'''


def test_tile_ranges_brute_force(tmp_path):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "tiles.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "tiles"
    inc = os.path.join(ROOT, "flashattention_backward_pass_gb300", "csrc")
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", inc, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad=0" in r.stdout


SLOTS_HARNESS = r'''
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "fa_tiles.h"
using namespace fa;
// Packed sequences: every query tile of every sequence gets its own slot below
// slot_count, and slot_owner maps each used slot back to its sequence; used lengths
// (seqused) keep the first row and clamp the length.  Also run with malformed
// (decreasing, negative, too large) offsets, where only the bound must hold.
int main() {
  long bad = 0, cases = 0;
  srand(7);
  for (int trial = 0; trial < 3000; ++trial) {
    const int B = 1 + rand() % 12;
    std::vector<int> cu(B + 1, 0);
    const bool malformed = trial % 5 == 4;
    for (int b = 0; b < B; ++b) {
      int len = rand() % 4 == 0 ? 0 : rand() % 700;
      if (rand() % 6 == 0) len = 128 * (1 + rand() % 3);
      cu[b + 1] = cu[b] + len;
    }
    long total = cu[B];
    if (malformed) {
      for (int b = 0; b <= B; ++b) cu[b] = rand() % 1500 - 300;
      total = rand() % 1200;
    }
    const long T = slot_count(total, B);
    std::vector<int> owner(T, -1);
    std::vector<int> used(B);
    for (int b = 0; b < B; ++b) used[b] = rand() % 900 - 100;
    for (int b = 0; b < B; ++b) {
      long s0, len;
      seq_rows(cu.data(), b, total, &s0, &len);
      if (s0 < 0 || s0 + len > total) ++bad;
      // used lengths: the same first row and a length clamped into [0, len], so the used
      // rows (and their slots) stay inside the sequence's own; null means all rows
      long s1, l1, s2, l2;
      seq_rows(cu.data(), used.data(), b, total, &s1, &l1);
      seq_rows(cu.data(), nullptr, b, total, &s2, &l2);
      const long want = used[b] < 0 ? 0 : (used[b] < len ? used[b] : len);
      if (s1 != s0 || l1 != want || s2 != s0 || l2 != len) ++bad;
      const long fs = first_slot(cu.data(), b, total);
      for (long m = 0; m * 128 < len; ++m) {
        const long t = fs + m;
        ++cases;
        if (t < 0 || t >= T) { ++bad; continue; }
        if (malformed) continue;
        if (owner[t] != -1) ++bad;
        owner[t] = b;
        if (slot_owner(cu.data(), B, total, t) != b) ++bad;
      }
    }
  }
  printf("cases=%ld bad=%ld\n", cases, bad);
  return bad != 0;
}
'''


def test_packed_sequence_slots(tmp_path):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "slots.cpp"
    src.write_text(SLOTS_HARNESS)
    exe = tmp_path / "slots"
    inc = os.path.join(ROOT, "flashattention_backward_pass_gb300", "csrc")
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", inc, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad=0" in r.stdout


ORDER_HARNESS = r'''
#include <cstdio>
#include <vector>
#include "fa_tiles.h"
using namespace fa;
// A model of the fused backward's ordered (deterministic) dQ mode: P persistent CTAs take
// key-tile tickets (n, batch, kv-head) in claim order; a ticket's steps visit its query
// tiles for each of its G q-heads (head-major); the step for dQ tile (b, h, m) may add
// only when the tile's counter equals this key tile's rank, then increments it.  Ranks:
// descending (highest key tile first, rank = n_end - 1 - n) or ascending (n - n_begin).
// Returns 1 if every step ran, 0 on a deadlock (no CTA can move); also checks that every
// counter ends at its query tile's number of contributing key tiles.
static int simulate(const std::vector<MaskGeom>& gs, int G, int P, bool claim_desc,
                    bool add_desc, long* bad) {
  // one geometry per (sequence, kv-head) group: packed sequences differ in length, and the
  // tickets run over the longest one's key tiles
  const int BHk = (int)gs.size();
  long Nb = 0, Mb = 0;
  for (const auto& g : gs) { Nb = g.Nb > Nb ? g.Nb : Nb; Mb = g.Mb > Mb ? g.Mb : Mb; }
  const long T = Nb * BHk;
  std::vector<int> cnt((size_t)BHk * G * Mb, 0);
  struct Cta { long t = -1; long step = 0, total = 0, n = 0, r = 0, mb = 0, mc = 0; };
  std::vector<Cta> c(P);
  long next = 0, done = 0;
  auto claim = [&](Cta& x) {
    while (next < T) {
      const long t = next++;
      const long n0 = t / BHk;
      x.r = t % BHk;
      x.n = claim_desc ? Nb - 1 - n0 : n0;
      long mb, me; m_range(gs[x.r], x.n, &mb, &me);
      x.mb = mb; x.mc = me - mb; x.total = x.mc * G; x.step = 0; x.t = t;
      if (x.total > 0) return;
      ++done;  // a ticket with no step finishes at once
    }
    x.t = -1;
  };
  for (auto& x : c) claim(x);
  while (true) {
    bool moved = false, busy = false;
    for (auto& x : c) {
      if (x.t < 0) continue;
      busy = true;
      const long gg = x.step / x.mc, m = x.mb + x.step % x.mc;
      long nb, ne; n_range(gs[x.r], m, &nb, &ne);
      const int want = (int)(add_desc ? ne - 1 - x.n : x.n - nb);
      int& k = cnt[((size_t)x.r * G + gg) * Mb + m];
      if (k != want) continue;
      ++k;
      moved = true;
      if (++x.step == x.total) { ++done; claim(x); }
    }
    if (!busy) break;
    if (!moved) return 0;
  }
  for (long r = 0; r < BHk; ++r)
    for (long gg = 0; gg < G; ++gg)
      for (long m = 0; m < gs[r].Mb; ++m) {
        long nb, ne; n_range(gs[r], m, &nb, &ne);
        if (cnt[((size_t)r * G + gg) * Mb + m] != (int)(ne - nb)) ++*bad;
      }
  if (done != T) ++*bad;
  return 1;
}
int main() {
  long bad = 0, runs = 0, neg_deadlocks = 0;
  const int lens[] = {128, 300, 512, 1000};
  const int wins[][3] = {{1, -1, -1}, {0, -1, -1}, {0, 200, 0}, {0, 100, 300}, {1, 130, -1}};
  const int ctas[] = {1, 2, 3, 7};
  for (int Sq : lens) for (int Sk : lens) for (auto& w : wins) for (int BHk = 1; BHk <= 3; ++BHk)
  for (int G = 1; G <= 2; ++G) for (int P : ctas) {
    // batched: every group has the same lengths; packed: group r's lengths are rotated
    // through the list (0 included: a sequence with no query or no key)
    for (int packed = 0; packed < 2; ++packed) {
      std::vector<MaskGeom> gs;
      for (int r = 0; r < BHk; ++r) {
        const int sq = packed ? (r == 2 ? 0 : lens[(r + Sq / 100) % 4]) : Sq;
        const int sk = packed ? lens[(r + Sk / 100 + 1) % 4] : Sk;
        gs.push_back(make_geom(sq, sk, w[0], w[1], w[2], 128, 128));
      }
      // the kernel's pairing: highest key tile claimed first, contributions added from
      // the highest key tile down; and the plain longest-first / ascending pairing
      if (!simulate(gs, G, P, true, true, &bad)) { ++bad; if (bad < 5) printf("deadlock desc Sq=%d Sk=%d c=%d P=%d packed=%d\n", Sq, Sk, w[0], P, packed); }
      if (!simulate(gs, G, P, false, false, &bad)) { ++bad; if (bad < 5) printf("deadlock asc Sq=%d Sk=%d c=%d P=%d packed=%d\n", Sq, Sk, w[0], P, packed); }
      // longest-first claims with descending adds must be able to deadlock
      long ignore = 0;
      if (!simulate(gs, G, P, false, true, &ignore)) ++neg_deadlocks;
      runs += 2;
    }
  }
  printf("runs=%ld bad=%ld neg_deadlocks=%ld\n", runs, bad, neg_deadlocks);
  return (bad != 0 || neg_deadlocks == 0) ? 1 : 0;
}
'''


def test_ordered_mode_schedule_never_deadlocks(tmp_path):
    """The ordered mode's pairing (highest key tile claimed first, dQ contributions added
    from the highest key tile down) lets every step run on any number of CTAs, and every
    counter ends at its contributor count; the mismatched pairing does deadlock, so the
    model can tell the two apart."""
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "order.cpp"
    src.write_text(ORDER_HARNESS)
    exe = tmp_path / "order"
    inc = os.path.join(ROOT, "flashattention_backward_pass_gb300", "csrc")
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", inc, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad=0" in r.stdout
