"""Host check of the weighted stream-K split that the decode and verify kernels
share (csrc/common.cuh: Split, unit_of, unit_segments), against brute force on
seeded cases. Compiled with nvcc as host code; no GPU needed.

Checked per case (unit tile counts, segment cost C, CTA count NC):
  * the CTA ranges [tile_at(bound(c)), tile_at(bound(c + 1))) partition the
    tiles in order;
  * unit_of(g) is the unit whose tile range holds g;
  * cta_of(x, u) is the CTA whose range holds tile x of unit u;
  * unit_segments(u) gives the first and last CTA holding tiles of u, the count
    of CTAs holding them, and the partial slot the first of them writes (its own
    slot when u starts its range, else NC + u);
  * the rule the tree-verify combine uses to skip CTAs of a unit's span that
    hold none of its tiles (a CTA strictly after the first holds tiles iff its
    weighted range is not empty) agrees with the ranges;
  * every partial slot is written by at most one (CTA, unit) segment.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_attention_kv_dattn_gb300", "csrc")

SHIM = r'''
#include <cstdio>
#include <vector>
#include "common.cuh"
using namespace dattn;

// stdin: cases "U C NC t_0 .. t_{U-1}"; prints "ok" or the first failure.
int main() {
  int U, C, NC, ncase = 0;
  while (std::scanf("%d %d %d", &U, &C, &NC) == 3) {
    std::vector<int> P(U + 1, 0);
    for (int u = 0; u < U; ++u) { int t; std::scanf("%d", &t); P[u + 1] = P[u] + t; }
    const int T = P[U];
    const Split sp{P.data(), U, C, NC, T + static_cast<long long>(C) * U};
    #define FAIL(...) do { std::printf("case %d (U=%d C=%d NC=%d): ", ncase, U, C, NC); \
        std::printf(__VA_ARGS__); std::printf("\n"); return 1; } while (0)
    std::vector<int> g0(NC), g1(NC);
    for (int c = 0; c < NC; ++c) { g0[c] = sp.tile_at(sp.bound(c)); g1[c] = sp.tile_at(sp.bound(c + 1)); }
    if (g0[0] != 0) FAIL("first range starts at %d", g0[0]);
    if (g1[NC - 1] != T) FAIL("last range ends at %d of %d", g1[NC - 1], T);
    for (int c = 0; c < NC; ++c) {
      if (g1[c] < g0[c]) FAIL("cta %d range [%d, %d)", c, g0[c], g1[c]);
      if (c + 1 < NC && g1[c] != g0[c + 1]) FAIL("cta %d ends at %d, next starts at %d", c, g1[c], g0[c + 1]);
    }
    std::vector<int> owner(T, -1);
    for (int c = 0; c < NC; ++c) for (int g = g0[c]; g < g1[c]; ++g) owner[g] = c;
    for (int u = 0; u < U; ++u)
      for (int g = P[u]; g < P[u + 1]; ++g) {
        if (unit_of(P.data(), U, g) != u) FAIL("unit_of(%d) = %d, want %d", g, unit_of(P.data(), U, g), u);
        if (sp.cta_of(g, u) != owner[g]) FAIL("cta_of(%d, %d) = %d, want %d", g, u, sp.cta_of(g, u), owner[g]);
      }
    std::vector<int> writers(NC + U, 0);
    for (int c = 0; c < NC; ++c) {  // the kernels' slots: first segment of a range -> c, later -> NC + u
      bool first = true;
      for (int u = 0; u < U; ++u) {
        const int lo = P[u] > g0[c] ? P[u] : g0[c], hi = P[u + 1] < g1[c] ? P[u + 1] : g1[c];
        if (hi <= lo) continue;
        ++writers[first ? c : NC + u];
        first = false;
      }
    }
    for (int s = 0; s < NC + U; ++s) if (writers[s] > 1) FAIL("slot %d written %d times", s, writers[s]);
    for (int u = 0; u < U; ++u) {
      int c_lo = 0, c_hi = -1, slot = 0;
      const int n = unit_segments(sp, P[u], P[u + 1], u, c_lo, c_hi, slot);
      int bc_lo = -1, bc_hi = -1, bn = 0;
      for (int c = 0; c < NC; ++c) {
        const int lo = P[u] > g0[c] ? P[u] : g0[c], hi = P[u + 1] < g1[c] ? P[u + 1] : g1[c];
        if (hi <= lo) continue;
        if (bc_lo < 0) bc_lo = c;
        bc_hi = c;
        ++bn;
      }
      if (P[u + 1] == P[u]) { if (n != 0) FAIL("empty unit %d has %d segments", u, n); continue; }
      if (n != bn || c_lo != bc_lo || c_hi != bc_hi)
        FAIL("unit %d segments n=%d [%d, %d], want n=%d [%d, %d]", u, n, c_lo, c_hi, bn, bc_lo, bc_hi);
      const int want_slot = g0[c_lo] == P[u] ? c_lo : NC + u;
      if (slot != want_slot) FAIL("unit %d first slot %d, want %d", u, slot, want_slot);
      for (int cc = c_lo + 1; cc <= c_hi; ++cc) {
        const bool holds = g1[cc] > g0[cc];  // strictly inside the span: any tiles are u's
        if (sp.has_tiles_inside(cc) != holds) FAIL("unit %d cta %d: non-empty range %d, holds tiles %d", u, cc,
                                                   (int)sp.has_tiles_inside(cc), (int)holds);
        if (holds && !(g0[cc] >= P[u] && g0[cc] < P[u + 1])) FAIL("unit %d cta %d starts outside it", u, cc);
      }
    }
    ++ncase;
  }
  std::printf("ok %d\n", ncase);
  return 0;
}
'''


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    return None


def _cases():
    rng = np.random.default_rng(20261202)
    out = [(1, 0, 1, [1]), (1, 8, 152, [3]), (3, 5, 4, [0, 0, 7]), (4, 12, 152, [0, 5, 0, 0]),
           (2, 0, 152, [1000, 1]), (5, 1, 3, [1, 1, 1, 1, 1])]
    for _ in range(400):
        U = int(rng.integers(1, 80))
        NC = int(rng.choice([1, 2, 7, 64, 152, 304]))
        C = int(rng.choice([0, 1, 5, 8, 12, 40]))
        kind = rng.integers(0, 4)
        if kind == 0:
            t = rng.integers(0, 4, U)            # many short or empty units
        elif kind == 1:
            t = rng.integers(0, 300, U)          # mixed lengths
        elif kind == 2:
            t = np.full(U, int(rng.integers(1, 64)))  # equal units
        else:
            t = np.where(rng.random(U) < 0.2, rng.integers(200, 2000, U), rng.integers(0, 3, U))
        out.append((U, C, NC, [int(x) for x in t]))
    return out


def test_split_matches_brute_force(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    src = tmp_path / "split_shim.cu"
    src.write_text(SHIM)
    exe = tmp_path / "split_shim"
    r = subprocess.run([nvcc, "-O1", "-std=c++17", "--expt-relaxed-constexpr",
                        "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC, "-o", str(exe), str(src)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    cases = _cases()
    text = "\n".join(f"{U} {C} {NC} " + " ".join(map(str, t)) for U, C, NC, t in cases) + "\n"
    r = subprocess.run([str(exe)], input=text, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == f"ok {len(cases)}", r.stdout + r.stderr
