"""Host checks of the tile-share arithmetic the tensor-core decode plans with (no GPU).

The decode gives cluster c of nc the units [share_begin(c), share_begin(c+1)) of all T units
(a sequence's tiles plus a few units for the start of its segment) and finds the owner of a
unit with share_owner. Host programs built with nvcc from the kernel header check, for many
(T, nc), that the shares tile [0, T) in order and that share_owner agrees with a brute-force
search; that the two workspace index maps (row-major Q_lat and chunk-major partial O) are
bijections onto their arrays; and that walking the shares visits every tile once.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r'''
#include <cstdio>
#include <vector>
#include "decode_tc.cuh"
using namespace mla::tcd;
int main() {
  long bad = 0, checked = 0;
  std::vector<long> Ts;
  for (long T = 1; T <= 700; ++T) Ts.push_back(T);
  for (long T : {1023L, 1024L, 1025L, 8191L, 65536L, 1114757L / 64, (1L << 21) + 3, (1L << 30) + 7}) Ts.push_back(T);
  for (long T : Ts) {
    for (long nc : {1L, 2L, 3L, 7L, 63L, 64L, 74L, 127L, 128L}) {
      if (share_begin(0, T, nc) != 0 || share_begin(nc, T, nc) != T) { ++bad; continue; }
      long c = 0;
      const long step = T > 5000 ? T / 4999 : 1;   // sample the huge cases
      for (long t = 0; t < T; t += step) {
        while (share_begin(c + 1, T, nc) <= t) ++c;          // brute force: c with begin(c) <= t < begin(c+1)
        if (share_begin(c, T, nc) > t) ++bad;
        if (share_owner(t, T, nc) != c) ++bad;
        ++checked;
      }
      for (long k = 0; k < nc; ++k) if (share_begin(k, T, nc) > share_begin(k + 1, T, nc)) ++bad;
    }
  }
  // index maps: every element of the arrays is hit exactly once
  const int B = 3, slots = 5;
  std::vector<int> q(static_cast<size_t>(B) * kH * kRow, 0), o(static_cast<size_t>(slots) * kOChunks * kH * 4, 0);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < kH; ++h)
      for (int k = 0; k < kRow; ++k) q.at(qlat_row_index(b, h, k))++;
  for (int s = 0; s < slots; ++s)
    for (int c = 0; c < kOChunks; ++c)
      for (int h = 0; h < kH; ++h)
        for (int e = 0; e < 4; ++e) o.at(parto_index(s, c, h) + e)++;
  for (int v : q) bad += v != 1;
  for (int v : o) bad += v != 1;
  printf("%ld %ld\n", checked, bad);
  return bad != 0;
}
'''


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="needs nvcc (host compile only)")
def test_shares_partition_the_tiles_and_owner_agrees():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "plan.cu")
        open(src, "w").write(SRC)
        exe = os.path.join(d, "plan")
        subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "head_latent_attention_22_b300", "csrc"),
                        "-o", exe, src], check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True)
    checked, bad = (int(x) for x in out.stdout.split())
    assert out.returncode == 0 and bad == 0 and checked > 1_000_000


SEG_SRC = r'''
#include <cstdio>
#include <cstdlib>
#include <set>
#include <vector>
#include "decode_tc.cuh"
using namespace mla::tcd;
int main() {
  long bad = 0, cases = 0;
  unsigned s = 12345u;
  auto rnd = [&](unsigned m) { s = s * 1664525u + 1013904223u; return (s >> 8) % m; };
  for (int trial = 0; trial < 3000; ++trial) {
    const int B = 1 + static_cast<int>(rnd(trial < 2000 ? 20 : 300));
    const int mode = static_cast<int>(rnd(4));
    std::vector<int> n(B);
    for (int b = 0; b < B; ++b) {   // tiles per sequence: empty, short, long and mixed batches
      const int r = static_cast<int>(rnd(100));
      n[b] = mode == 0 ? static_cast<int>(rnd(3)) : mode == 1 ? 64 : (r < 15 ? 0 : static_cast<int>(rnd(mode == 2 ? 8 : 200)));
    }
    std::vector<int32_t> cum(B + 1, 0);
    for (int b = 0; b < B; ++b) cum[b + 1] = cum[b] + (n[b] > 0 ? n[b] + kSegUnits : 0);
    const long T = cum[B];
    for (long nc : {1L, 2L, 7L, 74L, 128L}) {
      ++cases;
      std::vector<std::vector<int>> seen(B);
      std::vector<std::vector<long>> owners(B);
      std::set<long> slots;
      for (long c = 0; c < nc; ++c) {
        const long t0 = share_begin(c, T, nc), t1 = share_begin(c + 1, T, nc);
        int first = 0;
        while (first < B && cum[first + 1] <= t0) ++first;   // brute force: sequence holding unit t0
        if (first == B) first = B - 1;
        SegIter si{t0, t1, first};
        int b, j0, j1;
        long count = 0;
        int last_b = -1;
        std::vector<std::pair<int, int>> firsts;   // (sequence, tile) of the share's first kPlanRows tiles
        while (si.next(cum.data(), B, &b, &j0, &j1)) {
          for (int j = j0; j < j1 && static_cast<int>(firsts.size()) < kPlanRows; ++j) firsts.push_back({b, j});
          if (b <= last_b || j0 < 0 || j1 <= j0 || j1 > n[b]) ++bad;
          if (!seen[b].empty() && seen[b].back() != j0) ++bad;     // consecutive clusters continue the tiles
          if (seen[b].empty() && j0 != 0) ++bad;
          seen[b].push_back(j1);
          owners[b].push_back(c);
          if (!slots.insert(b + c).second) ++bad;                  // partial slot b + c is unique
          count += j1 - j0;
          last_b = b;
        }
        if (count != share_tile_count(cum.data(), B, first, t0, t1)) ++bad;
        int fb[kPlanRows], fj[kPlanRows];
        if (count != share_tile_count(cum.data(), B, first, t0, t1, fb, fj)) ++bad;
        for (int k = 0; k < static_cast<int>(firsts.size()); ++k)
          if (fb[k] != firsts[k].first || fj[k] != firsts[k].second) ++bad;
      }
      for (int b = 0; b < B; ++b) {
        if (n[b] == 0) { bad += !seen[b].empty(); continue; }
        if (seen[b].empty() || seen[b].back() != n[b]) { ++bad; continue; }   // every tile exactly once
        const long c0 = share_owner(cum[b] + kSegUnits, T, nc), c1 = share_owner(cum[b + 1] - 1, T, nc);
        if (owners[b].front() != c0 || owners[b].back() != c1) ++bad;
        // the clusters between hold b's tiles and nothing else: each non-empty share in [c0, c1] visits b
        long k = 0;
        for (long c = c0; c <= c1; ++c)
          if (share_begin(c, T, nc) < share_begin(c + 1, T, nc)) {
            if (k >= static_cast<long>(owners[b].size()) || owners[b][k] != c) ++bad;
            ++k;
          }
        if (k != static_cast<long>(owners[b].size())) ++bad;
      }
    }
  }
  printf("%ld %ld\n", cases, bad);
  return bad != 0;
}
'''


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="needs nvcc (host compile only)")
def test_segments_cover_every_tile_once():
    """Shares are cut in units (a sequence's tiles plus the segment-start units); walking each
    cluster's share must still visit every tile of every sequence exactly once, in order, with
    the tile count the plan stores (and the first tiles whose rows it stores), the merge's cluster
    range [c0, c1] and unique partial slots."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "seg.cu")
        open(src, "w").write(SEG_SRC)
        exe = os.path.join(d, "seg")
        subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "head_latent_attention_22_b300", "csrc"),
                        "-o", exe, src], check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True)
    cases, bad = (int(x) for x in out.stdout.split())
    assert out.returncode == 0 and bad == 0 and cases == 15000
