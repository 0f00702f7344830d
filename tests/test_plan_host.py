"""Host checks of the tile-share arithmetic the tensor-core decode plans with (no GPU).

The decode gives cluster c of nc the tiles [share_begin(c), share_begin(c+1)) of all T tiles
and finds the owner of a tile with share_owner. A host program built with nvcc from the
kernel header checks, for many (T, nc), that the shares tile [0, T) in order and that
share_owner agrees with a brute-force search; and that the two workspace index maps
(row-major Q_lat and chunk-major partial O) are bijections onto their arrays.
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
