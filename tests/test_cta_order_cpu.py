"""The CTA-order map (grouped_unit in csrc/kernels.cuh) on the host.

Every kernel that interleaves heads maps its linear CTA index u to a (head,
tile) unit with grouped_unit.  Compiled here with the host compiler against
the same header, it must be a bijection from [0, BH n) onto every
(head, tile) pair for any group size, put the units of one head group
before those of the next, and walk each group tile by tile with its heads
in ascending order; with a group of one it must be plain head-major order.
"""

import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_distillation_kl_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "kernels.cuh"
int main() {
  int bad = 0;
  const int BHs[] = {1, 2, 3, 7, 8, 13, 32, 64};
  const int ns[] = {1, 2, 5, 32, 129};
  for (int BH : BHs)
    for (int n : ns)
      for (int G = 1; G <= BH + 2; ++G) {
        std::vector<int> seen(size_t(BH) * n, 0);
        int prev_g0 = -1, prev_t = -1, prev_h = -1;
        for (int u = 0; u < BH * n; ++u) {
          int h = -1, t = -1;
          skl::grouped_unit(u, BH, n, G, h, t);
          if (h < 0 || h >= BH || t < 0 || t >= n) { ++bad; continue; }
          ++seen[size_t(h) * n + t];
          const int g0 = h / G * G;
          if (g0 < prev_g0) ++bad;  // groups in order
          if (g0 == prev_g0 && (t < prev_t || (t == prev_t && h <= prev_h))) ++bad;  // tile-major, heads ascending
          if (G == 1 && (h != u / n || t != u % n)) ++bad;
          prev_g0 = g0; prev_t = t; prev_h = h;
        }
        for (int c : seen) if (c != 1) ++bad;
      }
  std::printf("%d\n", bad);
  return bad != 0;
}
"""


def test_grouped_unit_is_an_ordered_bijection():
    cxx = shutil.which("g++") or shutil.which("c++")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if cxx is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("no host C++ compiler or CUDA headers")
    with tempfile.TemporaryDirectory() as tmp:
        src, exe = os.path.join(tmp, "order.cpp"), os.path.join(tmp, "order")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", cuda_inc, src, "-o", exe], check=True,
                       capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "0", r.stdout + r.stderr
