"""Host checks of the tensor-core kernel's fragment geometry (no GPU): the
channel assignment kchan(r, kq, s) of every code width is a bijection onto the
64 first-half channels and kslot is its inverse, and the rotation-table index
covers its buffer once. Compiled with nvcc as a host program from the same
header the kernels include."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_quantized_kv_append_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "kvq_tc_geom.cuh"
using namespace kvq::tc;
template <int BITS> int check() {
  int seen[64] = {0};
  for (int r = 0; r < 4; ++r)
    for (int kq = 0; kq < 4; ++kq)
      for (int s = 0; s < 4; ++s) {
        const int c = kchan<BITS>(r, kq, s);
        if (c < 0 || c >= 64) return 1;
        if (c / 16 != r) return 2;                      // lane quarter r owns [16r, 16r + 16)
        ++seen[c];
        int r2, kq2, s2;
        kslot<BITS>(c, r2, kq2, s2);
        if (r2 != r || kq2 != kq || s2 != s) return 3;
      }
  for (int c = 0; c < 64; ++c)
    if (seen[c] != 1) return 4;
  return 0;
}
int main() {
  int rc = check<2>() | (check<3>() << 4) | (check<4>() << 8) | (check<8>() << 12);
  int used[kRotFragQuads] = {0};
  for (int w = 0; w < kWarps; ++w)
    for (int nt = 0; nt < 2; ++nt)
      for (int kq = 0; kq < 4; ++kq)
        for (int lane = 0; lane < 32; ++lane) {
          const int i = rot_frag_index(w, nt, kq, lane);
          if (i < 0 || i >= kRotFragQuads) return 100;
          ++used[i];
        }
  for (int i = 0; i < kRotFragQuads; ++i)
    if (used[i] != 1) return 101;
  for (int n = 0; n < 8; ++n)
    if (tperm(tperm(n)) != n) return 102;               // token permutation is an involution
  std::printf("%d\n", rc);
  return rc;
}
"""


def test_fragment_geometry_is_a_bijection():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "geom.cu")
        exe = os.path.join(d, "geom")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.check_call([nvcc, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                               "--expt-relaxed-constexpr", src, "-o", exe])
        r = subprocess.run([exe], capture_output=True, text=True)
        assert r.returncode == 0, f"geometry check failed: code {r.returncode} {r.stdout}"
