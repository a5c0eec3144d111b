"""The GEMM's division-free work-unit mapping (`DivBy` in csrc/gemm.cu): floor(n / d) as a
multiply and a shift with a host-computed multiplier. The struct and its two functions are
taken from the source text, compiled for the host with g++, and compared with integer
division on every numerator below 2^16 for divisors 1 .. 2048, and on random and extreme
numerators (up to 2^31 - 1) for random and extreme divisors (up to 2^31 - 1)."""
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEMM_CU = os.path.join(ROOT, "fp8_mixed_precision_saturating_gb300", "csrc", "gemm.cu")

DRIVER = r"""
#include <cstdint>
#include <cstdio>
%s
int main() {
  unsigned long long bad = 0, n_checked = 0;
  // every numerator below 2^16 for divisors 1 .. 2048
  for (uint32_t d = 1; d <= 2048; ++d) {
    const DivBy m = make_div(d);
    for (uint32_t n = 0; n < 65536; ++n, ++n_checked)
      if (div_by(n, m) != n / d) ++bad;
  }
  // the cases given on stdin: pairs (n, d)
  unsigned long long n, d;
  while (std::scanf("%%llu %%llu", &n, &d) == 2) {
    ++n_checked;
    if (div_by(static_cast<uint32_t>(n), make_div(static_cast<uint32_t>(d))) != n / d) ++bad;
  }
  std::printf("%%llu %%llu\n", bad, n_checked);
  return 0;
}
"""


def _extract():
    src = open(GEMM_CU).read()
    a = src.index("struct DivBy {")
    b = src.index("__host__ __device__ __forceinline__ uint32_t div_by(")
    c = src.index("\n}\n", b) + 3
    return src[a:c].replace("__host__ __device__ __forceinline__", "inline")


def test_div_by_equals_integer_division():
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    code = DRIVER % _extract()
    rng = np.random.default_rng(0)
    pairs = []
    ds = list(rng.integers(1, 1 << 31, 300)) + [(1 << k) for k in range(31)] + [(1 << k) - 1 for k in range(1, 32)] + \
        [(1 << k) + 1 for k in range(1, 31)] + [3, 5, 7, 76, 152, 3 * 16, 12 * 16, 56 * 32]
    for d in ds:
        d = int(d)
        ns = list(rng.integers(0, 1 << 31, 200)) + [(1 << 31) - 1, (1 << 31) - 2, d - 1, d, d + 1, 2 * d - 1, 2 * d]
        pairs += [(int(n), d) for n in ns if 0 <= n < (1 << 31)]
    with tempfile.TemporaryDirectory() as tmp:
        cpp, exe = os.path.join(tmp, "divby.cpp"), os.path.join(tmp, "divby")
        open(cpp, "w").write(code)
        subprocess.run([cxx, "-O2", "-std=c++17", cpp, "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], input="\n".join(f"{n} {d}" for n, d in pairs), capture_output=True, text=True,
                             check=True).stdout.split()
    bad, checked = int(out[0]), int(out[1])
    assert checked == 2048 * 65536 + len(pairs)
    assert bad == 0
