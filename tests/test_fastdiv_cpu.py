"""The kernels' multiply-and-shift division (csrc/fastdiv.h) against the CPU's own integer
division, compiled with the host compiler: every divisor up to 4096 against the numerators
0..20000 and the top of the range, plus random and extreme divisors up to 2^31 - 1."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "fastdiv.h"
using attn::FastDiv;
static long bad = 0, checked = 0;
static void check(uint32_t d, uint32_t n) {
  const FastDiv f = FastDiv::make(d);
  ++checked;
  if (f.div(n) != n / d || f.mod(n) != n % d) {
    if (bad < 10) std::printf("d=%u n=%u got %u/%u want %u/%u\n", d, n, f.div(n), f.mod(n), n / d, n % d);
    ++bad;
  }
}
int main() {
  const uint32_t top = 0x7fffffffu;
  for (uint32_t d = 1; d <= 4096; ++d) {
    for (uint32_t n = 0; n <= 20000; ++n) check(d, n);
    for (uint32_t k = 0; k < 64; ++k) check(d, top - k);
    for (uint32_t q = 1; q < 2000; q += 7) {  // around multiples of d
      const uint64_t x = (uint64_t)q * d;
      for (int e = -1; e <= 1; ++e)
        if (x + e <= top && (int64_t)x + e >= 0) check(d, (uint32_t)(x + e));
    }
  }
  std::mt19937 rng(12345);
  for (int i = 0; i < 2000000; ++i) {
    const uint32_t d = 1 + rng() % top;
    const uint32_t n = rng() % (top + 1u);
    check(d, n);
    check(d, top);
    check(d, d - 1);
    check(d, d);
  }
  for (uint32_t l = 0; l < 31; ++l) {
    const uint32_t p = 1u << l;
    for (uint32_t d : {p, p + 1, p - 1 ? p - 1 : 1u}) {
      check(d, top);
      check(d, 0);
      check(d, top / d * d);
      if (top / d * d > 0) check(d, top / d * d - 1);
    }
  }
  check(top, top);
  check(top, top - 1);
  std::printf("checked %ld bad %ld\n", checked, bad);
  return bad != 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "fastdiv_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I",
                    os.path.join(ROOT, "attention_sm_flash_gb300", "csrc"), str(src), "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout
    assert " bad 0" in out.stdout
