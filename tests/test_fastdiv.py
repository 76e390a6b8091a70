"""Host check of the kernels' division by invariant integers (csrc/fastdiv.h):
compiled with the host compiler and compared with the `/` and `%` operators
over edge cases and random operands."""
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "softmax_attention_backward_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "fastdiv.h"
using namespace attn;
static uint64_t state = 88172645463325252ull;
static uint32_t next32() { state ^= state << 13; state ^= state >> 7; state ^= state << 17; return (uint32_t)state; }
int main() {
  const uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 8u, 9u, 16u, 24u, 32u, 64u, 100u, 127u, 128u, 129u, 152u, 255u,
                         256u, 1000u, 4096u, 65535u, 65536u, 1000003u, 2147483647u, 2147483648u,
                         4294967295u};
  const uint32_t ns[] = {0u, 1u, 2u, 3u, 127u, 128u, 65535u, 65536u, 2147483647u, 2147483648u,
                         4294967294u, 4294967295u};
  long bad = 0, checked = 0;
  auto check = [&](uint32_t n, const FastDiv& f) {
    ++checked;
    if (fdiv(n, f) != n / f.d || fmod_u(n, f) != n % f.d) {
      if (bad < 5) std::printf("mismatch n=%u d=%u got %u want %u\n", n, f.d, fdiv(n, f), n / f.d);
      ++bad;
    }
  };
  for (uint32_t d : ds) {
    const FastDiv f = make_fastdiv(d);
    for (uint32_t n : ns) check(n, f);
    for (uint32_t k = 0; k < 64; ++k) {   // around multiples of d
      const uint64_t base = (uint64_t)d * (next32() % 1024u);
      for (int o = -2; o <= 2; ++o) {
        const int64_t n = (int64_t)base + o;
        if (n >= 0 && n <= 4294967295ll) check((uint32_t)n, f);
      }
    }
    for (int k = 0; k < 20000; ++k) check(next32(), f);
  }
  for (int k = 0; k < 2000; ++k) {
    uint32_t d = next32() >> (next32() % 32u);
    if (d == 0) d = 1;
    const FastDiv f = make_fastdiv(d);
    for (int j = 0; j < 200; ++j) check(next32() >> (next32() % 32u), f);
  }
  std::printf("checked %ld bad %ld\n", checked, bad);
  return bad ? 1 : 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_fastdiv_matches_division(tmp_path):
    src = tmp_path / "fd.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fd"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
