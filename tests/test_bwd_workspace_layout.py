"""The backward's varlen workspace layout, checked on the host with the
library's own row function (`bwd_ws_row0` in the kernel header, which the
preprocess, dQ and dK/dV kernels index by): for random packed batches,
including empty sequences, every sequence's 128-row padded region starts on a
multiple of 4 floats (so each 512-byte bulk copy of it is 16-byte aligned),
no region overlaps the next, and every region ends inside the
total_q + 132*batch + 4 rows per q head that the workspace holds."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_qk_gb300", "csrc")

PROBE = r"""
#include <cstdio>
#include <cstdint>
#include <vector>
#include "fa_kernels.h"
int main() {
  uint64_t state = 12345;
  auto next = [&](uint32_t mod) {   // 64-bit LCG (Knuth's MMIX constants)
    state = state * 6364136223846793005ull + 1442695040888963407ull;
    return static_cast<uint32_t>(state >> 33) % mod;
  };
  for (int trial = 0; trial < 20000; ++trial) {
    const int B = 1 + next(24);
    std::vector<int> cu(B + 1, 0);
    for (int b = 0; b < B; ++b) {
      int len = next(4) == 0 ? 0 : static_cast<int>(next(1100));
      cu[b + 1] = cu[b] + len;
    }
    const int64_t rows = int64_t(cu[B]) + 132 * int64_t(B) + 4;
    int64_t prev_end = 0;
    for (int b = 0; b < B; ++b) {
      const int64_t r0 = fa::bwd_ws_row0(cu.data(), b);
      const int sq = cu[b + 1] - cu[b];
      const int64_t end = r0 + int64_t((sq + 127) / 128) * 128;
      if (r0 % 4 != 0) { std::printf("misaligned %d %d\n", trial, b); return 1; }
      if (r0 < prev_end) { std::printf("overlap %d %d\n", trial, b); return 1; }
      if (end > rows) { std::printf("past the end %d %d\n", trial, b); return 1; }
      if (sq > 0) prev_end = end;
    }
  }
  std::printf("ok\n");
  return 0;
}
"""


def test_varlen_workspace_regions(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    if not os.path.exists(os.path.join(inc, "cuda_runtime.h")) or shutil.which("g++") is None:
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "probe.cpp"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["g++", "-std=c++17", "-I", CSRC, "-I", inc, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
