"""The CTA split of the GEMV stages, on the host: unit_at_cost and split_target
(moe_expert_layer_gemv_gb300/csrc/common.cuh, host-and-device functions)
compiled into a small host program and checked against brute force.

unit_at_cost(target, ...) must return the unit whose cost interval holds the
target, for both unit numberings (group-major, tile-major), both cost models
(tok_w 0 and 1) and ragged last groups; split_target must start at 0, never
decrease in c and end at the stage's static cost (all of it, or the static
share when the stage has a dynamic tail), with and without the down skew."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r'''
#include <cstdio>
#include <vector>
#include "common.cuh"
using namespace moe;

static unsigned long long st = 0x9e3779b97f4a7c15ULL;
static int rnd(int lo, int hi) {
  st = st * 6364136223846793005ULL + 1442695040888963407ULL;
  return lo + (int)((st >> 33) % (unsigned long long)(hi - lo + 1));
}

int main() {
  long fails = 0, checks = 0;
  for (int it = 0; it < 3000; ++it) {
    const int n = rnd(1, 40), xt = rnd(1, 8), tiles = rnd(1, 24), base = rnd(1, 16);
    const int tw = rnd(0, 1);
    const bool tm = rnd(0, 1) != 0;
    const int groups = (n + xt - 1) / xt;
    std::vector<int> cost(tiles * groups);
    for (int t = 0; t < tiles; ++t)
      for (int g = 0; g < groups; ++g) {
        const int nt = g < groups - 1 ? xt : n - (groups - 1) * xt;
        cost[tm ? t * groups + g : g * tiles + t] = base + tw * nt;
      }
    const int c0 = rnd(0, 5000), u0 = rnd(0, 5000);
    int cum = 0;
    for (int u = 0; u < (int)cost.size(); ++u) {
      for (int r = cum; r < cum + cost[u]; ++r) {
        ++checks;
        const int got = unit_at_cost(c0 + r, c0, u0, tiles, n, xt, base, tw, tm);
        if (got != u0 + u && fails++ < 5)
          printf("unit_at_cost n=%d xt=%d tiles=%d base=%d tw=%d tm=%d r=%d: %d, want %d\n", n,
                 xt, tiles, base, tw, (int)tm, r, got - u0, u);
      }
      cum += cost[u];
    }
  }
  for (int it = 0; it < 3000; ++it) {
    const int grid = rnd(1, 1024), cost = rnd(0, 2000000);
    const bool tail = rnd(0, 1) != 0;
    const float skew = rnd(0, 1) ? kDownSkew : 0.f;
    const int fcost = tail ? (int)(kStaticShare * (float)cost) : cost;
    int prev = -1;
    for (int c = 0; c <= grid; ++c) {
      ++checks;
      const int v = split_target(c, grid, cost, tail, skew);
      const bool bad = (c == 0 && v != 0) || v < prev || v > fcost || (c == grid && v != fcost);
      if (bad && fails++ < 5)
        printf("split_target grid=%d cost=%d tail=%d skew=%g c=%d: %d (prev %d, end %d)\n", grid,
               cost, (int)tail, skew, c, v, prev, fcost);
      prev = v;
    }
  }
  printf("checks %ld fails %ld\n", checks, fails);
  return fails != 0;
}
'''


def test_unit_at_cost_and_split_target_against_brute_force(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc"
                                    if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("no nvcc")
    src = tmp_path / "split_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "split_check"
    csrc = os.path.join(ROOT, "moe_expert_layer_gemv_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-O2", f"-I{csrc}", f"-I{os.path.join(ROOT, 'include')}",
                    "-o", str(exe), str(src)], check=True, capture_output=True, timeout=300)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fails 0" in r.stdout
