"""The per-device set-up cache of the launchers (csrc/devcache.h) on the host:
one value per device ordinal, made once by the first call with that device
current, kept for later calls, and made once even when threads race.  The
header is plain C++; a small driver program exercises it."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "trellis_coded_weight_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "devcache.h"

int main() {
  trellis::PerDevice<int> cache;
  int made[trellis::kMaxDevices] = {};
  // first use per device computes; a second device gets its own value
  int a = cache.get(0, [&] { ++made[0]; return 100; }, -1);
  int b = cache.get(1, [&] { ++made[1]; return 200; }, -1);
  int a2 = cache.get(0, [&] { ++made[0]; return 999; }, -1);
  int b2 = cache.get(1, [&] { ++made[1]; return 999; }, -1);
  // out-of-range ordinals return the fallback and make nothing
  int neg = cache.get(-1, [&] { return 1; }, -7);
  int big = cache.get(trellis::kMaxDevices, [&] { return 1; }, -8);
  // many threads on a fresh device: made exactly once, all see the same value
  std::atomic<int> calls{0};
  std::vector<std::thread> th;
  std::vector<int> seen(16, 0);
  for (int i = 0; i < 16; ++i)
    th.emplace_back([&, i] { seen[i] = cache.get(5, [&] { calls.fetch_add(1); return 500 + 0 * i; }, -1); });
  for (auto& t : th) t.join();
  int same = 1;
  for (int v : seen) same &= (v == 500);
  std::printf("%d %d %d %d %d %d %d %d %d %d\n", a, b, a2, b2, made[0], made[1], neg, big, calls.load(), same);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_per_device_cache(tmp_path):
    src = tmp_path / "drv.cc"
    src.write_text(DRIVER)
    exe = tmp_path / "drv"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split()
    assert [int(v) for v in out] == [100, 200, 100, 200, 1, 1, -7, -8, 1, 1]
