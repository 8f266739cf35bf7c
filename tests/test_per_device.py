"""Per-device one-time set-up (kernel attributes, cached SM counts) is kept per CUDA device, so a process
that uses several GPUs sets up each one. The bookkeeping (PerDeviceOnce in csrc/cqsa_internal.h) is
compiled here with the host compiler and exercised without a GPU: marks are per device id, ids outside
[0, 64) are never marked, and concurrent marks from several threads all land."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_long_context_tcgen05_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "cqsa_internal.h"
int main() {
  cqsa::PerDeviceOnce once;
  int fails = 0;
  auto check = [&](bool c, const char* what) { if (!c) { std::printf("FAIL %s\n", what); ++fails; } };
  check(!once.seen(0) && !once.seen(1), "fresh");
  once.mark(0);
  check(once.seen(0) && !once.seen(1), "device 0 only");
  once.mark(1);
  check(once.seen(0) && once.seen(1) && !once.seen(2), "devices 0 and 1");
  once.mark(-1);
  once.mark(64);
  check(!once.seen(-1) && !once.seen(64), "out of range ids ignored");
  once.mark(63);
  check(once.seen(63), "device 63");
  cqsa::PerDeviceOnce par;
  std::vector<std::thread> th;
  for (int t = 0; t < 8; ++t)
    th.emplace_back([&par, t] { for (int d = t; d < 64; d += 8) par.mark(d); });
  for (auto& x : th) x.join();
  bool all = true;
  for (int d = 0; d < 64; ++d) all = all && par.seen(d);
  check(all, "concurrent marks");
  std::printf(fails ? "failed\n" : "ok\n");
  return fails ? 1 : 0;
}
"""


def test_per_device_once_bookkeeping(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.isdir(CUDA_INC):
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "per_device.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "per_device"
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-I",
                    CUDA_INC, str(src), "-o", str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
