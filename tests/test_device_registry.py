"""The per-device one-time set-up records of the library (csrc/device_registry.h),
compiled with the host C++ compiler and exercised without a GPU: each
(device, key) setting runs once per device, a failed setting is retried, the
records of different devices are independent, out-of-range ordinals are
refused, and concurrent first calls from many threads run a setting once."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "mla_latent_kv_72_b300", "csrc")

DRIVER = r"""
#include "device_registry.h"
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

int main() {
  mla::DeviceRegistry reg;
  int runs[mla::kMaxDevices][4] = {};
  // device 0, key 1: runs once
  for (int i = 0; i < 5; ++i)
    if (reg.once(0, 1, [&] { ++runs[0][1]; return 0; }) != 0) return 10;
  if (runs[0][1] != 1) return 11;
  // the same key on devices 1 and 3 is a separate setting
  for (int d : {1, 3, 1, 3})
    if (reg.once(d, 1, [&] { ++runs[d][1]; return 0; }) != 0) return 12;
  if (runs[1][1] != 1 || runs[3][1] != 1 || runs[2][1] != 0) return 13;
  // a failing setting reports its error and is retried until it succeeds
  int tries = 0;
  if (reg.once(2, 0, [&] { ++tries; return 7; }) != 7) return 14;
  if (reg.once(2, 0, [&] { ++tries; return 0; }) != 0) return 15;
  if (reg.once(2, 0, [&] { ++tries; return 0; }) != 0) return 16;
  if (tries != 2) return 17;
  // out-of-range ordinals and keys are refused without running anything
  bool ran = false;
  if (reg.once(-1, 0, [&] { ran = true; return 0; }) != -1) return 18;
  if (reg.once(mla::kMaxDevices, 0, [&] { ran = true; return 0; }) != -1) return 19;
  if (reg.once(0, mla::kMaxSetupKeys, [&] { ran = true; return 0; }) != -1) return 20;
  if (ran) return 21;
  // per-device values are computed once per device
  int calls = 0;
  if (reg.value(5, [&] { ++calls; return 10; }, -1) != 10) return 22;
  if (reg.value(5, [&] { ++calls; return 99; }, -1) != 10) return 23;
  if (reg.value(6, [&] { ++calls; return 11; }, -1) != 11) return 24;
  if (calls != 2) return 25;
  if (reg.value(-3, [&] { return 1; }, -7) != -7) return 26;
  // 32 threads race on the first call of 4 devices: each setting runs once
  std::atomic<int> hits[4];
  for (auto& h : hits) h = 0;
  std::vector<std::thread> ts;
  for (int t = 0; t < 32; ++t)
    ts.emplace_back([&, t] {
      for (int rep = 0; rep < 100; ++rep) {
        const int d = 10 + (t + rep) % 4;
        reg.once(d, 3, [&] { ++hits[d - 10]; return 0; });
      }
    });
  for (auto& th : ts) th.join();
  for (auto& h : hits)
    if (h.load() != 1) return 27;
  std::puts("ok");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_device_registry_bookkeeping(tmp_path):
    src = tmp_path / "registry_test.cpp"
    src.write_text(DRIVER)
    exe = tmp_path / "registry_test"
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-pthread", "-I", HEADER_DIR, str(src), "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, f"check {r.returncode} failed"
    assert r.stdout.strip() == "ok"
