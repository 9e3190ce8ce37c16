"""The once-per-device set-up (csrc/per_device.h) on the host, no GPU: a
kernel attribute set on one device must be set again on the next device a
process uses, never twice on one device while it succeeded, retried after a
failure, and refused for a device index out of range. Compiled with g++ and
run under several host threads."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "trellis_quantized_linear_rot_gb300", "csrc")

PROGRAM = r"""
#include "per_device.h"
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>

int main() {
  tfx::PerDeviceOnce<4> once;
  std::atomic<int> calls[4] = {};
  int fail_next = 1;  // device 2's first set-up fails
  auto setup = [&](int dev) {
    return [&, dev] {
      calls[dev]++;
      if (dev == 2 && fail_next) { fail_next = 0; return 7; }
      return 0;
    };
  };
  // Device 0 from many threads at once: one set-up.
  std::vector<std::thread> th;
  for (int i = 0; i < 16; ++i) th.emplace_back([&] { if (once.run(0, -1, setup(0)) != 0) std::abort(); });
  for (auto& t : th) t.join();
  if (calls[0] != 1) { std::printf("device 0 set up %d times\n", calls[0].load()); return 1; }
  // A second device gets its own set-up.
  if (once.run(1, -1, setup(1)) != 0 || calls[1] != 1) { std::printf("device 1 not set up\n"); return 1; }
  if (once.run(1, -1, setup(1)) != 0 || calls[1] != 1) { std::printf("device 1 set up twice\n"); return 1; }
  // A failed set-up returns its error and is retried.
  if (once.run(2, -1, setup(2)) != 7) { std::printf("device 2 error lost\n"); return 1; }
  if (once.run(2, -1, setup(2)) != 0 || calls[2] != 2) { std::printf("device 2 not retried\n"); return 1; }
  if (once.run(2, -1, setup(2)) != 0 || calls[2] != 2) { std::printf("device 2 set up again\n"); return 1; }
  // Out of range.
  if (once.run(4, -9, setup(0)) != -9 || once.run(-1, -9, setup(0)) != -9) { std::printf("range\n"); return 1; }
  if (calls[0] != 1 || calls[3] != 0) { std::printf("stray set-up\n"); return 1; }
  std::printf("ok\n");
  return 0;
}
"""


def test_per_device_once(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "per_device_test.cc"
    exe = tmp_path / "per_device_test"
    src.write_text(PROGRAM)
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I" + CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
