"""Host-side check of the per-device launch cache (PerDeviceOnce in csrc/internal.h): many host
threads racing to the first launch on a device run the initialisation once, and every thread
reads the finished data. Compiled with the host compiler; no GPU and no CUDA call involved."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "int4_w4a16_group_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>
#include "internal.h"

struct Data { int a, b; };

int main() {
  w4a16::PerDeviceOnce<Data> cache;
  std::atomic<int> inits{0}, bad{0}, go{0};
  std::vector<std::thread> ts;
  for (int t = 0; t < 32; ++t)
    ts.emplace_back([&, t] {
      while (!go.load()) {}
      const int dev = t % 4;
      const Data* d = nullptr;
      const cudaError_t e = cache.get(dev, [&](Data& x) {
        inits.fetch_add(1);
        x.a = 100 + dev;
        std::this_thread::yield();
        x.b = 200 + dev;
        return cudaSuccess;
      }, &d);
      if (e != cudaSuccess || d->a != 100 + dev || d->b != 200 + dev) bad.fetch_add(1);
    });
  go.store(1);
  for (auto& th : ts) th.join();
  std::printf("%d %d\n", inits.load(), bad.load());
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.exists(CUDA_INC),
                    reason="needs g++ and the CUDA headers")
def test_concurrent_first_use_initialises_once(tmp_path):
    src = tmp_path / "once.cpp"
    exe = tmp_path / "once"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-O2", "-pthread", "-I", CSRC, "-I", CUDA_INC, str(src),
                    "-o", str(exe)], check=True, capture_output=True)
    for _ in range(20):
        out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
        assert out == ["4", "0"], out  # one initialisation per device, no torn reads
