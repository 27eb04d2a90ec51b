"""The launch helper's per-device record of the dynamic shared-memory limit (host only).

cudaFuncSetAttribute applies to the current device, so every device must get the attribute
before its first large launch, however large the launches on other devices were; host threads
launching at once must neither race on the record nor skip a device. The record is compiled
here with a fake setter that logs its calls.
"""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "persistent_megakernel_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include <atomic>
#include "smem_attr.h"
using decimpl::SmemAttrCache;

int main() {
  SmemAttrCache c;
  std::vector<int> calls;
  auto ok = [&](size_t b) { calls.push_back((int)b); return 0; };
  // device 0 raised to 200000; device 1 still needs its own call, even for less
  std::printf("%d ", c.ensure(0, 200000, ok));
  std::printf("%d ", c.ensure(1, 100000, ok));
  std::printf("%d ", c.ensure(0, 150000, ok));   // no call: device 0 allows more already
  std::printf("%d ", c.ensure(1, 180000, ok));   // call: larger than device 1's record
  std::printf("%d ", c.ensure(-1, 1000, ok));    // untracked device: always called
  std::printf("%d ", c.ensure(64, 1000, ok));
  std::printf("%d ", c.ensure(64, 1000, ok));
  // a failing setter leaves the record unchanged and returns its code
  std::printf("%d ", c.ensure(2, 50000, [](size_t) { return 7; }));
  std::printf("%zu %zu %zu ", c.allowed(0), c.allowed(1), c.allowed(2));
  std::printf("%zu ", calls.size());
  for (int v : calls) std::printf("%d ", v);
  // 8 threads x 1000 launches on 4 devices: each device is set once per new maximum
  SmemAttrCache d;
  std::atomic<int> n{0};
  std::vector<std::thread> th;
  for (int i = 0; i < 8; ++i)
    th.emplace_back([&] {
      for (int k = 0; k < 1000; ++k) d.ensure(k % 4, 100000, [&](size_t) { n++; return 0; });
    });
  for (auto& x : th) x.join();
  std::printf("%d %zu\n", n.load(), d.allowed(3));
  return 0;
}
"""


def test_per_device_records(tmp_path):
    src = tmp_path / "t.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)]).split()
    vals = [int(x) for x in out]
    rets, allowed, ncalls = vals[:8], vals[8:11], vals[11]
    assert rets == [0, 0, 0, 0, 0, 0, 0, 7]
    assert allowed == [200000, 180000, 0]
    assert ncalls == 6
    assert vals[12:12 + ncalls] == [200000, 100000, 180000, 1000, 1000, 1000]
    assert vals[12 + ncalls:] == [4, 100000]
