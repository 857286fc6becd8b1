"""The library raises kernel attributes (dynamic shared memory, cluster size)
once per kernel AND device: such an attribute holds per device context, so
a process that runs on device 0 and then on device 1 must set it again on
device 1. This compiles the host-only bookkeeping class with g++ and checks
its keying without a GPU."""
import os
import subprocess

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "vision_transformer_sparse_route_b300", "csrc")

PROGRAM = r"""
#include "per_device.h"
#include <cstdio>
int main() {
  bra::PerDeviceOnce once;
  int k1 = 0, k2 = 0;
  const void *a = &k1, *b = &k2;
  int fails = 0;
  fails += once.done(0, a);            // nothing marked yet
  once.mark(0, a);
  fails += !once.done(0, a);           // marked on device 0
  fails += once.done(1, a);            // the same kernel on device 1 is not
  fails += once.done(0, b);            // another kernel on device 0 is not
  once.mark(1, a);
  once.mark(1, a);                     // marking twice is harmless
  fails += !once.done(1, a);
  fails += once.done(1, b);
  std::printf("%d\n", fails);
  return fails;
}
"""


def test_attribute_cache_is_keyed_by_device_and_kernel(tmp_path):
    src = tmp_path / "t.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe),
                           "-lpthread"])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert out.stdout.strip() == "0"
