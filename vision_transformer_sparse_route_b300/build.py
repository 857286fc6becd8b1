"""Builds libbra.so (the CUDA library behind include/bra.h) in-tree with nvcc
for sm_103a. Run as `python -m vision_transformer_sparse_route_b300.build`."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libbra.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

SOURCES = ["bra.cu"]
DEPS = ["bra.cu", "ptx.cuh", "route.cuh", "attend_bf16.cuh", "attend_f32.cuh", "per_device.h",
        "attend_image.cuh", "attend_tc.cuh", "tcgen05.cuh", "forward_image.cuh", "qkv_tc.cuh",
        "block.cuh", "backward.cuh"]


def nvcc_command(out: str, extra: list[str] | None = None) -> list[str]:
    return [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
            "-use_fast_math", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
            "-o", out] + [os.path.join(CSRC, s) for s in SOURCES] + (extra or [])


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    paths = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(ROOT, "include", "bra.h")]
    return any(os.path.getmtime(p) > t for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    if force or stale():
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else None)
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
