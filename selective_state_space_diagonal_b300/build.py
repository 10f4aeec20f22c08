"""Builds ``libcsscan.so`` in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", "csscan.cu")]
HEADERS = [os.path.join(HERE, "csrc", f) for f in ("scan_kernels.cuh", "device_util.cuh", "decode_kernel.cuh", "backward_kernels.cuh", "mimo_kernels.cuh")] + \
          [os.path.join(ROOT, "include", "csscan.h")]
OUTPUT = os.path.join(HERE, "libcsscan.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", "-I" + os.path.join(ROOT, "include")]


def up_to_date(output: str = OUTPUT) -> bool:
    if not os.path.exists(output):
        return False
    t = os.path.getmtime(output)
    return all(os.path.getmtime(s) <= t for s in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return OUTPUT
    cmd = [NVCC, *FLAGS, "-o", OUTPUT, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return OUTPUT


if __name__ == "__main__":
    print(build(force=True, verbose=True))
