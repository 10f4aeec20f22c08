"""Builds ``libcsscan.so`` in-tree with nvcc for sm_103a (B300).

The library is several translation units (the C ABI, the forward and backward scans per input
dtype, the MIMO scan), compiled in parallel into ``_build/`` and linked into one shared object
with the CUDA runtime linked statically.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("csscan.cu", "forward_f32.cu", "forward_bf16.cu", "backward_f32.cu",
                                           "backward_bf16.cu", "mimo_f32.cu", "mimo_bf16.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("scan_kernels.cuh", "nscan_kernels.cuh", "device_util.cuh",
                                           "decode_kernel.cuh", "backward_kernels.cuh", "ngrad_kernels.cuh", "mimo_kernels.cuh", "mscan_kernels.cuh",
                                           "mgrad_kernels.cuh",
                                           "forward_launch.cuh", "backward_launch.cuh", "mimo_launch.cuh", "host_common.h")] + \
          [os.path.join(ROOT, "include", "csscan.h")]
OUTPUT = os.path.join(HERE, "libcsscan.so")
BUILD_DIR = os.path.join(HERE, "_build")
# the bounds-checked variant (compiled with CSSCAN_BOUNDS_CHECK): see build_checked
CHECKED_OUTPUT = os.path.join(HERE, "libcsscan_checked.so")
CHECKED_BUILD_DIR = os.path.join(HERE, "_build_checked")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include")]


def up_to_date(output: str = OUTPUT) -> bool:
    if not os.path.exists(output):
        return False
    t = os.path.getmtime(output)
    return all(os.path.getmtime(s) <= t for s in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False, output: str = OUTPUT, defines=(), build_dir: str = BUILD_DIR,
          jobs: int = 0) -> str:
    """Compile every unit (in parallel) and link ``output``. ``defines`` are extra ``-D``
    macros (compile-time tuning knobs of the kernels) and go with their own ``build_dir``."""
    if not force and not defines and output == OUTPUT and up_to_date(output):
        return output
    os.makedirs(build_dir, exist_ok=True)
    extra = [f"-D{d}" for d in defines] + (["-Xptxas=-v"] if verbose else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
        subprocess.run([NVCC, *FLAGS, *extra, "-c", "-o", obj, src], check=True)
        return obj

    jobs = jobs or min(len(SOURCES), os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=jobs) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    subprocess.run([NVCC, *ARCH, "-shared", "-cudart", "static", "-o", output, *objs], check=True)
    return output


def build_checked(force: bool = False) -> str:
    """The bounds-checked library: the same sources compiled with CSSCAN_BOUNDS_CHECK, under which
    the kernels range-check their shared-memory and global indices, record CSSCAN_ERR_BOUNDS for
    csscan_get_device_status and redirect the access instead of leaving its array (a debugging
    build; slower than libcsscan.so)."""
    if not force and up_to_date(CHECKED_OUTPUT):
        return CHECKED_OUTPUT
    return build(force=True, output=CHECKED_OUTPUT, defines=("CSSCAN_BOUNDS_CHECK",), build_dir=CHECKED_BUILD_DIR)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
