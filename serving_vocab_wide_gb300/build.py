"""Build step for the CUDA library: one nvcc invocation for sm_103a.

Produces ``serving_vocab_wide_gb300/_build/libsvw.so`` in-tree.  Needs only
nvcc and a host C++ compiler (no cmake, no PyTorch headers).
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libsvw.so")
SOURCES = ["api.cu", "verify.cu", "early.cu", "filtered.cu", "opd.cu", "fused.cu", "lengthhead.cu", "noalloc.cu"]
HEADERS = ["svw_device.cuh", "svw_internal.h", "svw_sample.cuh", "opd_common.cuh"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise FileNotFoundError("nvcc not found")


def _inputs():
    root = os.path.dirname(HERE)
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(root, "include", "svw.h"), os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        t = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(p) <= t for p in _inputs()):
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "--threads", "0", "-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True, cwd=CSRC)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
