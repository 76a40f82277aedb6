"""Build libspecverify.so in-tree for sm_103a with nvcc (no CMake, no torch extension machinery)."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "spec_verify.cu")
SRC_CTRL = os.path.join(PKG, "csrc", "spec_control.cpp")
HDR = os.path.join(ROOT, "include", "spec_verify.h")
HDR_CTRL = os.path.join(ROOT, "include", "spec_control.h")
LIB = os.path.join(PKG, "libspecverify.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in (SRC, SRC_CTRL, HDR, HDR_CTRL, __file__))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; returns its path."""
    if not force and not stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), SRC, SRC_CTRL, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)  # atomic: a process that already mapped the old file keeps it intact
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
