"""Build libnf4q.so (the CUDA kernels and their C ABI) in-tree for sm_103a.

    python -m dequant_matmul_quantize_b300.build [--verbose]

The library is one translation unit, ``csrc/nf4q.cu``.  The CUDA runtime is
linked statically, so the .so only needs the driver at run time.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "nf4q.cu")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libnf4q.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    out = [SRC, os.path.join(INCLUDE, "nf4q.h")]
    csrc = os.path.join(PKG, "csrc")
    out += [os.path.join(csrc, f) for f in os.listdir(csrc)
            if f.endswith((".cuh", ".h", ".cu"))]
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    cmd = [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "-I", INCLUDE, "-I", os.path.join(PKG, "csrc"),
           "-o", LIB + ".tmp", SRC]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="--verbose" in sys.argv)
    print(LIB)
