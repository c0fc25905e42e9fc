"""Builds libgqa_attn.so for sm_103a with nvcc (in-tree, next to this file)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgqa_attn.so")
SOURCES = [os.path.join(CSRC, "attn_fwd.cu")]
# every header under csrc/ (and the public one) is a dependency of the library
HEADERS = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
DEPENDS = SOURCES + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "gqa_attn.h")]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False, out: str = LIB) -> str:
    if not force and not is_stale(out):
        return out
    cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-o", out + ".tmp", *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
