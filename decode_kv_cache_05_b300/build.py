"""Builds librkv.so (the CUDA library) in-tree for sm_103a with nvcc.

Usage: python -m decode_kv_cache_05_b300.build [--force] [--verbose-ptxas]
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "librkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def inputs() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "rkv.h")]


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in inputs())


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           "-I", INCLUDE, "-I", CSRC, "-o", tmp, *sources()]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines: dict, force: bool = False) -> str:
    """A test build of the library with extra preprocessor definitions, as
    librkv_<name>.so next to librkv.so. Used only by tests (for instance the
    one that makes a bounded in-kernel wait run out); never loaded by the
    package itself."""
    out = os.path.join(PKG, f"librkv_{name}.so")
    if not force and os.path.exists(out) and all(os.path.getmtime(f) <= os.path.getmtime(out) for f in inputs()):
        return out
    tmp = out + f".tmp{os.getpid()}"
    flags = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           *flags, "-I", INCLUDE, "-I", CSRC, "-o", tmp, *sources()]
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv)
    print(LIB)
