"""Builds libspecverify.so in-tree for sm_103a with nvcc (no cmake)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "spec_verify.cu")
HDR = os.path.join(ROOT, "include", "spec_verify.h")
LIB = os.path.join(PKG, "libspecverify.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def cuda_lib_dir() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        d = os.path.join(home, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")) or os.path.isdir(d):
            return d
    return os.path.join(home, "lib64")


def command(out: str = LIB, verbose_ptxas: bool = False) -> list:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "shared", "-Xlinker", "-rpath," + cuda_lib_dir(),
           "-I", os.path.join(ROOT, "include"), "-o", out, SRC]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    return cmd


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the CUDA library if it is missing or older than its sources."""
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if force or verbose_ptxas or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(command(tmp, verbose_ptxas))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose_ptxas=True)
