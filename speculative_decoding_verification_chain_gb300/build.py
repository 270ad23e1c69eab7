"""Builds libspecverify.so in-tree for sm_103a with nvcc (no cmake)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRCS = [os.path.join(PKG, "csrc", f)
        for f in ("spec_verify.cu", "chain_cluster.cu", "greedy_cluster.cu", "tree_sampled.cu", "next_step.cu", "ngram.cu")]
HDRS = [os.path.join(ROOT, "include", "spec_verify.h"), os.path.join(PKG, "csrc", "common.h"),
        os.path.join(PKG, "csrc", "ptx.cuh"), os.path.join(PKG, "csrc", "twofloat.cuh")]
SRC = SRCS[0]
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


def _flags() -> list:
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def compile_command(src: str, obj: str, verbose_ptxas: bool = False) -> list:
    cmd = [nvcc(), *_flags(), "-c", "-o", obj, src]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    return cmd


def link_command(objs: list, out: str) -> list:
    return [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath," + cuda_lib_dir(), "-o", out, *objs]


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the CUDA library if it is missing or older than its sources.
    The translation units compile in parallel, then link into one .so."""
    newest = max(os.path.getmtime(f) for f in SRCS + HDRS)
    if force or verbose_ptxas or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tag = "%d" % os.getpid()
        objs = [os.path.join(PKG, "csrc", os.path.basename(f) + ".%s.o" % tag) for f in SRCS]
        procs = [subprocess.Popen(compile_command(s, o, verbose_ptxas)) for s, o in zip(SRCS, objs)]
        rcs = [p.wait() for p in procs]
        try:
            for rc, s in zip(rcs, SRCS):
                if rc != 0:
                    raise subprocess.CalledProcessError(rc, "nvcc " + os.path.basename(s))
            tmp = LIB + ".tmp" + tag
            subprocess.check_call(link_command(objs, tmp))
            os.replace(tmp, LIB)
        finally:
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose_ptxas=True)
