"""Builds libmuon.so in-tree for sm_103a with nvcc (no cmake, no torch).

    python -m newton_schulz_06_gb300.build [--force]

Translation units compile in parallel; a unit is rebuilt only when it or a
header is newer than its object.  The shared library links the CUDA runtime
statically and resolves the one driver function it needs
(cuTensorMapEncodeTiled) at run time, so it loads on any machine with the
NVIDIA driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmuon.so")
SOURCES = ["ew_kernels.cu", "ns_kernels.cu", "ns2_kernels.cu", "muon_api.cpp",
           "muon_noalloc.cu"]
HEADERS = [os.path.join(CSRC, "muon_internal.h"), os.path.join(CSRC, "tc_ptx.cuh"),
           os.path.join(ROOT, "include", "muon.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return exe


def _flags():
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _compile(src: str, force: bool) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src + ".o")
    deps = [path] + HEADERS
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in deps)):
        return obj
    cmd = [nvcc()] + _flags() + ["-x", "cu", "-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force), SOURCES))
    if (force or not os.path.exists(LIB)
            or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs)):
        tmp = LIB + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
