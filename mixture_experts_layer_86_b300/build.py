"""Builds the in-tree shared library ``libmoe_b300.so`` for sm_103a with nvcc.

Usage: ``python -m mixture_experts_layer_86_b300.build [--force]``.
Object files go to ``_build/`` at the repository root; the library is written
next to this file so that it travels with the package.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe_b300.so")

SOURCES = ["api.cu", "route.cu", "dispatch.cu", "gemm_simt.cu", "gemm_tc.cu", "gate_tc.cu",
           "gate_route.cu", "gate_static.cu", "backward.cu"]
HEADERS = ["common.cuh", "kernels.h", "tc_ptx.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
         "-Xcompiler", "-fPIC,-O3", "-Xptxas", "-v",
         "-I", INCLUDE, "-I", CSRC]


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else 0.0


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "moe_b300.h"),
                                                         os.path.abspath(__file__)]
    return max(_mtime(f) for f in files)


def _compile(src: str, force: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    s = os.path.join(CSRC, src)
    if not force and _mtime(obj) > max(_mtime(s), _deps_mtime()):
        return obj
    log = os.path.join(BUILD, os.path.splitext(src)[0] + ".ptxas.log")
    cmd = [NVCC, *ARCH, *FLAGS, "-c", s, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as fh:
        fh.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False) -> str:
    """Compile (if stale) and link the library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force), SOURCES))
    if force or _mtime(LIB) < max(_mtime(o) for o in objs):
        cmd = [NVCC, *ARCH, "-shared", "-o", LIB, *objs, "-lcudart_static", "-ldl", "-lrt",
               "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
