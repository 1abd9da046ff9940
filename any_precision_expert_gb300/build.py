"""Build the C-ABI library (libpw.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/`` next to this
file and linked into ``libpw.so`` in the package directory (static CUDA
runtime, so the library only needs the driver at run time).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpw.so")

SOURCES = ["pw_runtime.cpp", "pw_pack.cpp", "pw_planner.cpp", "pw_kernels.cu", "pw_ffn.cu", "pw_decode.cu",
           "pw_prefill.cu", "pw_noalloc.cu"]
# the planner compares doubles: no fused multiply-adds, so x86 and Arm hosts plan alike
SOURCE_FLAGS = {"pw_planner.cpp": ["-Xcompiler", "-ffp-contract=off"]}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags(extra=()):
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
            "-DNDEBUG", *ARCH, *extra]


def _compile(src: str, extra, verbose: bool):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *_flags([*extra, *SOURCE_FLAGS.get(src, [])]), "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every source and link libpw.so; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, verbose), SOURCES))
    if ptxas_info:
        for _, err in results:
            sys.stderr.write(err)
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), "-shared", *ARCH, "--cudart", "static", "-o", tmp] + [o for o, _ in results]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info="-v" in sys.argv)
