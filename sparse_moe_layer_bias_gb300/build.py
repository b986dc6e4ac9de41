"""Build liblmoe.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled in parallel to an object under
_build/ (git-ignored), then linked into sparse_moe_layer_bias_gb300/liblmoe.so.
An up-to-date library is not rebuilt.  build(debug=True) makes
liblmoe_debug.so instead: the same sources with -DLMOE_DEBUG, whose kernels
check every index they read from a device list (objects under _build/debug).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "liblmoe.so")
LIB_DEBUG = os.path.join(PKG, "liblmoe_debug.so")
SOURCES = ["gemm.cu", "gemm_pair.cu", "splitk.cu", "gemm_bwd.cu", "backward.cu", "pack.cu", "route.cu", "route_static.cu", "combine.cu", "qb.cu",
           "selftest.cu", "lmoe_api.cu"]
HEADERS = ["kernels.h", "ptx.cuh", "gemm_kernel.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build liblmoe.so")


def _newest_dep() -> float:
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "lmoe.h"))
    deps.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_dep():
        return lib
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = FLAGS + (["-DLMOE_DEBUG"] if debug else []) + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *flags, "-I", os.path.join(ROOT, "include"), "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
