"""Builds libbi_gemm.so in-tree with nvcc for sm_103a (and, on request, its
debug-bounds variant libbi_gemm_debug.so, compiled with -DBI_DEBUG_BOUNDS).

Each .cu file is compiled to an object in parallel, then linked into a shared
library next to this file.  The CUDA runtime is linked statically, so the
library needs nothing at run time but the NVIDIA driver.  No fast-math: the
kernels rely on IEEE division and square root.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbi_gemm.so")
OBJDIR_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libbi_gemm_debug.so")
DEBUG_FLAGS = ["-DBI_DEBUG_BOUNDS"]
SOURCES = ["api.cu", "gemm.cu", "gemm_fused.cu", "rmsnorm.cu", "glue.cu", "noalloc.cu", "logsoftmax.cu", "quant.cu", "attention.cu"]
HEADERS = ["internal.h", "ptx.cuh", "attention.h", "rowmath.cuh", "gemm_kernel.cuh", "bounds.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
              "-fvisibility=hidden", "--expt-relaxed-constexpr"] + ARCH


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbi_gemm.so")


def _fingerprint(debug: bool = False) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "bi_gemm.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + (DEBUG_FLAGS if debug else [])).encode())
    return h.hexdigest()


def _stamp_path(debug: bool = False) -> str:
    return (LIB_DEBUG if debug else LIB) + ".stamp"


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib) or not os.path.exists(_stamp_path(debug)):
        return False
    with open(_stamp_path(debug)) as f:
        return f.read().strip() == _fingerprint(debug)


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    """Compile and link the library if any source changed; returns its path.
    debug=True builds the debug-bounds variant (libbi_gemm_debug.so)."""
    lib_path = LIB_DEBUG if debug else LIB
    objdir = OBJDIR_DEBUG if debug else OBJDIR
    if not force and up_to_date(debug):
        return lib_path
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (DEBUG_FLAGS if debug else []) + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc] + flags + ["-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, " ".join(cmd), r.stdout + r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp.%d" % os.getpid()
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stdout + r.stderr))
    os.replace(tmp, lib_path)
    with open(_stamp_path(debug), "w") as f:
        f.write(_fingerprint(debug))
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
