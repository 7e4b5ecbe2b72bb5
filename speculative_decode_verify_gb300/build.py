"""Compile the CUDA library (libverify_attn.so) for sm_103a with nvcc, in-tree.

Each ``csrc/*.cu`` file is compiled to an object in parallel, then linked into one shared
library with the CUDA runtime linked statically (so the library loads on a machine without a
GPU driver; it only needs one when a call launches work).  Whole-program compilation: no
``-rdc``.  Exported symbols are the ``VA_API`` functions of ``include/verify_attn.h``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def lib_path(variant: str = "") -> str:
    return os.path.join(BUILD_DIR, f"libverify_attn{variant}.so")


def _sources():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return srcs, deps


def build(variant: str = "", defines=(), force: bool = False, verbose_ptxas: bool = False) -> str:
    """Build libverify_attn{variant}.so; returns its path.  Rebuilds only if a source changed."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    out = lib_path(variant)
    srcs, deps = _sources()
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(p) for p in deps)
        if os.path.getmtime(out) >= newest:
            return out
    obj_dir = os.path.join(BUILD_DIR, f"obj{variant}")
    os.makedirs(obj_dir, exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
              "-Xcompiler", "-fPIC,-fvisibility=hidden", *[f"-D{d}" for d in defines]]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        proc = subprocess.run(common + ["-c", src, "-o", obj], capture_output=True, text=True)
        if proc.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{proc.stdout}\n{proc.stderr}")
        return obj, proc.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose_ptxas:
        for _, err in results:
            if err.strip():
                print(err)
    tmp = out + f".tmp{os.getpid()}"
    link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    proc = subprocess.run(link, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{proc.stdout}\n{proc.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
