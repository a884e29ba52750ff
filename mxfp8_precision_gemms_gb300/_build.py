"""Compile the CUDA sources into the in-tree shared library ``libmxfp8.so``.

sm_103a only (``-gencode arch=compute_103a,code=sm_103a``); the translation
units compile in parallel, then link with nvcc (static CUDA runtime).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmxfp8.so")
# the bounds-checked build (index checks that record a status, see
# csrc/mx_common.cuh): test infrastructure, same sources
LIB_BC = os.path.join(PKG, "libmxfp8_bc.so")
BUILD_BC = os.path.join(PKG, "_build_bc")
SOURCES = ["api.cu", "quantize.cu", "fused.cu", "gemm.cu"]
HEADERS = ["ptx.cuh", "mx_common.cuh", "internal.h", "swiglu_round.cuh", "ff_consts.h"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-O2",
    "--expt-relaxed-constexpr",
    "-I" + os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    paths.append(os.path.join(ROOT, "include", "mxfp8.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, bounds_check: bool = False) -> str:
    """Build libmxfp8.so (libmxfp8_bc.so with bounds_check) if any source is
    newer than it; return its path."""
    lib, bdir = (LIB_BC, BUILD_BC) if bounds_check else (LIB, BUILD)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DMXFP8_BOUNDS_CHECK"] if bounds_check else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([cc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
