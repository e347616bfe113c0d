"""Build libditattn.so (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: python -m diffusion_transformer_attention_gb300.build_lib [--verbose] [--bounds-check]

The translation units are compiled in parallel and linked with the static CUDA runtime, so the
library loads on machines without a GPU (its calls then return DIT_E_UNSUPPORTED). --bounds-check
builds a debug variant into _lib_bounds/ instead: the attention kernels check their computed global
and shared-memory indices and report one outside its buffer as DIT_E_BOUNDS (set DITATTN_LIBRARY to
its path to load it).
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
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libditattn.so")
SOURCES = ["api.cu", "prepass.cu", "fmha_sm103.cu", "fmha_dense.cu", "fmha_sage_i8.cu", "fmha_sage_f8.cu",
           "fmha_qk16pv8.cu", "fmha_mxfp8.cu", "fmha_nvfp4.cu", "noalloc.cu",
           "host_copy.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libditattn.so")
    return path


BOUNDS_DIR = os.path.join(PKG, "_lib_bounds")


def _compile(src: str, verbose: bool, out_dir: str = OUT_DIR, defines=()) -> str:
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
           *[f"-D{d}" for d in defines], "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    return obj


def build(verbose: bool = False, bounds_check: bool = False) -> str:
    out_dir = BOUNDS_DIR if bounds_check else OUT_DIR
    lib = os.path.join(out_dir, "libditattn.so")
    defines = ("DITATTN_BOUNDS_CHECK",) if bounds_check else ()
    os.makedirs(out_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, out_dir, defines), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, bounds_check="--bounds-check" in sys.argv))
