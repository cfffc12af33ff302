"""Build the CUDA library in-tree: ``exact_tiled_attention_27_gb300/lib/libfa_gb300.so``.

Three translation units (host API, forward kernels, backward kernels) are compiled
in parallel for sm_103a only, then linked into one shared library with the CUDA
runtime linked statically, so the library needs nothing but the driver at run time.

    python -m exact_tiled_attention_27_gb300.build [--force] [--verbose]
"""

from __future__ import annotations

import argparse
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
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libfa_gb300.so")

SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "decode.cu", "noalloc.cu", "fwd_fp8.cu", "quant.cu"]
HEADERS = ["ptx.cuh", "internal.h", "fwd_tiles.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc():
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found")
    return exe


def _mtime(path):
    return os.path.getmtime(path) if os.path.exists(path) else -1.0


def _deps_mtime():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "fa.h"), __file__]
    return max(_mtime(f) for f in files)


def _compile(src, verbose):
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
    if verbose:
        sys.stderr.write(p.stderr)
    log = os.path.join(BUILD, src + ".ptxas.txt")
    with open(log, "w") as f:
        f.write(p.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link if any source is newer than the library; return its path."""
    if not force and _mtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
