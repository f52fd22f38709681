"""Build libpointcloud.so (the CUDA kernels + C ABI) in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into ``point_cloud_neighbor_gb300/_build/libpointcloud.so`` against the shared
CUDA runtime.  Floating point flags: no FMA contraction (``--fmad=false``),
IEEE division and square root, subnormals kept (``-ftz=false``) -- the kernels
also spell every operation of the squared distance with round-to-nearest
intrinsics, so the flags are a second line of defence, not the only one.

Usage: ``python -m point_cloud_neighbor_gb300.build [--force] [--verbose]``.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpointcloud.so")

SOURCES = ["pc_api.cu", "pc_fps.cu", "pc_knn.cu", "pc_ball_query.cu",
           "pc_fps_static.cu", "pc_grid.cu", "pc_chamfer.cu", "pc_interp.cu",
           "pc_knn_d.cu"]
HEADERS = ["pc_device.cuh", "pc_tiles.cuh", "pc_filter.cuh", "pc_stream.cuh",
           "pc_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH, "-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-ftz=false",
    "-prec-div=true", "-prec-sqrt=true", "-Xcompiler", "-fPIC",
    "-Xcompiler", "-ffp-contract=off", "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return path


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "pointcloud.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libpointcloud.so."""
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _inputs_mtime():
        return LIB
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp,
           *[o for o, _ in results],
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
