"""Build libnvfp4_ggemm.so in-tree with nvcc for sm_103a.

    python -m block_scaled_fp4_grouped_gb300.build [--force] [--verbose] [--debug]

Each translation unit is compiled in parallel to an object under `_build/`,
then linked (CUDA runtime linked statically; the driver's tensor-map encoder
is fetched at run time, so loading the library needs no GPU driver).
--debug builds libnvfp4_ggemm_debug.so (objects under `_build_debug/`) with
-DNVFP4_DEBUG: the GEMM kernel then checks every shared-memory and TMEM
range, TMA coordinate and alignment before the operation it guards, and a
failed check is reported through the plan's error word (the operation is
skipped and the kernel ends through its abort flag) instead of running.
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
LIB = os.path.join(PKG, "libnvfp4_ggemm.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libnvfp4_ggemm_debug.so")

SOURCES = ["ggemm_kernels.cu", "sf_relayout.cu", "ggemm_host.cpp", "ggemm_noalloc.cu", "io_copy.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + COMMON + (["-DNVFP4_DEBUG"] if debug else [])
    if src.endswith(".cu"):
        cmd += ARCH
        if verbose:
            cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        sys.stderr.write(res.stdout + res.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile (if stale) and return the path of libnvfp4_ggemm.so, or of
    libnvfp4_ggemm_debug.so with debug."""
    lib, out_dir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(out_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--debug", action="store_true", help="the device-check build, libnvfp4_ggemm_debug.so")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug=a.debug))
