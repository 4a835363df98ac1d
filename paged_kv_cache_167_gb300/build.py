"""Builds ``libpa.so`` (the C-ABI library) in-tree for sm_103a.

Every CUDA translation unit is compiled by nvcc with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``; the host units
with g++.  Units compile in parallel and are skipped when their object is
newer than every source and header; the objects are linked with nvcc into
``paged_kv_cache_167_gb300/libpa.so`` (static CUDA runtime).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIBRARY = os.path.join(PKG, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--use_fast_math",
                     "-Xptxas", "-warn-spills", "-I", INCLUDE, "-I", CSRC]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-I", CSRC]


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _nvcc() -> str:
    return shutil.which("nvcc") or os.path.join(_cuda_home(), "bin", "nvcc")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src, __file__] + _headers())


def _compile(src: str, verbose: bool, extra=()):
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    if not _stale(obj, src):
        return obj, None
    if src.endswith(".cu"):
        cmd = [_nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    else:
        cmd = ["g++"] + CXX_FLAGS + ["-I", os.path.join(_cuda_home(), "include"), "-c", src, "-o", obj]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    log = proc.stdout + proc.stderr
    if proc.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{log}")
    return obj, log if verbose else None


def build(verbose: bool = False, jobs: int | None = None, ptxas_verbose: bool = False) -> str:
    """Compiles and links libpa.so; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if ptxas_verbose:
        for src in sources:  # force recompilation so ptxas reports
            obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
            if os.path.exists(obj):
                os.remove(obj)
    jobs = jobs or min(len(sources), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose or ptxas_verbose, extra), sources))
    objs = [o for o, _ in results]
    for _, log in results:
        if log:
            sys.stderr.write(log)
    if not os.path.exists(LIBRARY) or any(os.path.getmtime(o) > os.path.getmtime(LIBRARY) for o in objs):
        tmp = LIBRARY + ".tmp"
        cmd = [_nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{proc.stdout}{proc.stderr}")
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(verbose=True, ptxas_verbose="-v" in sys.argv)
