"""Builds ``libkvevict.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` compiles to an object in parallel, then nvcc links the
shared library with the CUDA runtime linked statically.  Nothing here needs
a GPU: nvcc cross-compiles.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libkvevict.so")
# The bounds-checked variant (-DKV_DEBUG_BOUNDS): every TMA coordinate, workspace
# offset and gather index checked against its tensor's extent; a failed check posts
# KV_ERR_INVALID_ARG instead of touching memory.  Same sources, same ABI.
BUILD_DIR_DEBUG = os.path.join(PKG, "_build_debug")
LIB_PATH_DEBUG = os.path.join(PKG, "libkvevict_debug.so")
HEADER = os.path.join(ROOT, "include", "kvevict.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-ffp-contract=off", "-Xptxas", "-O3"]
_locks = {False: threading.Lock(), True: threading.Lock()}   # per variant


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvevict.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [HEADER]


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          debug: bool = False) -> str:
    """Compile and link; returns the library path.  Rebuilds only when sources changed.
    debug=True builds the bounds-checked variant libkvevict_debug.so."""
    lib_path = LIB_PATH_DEBUG if debug else LIB_PATH
    build_dir = BUILD_DIR_DEBUG if debug else BUILD_DIR
    with _locks[debug]:
        if not force and up_to_date(lib_path):
            return lib_path
        os.makedirs(build_dir, exist_ok=True)
        cc = nvcc()
        flags = NVCC_FLAGS + ARCH + ["-I", os.path.join(ROOT, "include")] + list(extra_flags or [])
        if debug:
            flags.append("-DKV_DEBUG_BOUNDS")

        def compile_one(src):
            obj = os.path.join(build_dir, os.path.basename(src) + ".o")
            cmd = [cc, "-c", src, "-o", obj] + flags
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, res.stdout, res.stderr))
            if verbose and (res.stdout or res.stderr):
                print(res.stdout + res.stderr)
            return obj

        with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
            objs = list(ex.map(compile_one, _sources()))
        tmp = lib_path + ".%d.tmp" % os.getpid()
        cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static", "-ldl"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n%s%s" % (res.stdout, res.stderr))
        os.replace(tmp, lib_path)
        return lib_path
