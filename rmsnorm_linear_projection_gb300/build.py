"""Compile the CUDA library ``librnl.so`` in-tree with nvcc for sm_103a.

    python -m rmsnorm_linear_projection_gb300.build [--force] [--verbose] [--debug]

Each ``csrc/*.cu`` translation unit is compiled in parallel to an object in
``_build/``; the objects are linked into ``librnl.so`` next to this file with
the CUDA runtime linked statically (the library then loads on machines
without a GPU driver, and only talks to the driver once it is called).

``--debug`` builds ``librnl_debug.so`` from objects in ``_build_debug/`` with
``RNL_DEBUG`` defined: the same kernels with device-side bounds checks that
report RNL_ERR_BOUNDS through rnl_check_device_error() instead of accessing
out of range (include/rnl.h, rnl_debug_build).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "librnl.so")
DEBUG_OBJ_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "librnl_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Build (incrementally) and return the path of librnl.so, or of
    librnl_debug.so with ``debug=True``."""
    obj_dir = DEBUG_OBJ_DIR if debug else OBJ_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    if debug:
        extra_flags = (*extra_flags, "-DRNL_DEBUG")
    os.makedirs(obj_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = _headers()
    nvcc = _nvcc()
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *hdrs]):
            jobs.append([nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed: " + os.path.basename(cmd[-3]))
        return r

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                debug="--debug" in sys.argv))
