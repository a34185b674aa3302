"""Builds libgemm_gb300.so in-tree with nvcc for sm_103a.

Each .cu file is compiled on its own thread (they are independent
translation units) and the objects are linked into one shared library under
``dense_gemm_02_gb300/_lib``.  A rebuild happens only when a source or header
is newer than the library, and then recompiles only the objects older than
their source or than any header.

``build(debug=True)`` makes the debug variant, libgemm_gb300_debug.so, from
the same sources with GEMM_DEBUG=1: its kernels check the indices, copy
coordinates and shared/tensor-memory ranges they compute and report a failed
check as GEMM_ERR_DEVICE_CHECK (the binding loads it when the environment
variable GEMM_GB300_DEBUG is 1).
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG_DIR, "_lib")
OBJ_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(LIB_DIR, "libgemm_gb300.so")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libgemm_gb300_debug.so")
DEBUG_OBJ_DIR = os.path.join(PKG_DIR, "_build_debug")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgemm_gb300")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + _headers()


def up_to_date(debug: bool = False) -> bool:
    lib = DEBUG_LIB_PATH if debug else LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _obj_path(src: str, debug: bool = False) -> str:
    return os.path.join(DEBUG_OBJ_DIR if debug else OBJ_DIR, os.path.basename(src) + ".o")


def _obj_current(src: str, newest_header: float, debug: bool = False) -> bool:
    obj = _obj_path(src, debug)
    return os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src),
                                                                newest_header)


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = _obj_path(src, debug)
    cmd = [nvcc(), *ARCH_FLAGS, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if debug:
        cmd[1:1] = ["-DGEMM_DEBUG=1"]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas and res.stderr:
        print(res.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile and link the library (debug: the checked variant); returns its
    path."""
    lib = DEBUG_LIB_PATH if debug else LIB_PATH
    obj_dir = DEBUG_OBJ_DIR if debug else OBJ_DIR
    if not force and not verbose_ptxas and up_to_date(debug):
        return lib
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = sources()
    # Objects newer than their source and every header are reused.
    newest_header = max(os.path.getmtime(h) for h in _headers())
    stale = [s for s in srcs
             if force or verbose_ptxas or not _obj_current(s, newest_header, debug)]
    if stale:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(stale), os.cpu_count() or 1))) as ex:
            list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), stale))
    objs = [_obj_path(s, debug) for s in srcs]
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys

    print(build(force=True, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
