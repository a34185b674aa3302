"""The debug build (libgemm_gb300_debug.so, compiled with GEMM_DEBUG=1) on the
GPU.  Its kernels check the copy coordinates (a TMA x coordinate must be a
multiple of 16 bytes), the shared- and tensor-memory ranges and the split-K
workspace indices they compute; a failed check skips the access, records
its site and surfaces as GEMM_ERR_DEVICE_CHECK.  Without compute-sanitizer,
the debug library is how the tests look for out-of-range indices the guard
bands around C cannot see.

The parity tests of the kernels' edge paths run again in a child process
that loads the debug build (GEMM_GB300_DEBUG=1): the CTA-pair kernel's K-pair
copies and partial waves, the single-CTA kernel's split-K and stream-K, the
grouped and batched GEMMs, the allocation-free entry point and the FP32
kernels' tails.  Every check must hold on all of them: each of those tests
compares with the oracle and reads the device status after its call.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MODULES = ["test_gpu_kpair.py", "test_gpu_pair_tail.py", "test_gpu_grouped.py",
           "test_gpu_batched.py", "test_zz_no_alloc.py"]
# From the broad parity module: split-K, stream-K, partial waves (BF16 and
# FP32), both tcgen05 kernels on the same shapes, pitched operands and the
# tensor-map cache.
PARITY_SELECTION = ("split_k or stream_k or partial_wave or tail or single_and_pair or pitched "
                    "or tensor_map_reuse")


def _child(args, timeout):
    env = dict(os.environ, GEMM_GB300_DEBUG="1")
    return subprocess.run([sys.executable, *args], env=env, cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_child_loads_the_debug_build():
    from dense_gemm_02_gb300 import _build

    _build.build(debug=True)
    code = ("import dense_gemm_02_gb300 as g; b = g.binding; "
            "print(b.library_path(), b.debug_checks())")
    res = _child(["-c", code], 300)
    assert res.returncode == 0, res.stderr[-2000:]
    path, flag = res.stdout.split()
    assert path == _build.DEBUG_LIB_PATH and flag == "True"


def test_edge_path_parity_under_the_debug_build():
    from dense_gemm_02_gb300 import _build

    _build.build(debug=True)
    tests = [os.path.join("tests", m) for m in MODULES]
    res = _child(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *tests],
                 3000)
    tail = res.stdout[-3000:] + res.stderr[-2000:]
    assert res.returncode == 0, tail
    assert " passed" in res.stdout and " failed" not in res.stdout, tail
    res = _child(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                  "-k", PARITY_SELECTION, os.path.join("tests", "test_gpu_parity.py")], 3000)
    tail = res.stdout[-3000:] + res.stderr[-2000:]
    assert res.returncode == 0, tail
    assert " passed" in res.stdout, tail
