"""Python handle on the CPU GEMM oracle (``gemm_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The library's compute
path never imports this package, and this package imports nothing from the
library.  Operands are numpy arrays; fp32 operands are float32 arrays and
bf16 operands are uint16 arrays holding the bf16 bits.

Each function is a thin ctypes call into the C oracle, which states the
definition it follows (C = alpha*A*B + beta*C, double accumulation) in its
header.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgemm_oracle.so")

F32, BF16, F64 = 0, 1, 2
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no GPU involved)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-O2",
           "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.oracle_gemm.argtypes = [i64, i64, i64, dbl, ci, vp, i64, ci, vp, i64,
                                    dbl, ci, vp, i64, vp, i64, ci]
        lib.oracle_gemm.restype = ci
        lib.oracle_gemm_entries.argtypes = [i64, i64, i64, dbl, ci, vp, i64, ci, vp, i64,
                                            dbl, ci, vp, i64, i64, vp, vp, vp]
        lib.oracle_gemm_entries.restype = ci
        lib.oracle_round_bf16.argtypes = [vp, vp, i64]
        lib.oracle_round_bf16.restype = None
        lib.oracle_round_f32.argtypes = [vp, vp, i64]
        lib.oracle_round_f32.restype = None
        lib.oracle_widen_bf16.argtypes = [vp, vp, i64]
        lib.oracle_widen_bf16.restype = None
        lib.oracle_epilogue.argtypes = [i64, i64, vp, i64, ci, vp, ci, dbl, ci, vp, i64]
        lib.oracle_epilogue.restype = ci
        _lib = lib
        return lib


def _operand(x, name):
    """(type code, pointer, leading dimension) of a 2-D row-major operand."""
    if x is None:
        return F32, None, 1, None
    if x.ndim != 2:
        raise ValueError(f"{name} must be 2-D")
    if x.dtype == np.float32:
        t = F32
    elif x.dtype == np.uint16:
        t = BF16
    elif x.dtype == np.float64:
        t = F64
    else:
        raise TypeError(f"{name}: unsupported dtype {x.dtype}")
    if x.size == 0:
        return t, x.ctypes.data, max(1, x.shape[1]), x
    if x.strides[1] != x.itemsize or x.strides[0] % x.itemsize:
        raise ValueError(f"{name} must be row-major with unit column stride")
    ld = max(1, x.strides[0] // x.itemsize)
    return t, x.ctypes.data, ld, x


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def gemm(A, B, C=None, alpha=1.0, beta=0.0, threads=None, M=None, N=None, K=None):
    """alpha*A@B + beta*C in double, as an (M, N) float64 array.

    Shapes come from A (M x K) and B (K x N) unless given, which lets a test
    pass K=0 with empty operands.
    """
    lib = _load()
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[1] if N is None else N
    ta, pa, lda, _ka = _operand(A, "A") if A is not None else (F32, None, 1, None)
    tb, pb, ldb, _kb = _operand(B, "B") if B is not None else (F32, None, 1, None)
    tc, pc, ldc, _kc = _operand(C, "C")
    R = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_gemm(M, N, K, float(alpha), ta, pa, lda, tb, pb, ldb,
                         float(beta), tc, pc, ldc, R.ctypes.data, max(1, N),
                         int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return R


def gemm_entries(A, B, rows, cols, C=None, alpha=1.0, beta=0.0):
    """The (rows[e], cols[e]) entries of alpha*A@B + beta*C, in double."""
    lib = _load()
    M, K = A.shape
    N = B.shape[1]
    ta, pa, lda, _ka = _operand(A, "A")
    tb, pb, ldb, _kb = _operand(B, "B")
    tc, pc, ldc, _kc = _operand(C, "C")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    out = np.empty(r.shape, dtype=np.float64)
    rc = lib.oracle_gemm_entries(M, N, K, float(alpha), ta, pa, lda, tb, pb, ldb,
                                 float(beta), tc, pc, ldc, r.size, r.ctypes.data,
                                 c.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return out


ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2


def _vector(x, name):
    if x is None:
        return F32, None, None
    x = np.ascontiguousarray(x)
    t = {np.dtype(np.float32): F32, np.dtype(np.uint16): BF16, np.dtype(np.float64): F64}.get(x.dtype)
    if t is None:
        raise TypeError(f"{name}: unsupported dtype {x.dtype}")
    return t, x.ctypes.data, x


def gemm_fused(A, B, C=None, alpha=1.0, beta=0.0, bias=None, act=ACT_NONE, threads=None,
               M=None, N=None, K=None):
    """act(alpha * A @ B + bias) + beta * C in double (A, B logical, row-major).
    Without bias and activation this is the plain gemm (alpha == 0 then gives
    beta * C itself, as there)."""
    if bias is None and int(act) == ACT_NONE:
        return gemm(A, B, C, alpha=alpha, beta=beta, threads=threads, M=M, N=N, K=K)
    lib = _load()
    R = gemm(A, B, None, alpha=alpha, beta=0.0, threads=threads, M=M, N=N, K=K)
    tb, pb, _kb = _vector(bias, "bias")
    if bias is not None and _kb.size != R.shape[1]:
        raise ValueError("bias must hold N values")
    tc, pc, ldc, _kc = _operand(C, "C")
    rc = lib.oracle_epilogue(R.shape[0], R.shape[1], R.ctypes.data, max(1, R.shape[1]), tb, pb,
                             int(act), float(beta), tc, pc, ldc)
    if rc != 0:
        raise ValueError("oracle_epilogue rejected its arguments")
    return R


def act_values(x, act) -> np.ndarray:
    """The oracle's activation applied to double values (via its epilogue)."""
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(1, -1).copy()
    lib = _load()
    rc = lib.oracle_epilogue(1, x.shape[1], x.ctypes.data, x.shape[1], F32, None, int(act), 0.0,
                             F32, None, 1)
    if rc != 0:
        raise ValueError("oracle_epilogue rejected its arguments")
    return x.reshape(-1)


def round_bf16(x) -> np.ndarray:
    """Double -> bf16 bits (uint16), round to nearest even."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_round_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def round_f32(x) -> np.ndarray:
    """Double -> fp32, round to nearest even."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float32)
    lib.oracle_round_f32(x.ctypes.data, out.ctypes.data, x.size)
    return out


def widen_bf16(b) -> np.ndarray:
    """bf16 bits (uint16) -> double, exactly."""
    lib = _load()
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_widen_bf16(b.ctypes.data, out.ctypes.data, b.size)
    return out

