"""ctypes binding to libgemm_gb300.so (C ABI in include/gemm_gb300.h).

Argument marshalling only: every arithmetic step runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  If the compiled
library is missing the import of the entry points raises; there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_NULLPTR = -2
GEMM_ERR_BAD_LD = -3
GEMM_ERR_UNSUPPORTED_DEVICE = -4
GEMM_ERR_CUDA = -5
GEMM_ERR_DEVICE_TIMEOUT = -6
GEMM_ERR_ALIAS = -7
GEMM_ERR_TOO_LARGE = -8
GEMM_ERR_SCRATCH_LIMIT = -9
GEMM_ERR_DEVICE_CHECK = -10

GEMM_OUT_BF16 = 0
GEMM_OUT_F32 = 1

GEMM_ACT_NONE = 0
GEMM_ACT_RELU = 1
GEMM_ACT_GELU_TANH = 2

GEMM_HOST_F32 = 0
GEMM_HOST_BF16 = 1
GEMM_HOST_BATCH_MAX = 64


class GemmOpts(ctypes.Structure):
    """gemm_opts_t: operand layouts and fused epilogue of the *_ex calls."""

    _fields_ = [("trans_a", ctypes.c_int), ("trans_b", ctypes.c_int),
                ("bias", ctypes.c_void_p), ("bias_type", ctypes.c_int),
                ("act", ctypes.c_int)]

class GemmGroup(ctypes.Structure):
    """gemm_group_t: one problem of a grouped GEMM (device addresses)."""

    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float)]

# Every exported symbol of the C ABI, with (restype, argtypes).
class GemmHostOp(ctypes.Structure):
    """gemm_host_op_t: one product of gemm_host_batch (host addresses)."""

    _fields_ = [("dtype", ctypes.c_int), ("c_type", ctypes.c_int), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("alpha", ctypes.c_float),
                ("beta", ctypes.c_float), ("A", ctypes.c_void_p), ("lda", ctypes.c_int64),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("C", ctypes.c_void_p),
                ("ldc", ctypes.c_int64)]


_i64, _f32, _vp, _int, _cp = (ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                              ctypes.c_char_p)
SIGNATURES = {
    "gemm_f32": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "gemm_bf16": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _int,
                         _vp]),
    "gemm_bf16_noalloc": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                                 _int, _vp]),
    "gemm_bf16_ex": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _int,
                            ctypes.POINTER(GemmOpts), _vp]),
    "gemm_f32_ex": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                           ctypes.POINTER(GemmOpts), _vp]),
    "gemm_bf16_batched": (_int, [_i64, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp, _i64, _i64,
                                 _f32, _vp, _i64, _i64, _int, ctypes.POINTER(GemmOpts), _vp]),
    "gemm_f32_batched": (_int, [_i64, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp, _i64, _i64,
                                _f32, _vp, _i64, _i64, ctypes.POINTER(GemmOpts), _vp]),
    "gemm_bf16_grouped": (_int, [_i64, ctypes.POINTER(GemmGroup), _int, ctypes.POINTER(GemmOpts),
                                 _vp]),
    "gemm_f32_grouped": (_int, [_i64, ctypes.POINTER(GemmGroup), ctypes.POINTER(GemmOpts), _vp]),
    "gemm_f32_host": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64]),
    "gemm_host_batch": (_int, [_i64, ctypes.POINTER(GemmHostOp)]),
    "gemm_bf16_host": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                              _int]),
    "gemm_noalloc_get_status": (_int, [_vp, ctypes.POINTER(_i64)]),
    "gemm_get_device_status": (_int, [_vp]),
    "gemm_get_device_fault_info": (_i64, []),
    "gemm_debug_checks": (_int, []),
    "gemm_status_string": (_cp, [_int]),
    "gemm_set_config": (_int, [_cp, _i64]),
    "gemm_get_config": (_int, [_cp, ctypes.POINTER(_i64)]),
    "gemm_last_kernel": (_cp, []),
    "gemm_shutdown": (_int, []),
    "gemm_abi_version": (_int, []),
}

_lib = None
_lock = threading.Lock()


class GemmError(RuntimeError):
    """A non-zero gemm_status_t returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def debug_build_requested() -> bool:
    """Whether this process loads the checked variant of the library
    (environment variable GEMM_GB300_DEBUG=1)."""
    return os.environ.get("GEMM_GB300_DEBUG", "0") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if debug_build_requested() else _build.LIB_PATH


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            what = "the debug build " if debug_build_requested() else ""
            raise RuntimeError(
                f"{what}{os.path.basename(path)} is not built ({path}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != GEMM_OK:
        raise GemmError(status, where)


# ------------------------------------------------------------ raw entry points

def gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream) -> int:
    """Raw call; pointers and stream are integers (device addresses)."""
    return lib().gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, stream) -> int:
    """Raw call; A/B/C are device addresses, c_type GEMM_OUT_BF16/F32."""
    return lib().gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, stream)


def gemm_bf16_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, stream) -> int:
    """Raw call of the allocation-free variant (split-K scratch in a static
    device array); same arguments as gemm_bf16."""
    return lib().gemm_bf16_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, stream)


def make_opts(trans_a=False, trans_b=False, bias=None, bias_type=GEMM_OUT_F32,
              act=GEMM_ACT_NONE) -> GemmOpts:
    """A gemm_opts_t; bias is a device address (int) or None."""
    return GemmOpts(int(bool(trans_a)), int(bool(trans_b)), bias, int(bias_type), int(act))


def gemm_bf16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, opts, stream) -> int:
    """Raw call of the extended BF16 GEMM; opts is a GemmOpts or None."""
    ptr = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_bf16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, ptr, stream)


def gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, opts, stream) -> int:
    """Raw call of the extended FP32 GEMM; opts is a GemmOpts or None."""
    ptr = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ptr, stream)


def gemm_bf16_batched(batch, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc,
                      stride_c, c_type, opts, stream) -> int:
    """Raw call of the strided batched BF16 GEMM; opts is a GemmOpts or None."""
    ptr = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_bf16_batched(batch, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b,
                                   beta, C, ldc, stride_c, c_type, ptr, stream)


def gemm_f32_batched(batch, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc,
                     stride_c, opts, stream) -> int:
    """Raw call of the strided batched FP32 GEMM; opts is a GemmOpts or None."""
    ptr = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_f32_batched(batch, M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b,
                                  beta, C, ldc, stride_c, ptr, stream)


def make_groups(problems) -> ctypes.Array:
    """A gemm_group_t array from (M, N, K, A, lda, B, ldb, C, ldc, alpha,
    beta) tuples (A, B, C device addresses)."""
    arr = (GemmGroup * max(1, len(problems)))()
    for i, pr in enumerate(problems):
        arr[i] = GemmGroup(*pr)
    return arr


def gemm_bf16_grouped(groups, count, c_type, opts, stream) -> int:
    """Raw call of the grouped BF16 GEMM; groups from make_groups."""
    ptr = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_bf16_grouped(count, groups, c_type, ptr, stream)


def gemm_f32_grouped(groups, count, opts, stream) -> int:
    """Raw call of the grouped FP32 GEMM; groups from make_groups."""
    ptr = ctypes.byref(opts) if opts is not None else None
    return lib().gemm_f32_grouped(count, groups, ptr, stream)


def gemm_f32_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc) -> int:
    """Raw call of the host-buffer FP32 GEMM; A, B, C are host addresses."""
    return lib().gemm_f32_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)


def gemm_bf16_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type) -> int:
    """Raw call of the host-buffer BF16 GEMM; A, B, C are host addresses."""
    return lib().gemm_bf16_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type)


def make_host_ops(problems) -> ctypes.Array:
    """A gemm_host_op_t array from (dtype, c_type, M, N, K, alpha, beta, A,
    lda, B, ldb, C, ldc) tuples (A, B, C host addresses)."""
    arr = (GemmHostOp * max(1, len(problems)))()
    for i, pr in enumerate(problems):
        arr[i] = GemmHostOp(*pr)
    return arr


def gemm_host_batch(ops, count) -> int:
    """Raw call of the batched host-buffer GEMM; ops from make_host_ops."""
    return lib().gemm_host_batch(count, ops)


def noalloc_get_status(stream=None) -> tuple[int, int]:
    """(status, fault info) of the allocation-free calls on the current
    device; reading clears a recorded fault."""
    info = ctypes.c_int64(0)
    rc = lib().gemm_noalloc_get_status(stream, ctypes.byref(info))
    return int(rc), int(info.value)


def get_device_status(stream=None) -> int:
    return lib().gemm_get_device_status(stream)


def get_device_fault_info() -> int:
    return int(lib().gemm_get_device_fault_info())


def debug_checks() -> bool:
    """Whether the loaded library is the debug build."""
    return bool(lib().gemm_debug_checks())


def set_config(key: str, value: int) -> None:
    check(lib().gemm_set_config(key.encode(), int(value)), f"gemm_set_config({key})")


def get_config(key: str) -> int:
    v = ctypes.c_int64(0)
    check(lib().gemm_get_config(key.encode(), ctypes.byref(v)), f"gemm_get_config({key})")
    return int(v.value)


def last_kernel() -> str:
    return lib().gemm_last_kernel().decode()


def shutdown() -> None:
    check(lib().gemm_shutdown(), "gemm_shutdown")


def abi_version() -> int:
    return int(lib().gemm_abi_version())
