"""Tensor-level entry points over the C ABI.

``sgemm`` and ``gemm_bf16`` take CUDA tensors (row-major, unit column
stride) and enqueue one library call on the current torch stream.
``gemm`` additionally accepts host (CPU) tensors: it copies them to the
device, runs the same call and copies C back, which is the end-to-end path
a caller holding host buffers uses.  Nothing here computes: shapes, strides
and pointers are read from the tensors and handed to the library.
"""

from __future__ import annotations

import torch

from . import binding as _b


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _row_major(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    return max(1, t.stride(0)) if t.size(0) > 1 else max(1, t.size(1))


def _shapes(A, B, C):
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if C is not None and tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    return M, N, K


def sgemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
          alpha: float = 1.0, beta: float = 0.0, stream=None) -> torch.Tensor:
    """C = alpha * A @ B + beta * C with fp32 CUDA tensors (FP32 SGEMM)."""
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
    M, N, K = _shapes(A, B, C)
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif C.dtype != torch.float32 or not C.is_cuda:
        raise TypeError("C must be a float32 CUDA tensor")
    rc = _b.gemm_f32(M, N, K, float(alpha), A.data_ptr(), _row_major(A, "A"), B.data_ptr(),
                     _row_major(B, "B"), float(beta), C.data_ptr(), _row_major(C, "C"),
                     _stream_handle(stream))
    _b.check(rc, "gemm_f32")
    return C


def gemm_bf16(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
              alpha: float = 1.0, beta: float = 0.0, out_dtype=torch.bfloat16,
              stream=None) -> torch.Tensor:
    """C = alpha * A @ B + beta * C with bf16 CUDA A, B; fp32 accumulation;
    C in ``out_dtype`` (bfloat16 or float32)."""
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bfloat16 CUDA tensor")
    M, N, K = _shapes(A, B, C)
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if C.dtype == torch.bfloat16:
        c_type = _b.GEMM_OUT_BF16
    elif C.dtype == torch.float32:
        c_type = _b.GEMM_OUT_F32
    else:
        raise TypeError("C must be bfloat16 or float32")
    if not C.is_cuda:
        raise TypeError("C must be a CUDA tensor")
    rc = _b.gemm_bf16(M, N, K, float(alpha), A.data_ptr(), _row_major(A, "A"), B.data_ptr(),
                      _row_major(B, "B"), float(beta), C.data_ptr(), _row_major(C, "C"), c_type,
                      _stream_handle(stream))
    _b.check(rc, "gemm_bf16")
    return C


def gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
         alpha: float = 1.0, beta: float = 0.0, out_dtype=None,
         out: torch.Tensor | None = None, device="cuda", stream=None) -> torch.Tensor:
    """C = alpha * A @ B + beta * C, dispatching on A's dtype (float32 ->
    FP32 SGEMM, bfloat16 -> BF16 tensor-core GEMM).

    Device tensors are used in place and the call returns without
    synchronising.  Host tensors are copied to ``device`` (asynchronously
    when pinned; C only if beta != 0), the product is computed there, and
    the result is copied back into ``out`` (or C, or a new pinned tensor);
    the call returns after that copy has completed.
    """
    if A.is_cuda:
        return _dispatch(A, B, C, alpha, beta, out_dtype, stream)
    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        dA = A.to(device, non_blocking=True)
        dB = B.to(device, non_blocking=True)
        dC = C.to(device, non_blocking=True) if (C is not None and beta != 0.0) else None
        if dC is None and C is not None:
            od = C.dtype
        else:
            od = out_dtype
        dC = _dispatch(dA, dB, dC, alpha, beta, od, s)
        if out is None:
            out = C if C is not None else torch.empty(dC.shape, dtype=dC.dtype,
                                                      pin_memory=True)
        out.copy_(dC, non_blocking=True)
    s.synchronize()
    return out


def _dispatch(A, B, C, alpha, beta, out_dtype, stream):
    if A.dtype == torch.float32:
        return sgemm(A, B, C, alpha, beta, stream)
    if A.dtype == torch.bfloat16:
        od = out_dtype or (C.dtype if C is not None else torch.bfloat16)
        return gemm_bf16(A, B, C, alpha, beta, od, stream)
    raise TypeError(f"unsupported dtype {A.dtype}")
