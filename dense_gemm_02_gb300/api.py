"""Tensor-level entry points over the C ABI.

``sgemm`` and ``gemm_bf16`` take CUDA tensors (row-major, unit column
stride) and enqueue one library call on the current torch stream.
``gemm_ex`` adds transposed operands (a ``X.t()`` view is read in place)
and the fused bias / activation epilogue; ``gemm_batched`` runs a strided
batch of such products in one launch, ``gemm_grouped`` a list of problems of
different shapes.
``gemm`` additionally accepts host (CPU) tensors, which it hands to the
library's host-buffer entry points (copies pipelined with the computation):
the end-to-end path of a caller holding host buffers.  Nothing here
computes: shapes, strides and pointers are read from the tensors and handed
to the library.
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
    if t.numel() == 0:  # no element is read: any pitch that passes the checks
        return max(1, t.size(1))
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


_ACTS = {"none": _b.GEMM_ACT_NONE, "relu": _b.GEMM_ACT_RELU, "gelu": _b.GEMM_ACT_GELU_TANH,
         "gelu_tanh": _b.GEMM_ACT_GELU_TANH}


def _layout(t: torch.Tensor, name: str):
    """(trans, ld) of a 2-D operand as stored: row-major (unit column
    stride), or the transposed view of a row-major matrix (unit row
    stride), whose stored form has the two dimensions swapped."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    r, c = t.shape
    if c <= 1 or t.stride(1) == 1:
        return 0, (max(1, t.stride(0)) if r > 1 else max(1, c))
    if r <= 1 or t.stride(0) == 1:
        return 1, (max(1, t.stride(1)) if c > 1 else max(1, r))
    raise ValueError(f"{name} must be row-major or the transpose of a row-major matrix")


def gemm_ex(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
            alpha: float = 1.0, beta: float = 0.0, bias: torch.Tensor | None = None,
            act: str = "none", out_dtype=None, stream=None) -> torch.Tensor:
    """C = act(alpha * A @ B + bias) + beta * C on CUDA tensors.

    A (M x K) and B (K x N) may each be row-major or a transposed view of a
    row-major matrix (``W.t()``); the library reads the stored layout
    directly.  ``bias`` is None or a contiguous N-vector (float32 or
    bfloat16); ``act`` is "none", "relu" or "gelu" (tanh form).  float32
    A, B run the FP32 path (C float32); bfloat16 A, B the tensor cores (C
    bfloat16 or float32)."""
    if A.dtype != B.dtype or A.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("A and B must both be float32 or both bfloat16")
    if not (A.is_cuda and B.is_cuda):
        raise TypeError("A and B must be CUDA tensors")
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(_ACTS)}")
    M, N, K = _shapes(A, B, C)
    ta, lda = _layout(A, "A")
    tb, ldb = _layout(B, "B")
    bias_ptr, bias_type = None, _b.GEMM_OUT_F32
    if bias is not None:
        if bias.dim() != 1 or bias.numel() != N or not bias.is_cuda or not bias.is_contiguous():
            raise ValueError(f"bias must be a contiguous CUDA vector of {N} values")
        if bias.dtype == torch.float32:
            bias_type = _b.GEMM_OUT_F32
        elif bias.dtype == torch.bfloat16:
            bias_type = _b.GEMM_OUT_BF16
        else:
            raise TypeError("bias must be float32 or bfloat16")
        bias_ptr = bias.data_ptr()
    opts = _b.make_opts(ta, tb, bias_ptr, bias_type, _ACTS[act])
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        od = torch.float32 if A.dtype == torch.float32 else (out_dtype or torch.bfloat16)
        C = torch.empty((M, N), dtype=od, device=A.device)
    if not C.is_cuda:
        raise TypeError("C must be a CUDA tensor")
    if A.dtype == torch.float32:
        if C.dtype != torch.float32:
            raise TypeError("C must be float32 for float32 operands")
        rc = _b.gemm_f32_ex(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                            float(beta), C.data_ptr(), _row_major(C, "C"), opts,
                            _stream_handle(stream))
        _b.check(rc, "gemm_f32_ex")
        return C
    if C.dtype == torch.bfloat16:
        c_type = _b.GEMM_OUT_BF16
    elif C.dtype == torch.float32:
        c_type = _b.GEMM_OUT_F32
    else:
        raise TypeError("C must be bfloat16 or float32")
    rc = _b.gemm_bf16_ex(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                         float(beta), C.data_ptr(), _row_major(C, "C"), c_type, opts,
                         _stream_handle(stream))
    _b.check(rc, "gemm_bf16_ex")
    return C


def gemm_grouped(As, Bs, Cs=None, alphas=1.0, betas=0.0, out_dtype=None,
                 stream=None) -> list:
    """C_i = alpha_i * A_i @ B_i + beta_i * C_i for problems of different
    shapes, in one library call (one launch per 64 problems).

    As, Bs: sequences of CUDA tensors, all float32 (FP32 path) or all
    bfloat16 (tensor cores); each A_i may be row-major or a transposed view
    (``W.t()``), the same for every problem (likewise B_i).  Cs: None or a
    sequence of C tensors (created when None; beta must then be 0).  alphas,
    betas: a number or one per problem.  Returns the list of C tensors."""
    As, Bs = list(As), list(Bs)
    n = len(As)
    if len(Bs) != n:
        raise ValueError("As and Bs differ in length")
    if n == 0:
        return []
    dt = As[0].dtype
    if dt not in (torch.float32, torch.bfloat16) or any(t.dtype != dt for t in As + Bs):
        raise TypeError("all operands must be float32, or all bfloat16")
    if not all(t.is_cuda for t in As + Bs):
        raise TypeError("operands must be CUDA tensors")
    alphas = [float(alphas)] * n if isinstance(alphas, (int, float)) else [float(a) for a in alphas]
    betas = [float(betas)] * n if isinstance(betas, (int, float)) else [float(b) for b in betas]
    if len(alphas) != n or len(betas) != n:
        raise ValueError("alphas and betas need one value per problem")
    if dt == torch.float32:
        out_dtype = torch.float32
    elif out_dtype is None:
        out_dtype = torch.bfloat16 if Cs is None else Cs[0].dtype
    if Cs is None:
        if any(b != 0.0 for b in betas):
            raise ValueError("beta != 0 needs input Cs")
        Cs = [torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype, device=a.device)
              for a, b in zip(As, Bs)]
    Cs = list(Cs)
    if len(Cs) != n or any(c.dtype != out_dtype or not c.is_cuda for c in Cs):
        raise TypeError(f"Cs must be {n} CUDA tensors of {out_dtype}")
    layouts = [(_layout(a, "A"), _layout(b, "B")) for a, b in zip(As, Bs)]
    ta, tb = layouts[0][0][0], layouts[0][1][0]
    if any(la[0] != ta or lb[0] != tb for la, lb in layouts):
        raise ValueError("every A (and every B) must have the same layout")
    problems = []
    for (a, b, c, al, be, (la, lb)) in zip(As, Bs, Cs, alphas, betas, layouts):
        M, N, K = _shapes(a, b, c)
        problems.append((M, N, K, a.data_ptr(), la[1], b.data_ptr(), lb[1], c.data_ptr(),
                         _row_major(c, "C"), al, be))
    groups = _b.make_groups(problems)
    opts = _b.make_opts(trans_a=ta, trans_b=tb)
    if dt == torch.float32:
        rc = _b.gemm_f32_grouped(groups, n, opts, _stream_handle(stream))
        _b.check(rc, "gemm_f32_grouped")
    else:
        c_type = _b.GEMM_OUT_F32 if out_dtype == torch.float32 else _b.GEMM_OUT_BF16
        rc = _b.gemm_bf16_grouped(groups, n, c_type, opts, _stream_handle(stream))
        _b.check(rc, "gemm_bf16_grouped")
    return Cs


def gemm_batched(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
                 alpha: float = 1.0, beta: float = 0.0, bias: torch.Tensor | None = None,
                 act: str = "none", out_dtype=None, stream=None) -> torch.Tensor:
    """C[i] = act(alpha * A[i] @ B[i] + bias) + beta * C[i] for every i, in one
    launch (strided batched GEMM).

    A (batch x M x K) and B (batch x K x N) are CUDA tensors whose matrices
    are each row-major or a transposed view; a batch dimension of size 1 (or
    stride 0, as from ``expand``) shares that operand among all products.
    C is batch x M x N with row-major matrices.  Dtypes and ``bias`` /
    ``act`` as in ``gemm_ex``."""
    if A.dim() != 3 or B.dim() != 3:
        raise ValueError("A and B must be 3-D (batch x rows x cols)")
    if A.dtype != B.dtype or A.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("A and B must both be float32 or both bfloat16")
    if not (A.is_cuda and B.is_cuda):
        raise TypeError("A and B must be CUDA tensors")
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(_ACTS)}")
    batch = max(A.size(0), B.size(0))
    for name, t in (("A", A), ("B", B)):
        if t.size(0) not in (1, batch):
            raise ValueError(f"{name} has batch {t.size(0)}, expected 1 or {batch}")
    M, N, K = _shapes(A[0], B[0], None)
    ta, lda = _layout(A[0], "A")
    tb, ldb = _layout(B[0], "B")
    stride_a = A.stride(0) if A.size(0) > 1 else 0
    stride_b = B.stride(0) if B.size(0) > 1 else 0
    bias_ptr, bias_type = None, _b.GEMM_OUT_F32
    if bias is not None:
        if bias.dim() != 1 or bias.numel() != N or not bias.is_cuda or not bias.is_contiguous():
            raise ValueError(f"bias must be a contiguous CUDA vector of {N} values")
        if bias.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("bias must be float32 or bfloat16")
        bias_type = _b.GEMM_OUT_F32 if bias.dtype == torch.float32 else _b.GEMM_OUT_BF16
        bias_ptr = bias.data_ptr()
    opts = _b.make_opts(ta, tb, bias_ptr, bias_type, _ACTS[act])
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        od = torch.float32 if A.dtype == torch.float32 else (out_dtype or torch.bfloat16)
        C = torch.empty((batch, M, N), dtype=od, device=A.device)
    if C.dim() != 3 or tuple(C.shape) != (batch, M, N) or not C.is_cuda:
        raise ValueError(f"C must be a CUDA tensor of shape {(batch, M, N)}")
    ldc = _row_major(C[0], "C")
    stride_c = C.stride(0) if batch > 1 else max(1, M * ldc)
    h = _stream_handle(stream)
    if A.dtype == torch.float32:
        if C.dtype != torch.float32:
            raise TypeError("C must be float32 for float32 operands")
        rc = _b.gemm_f32_batched(batch, M, N, K, float(alpha), A.data_ptr(), lda, stride_a,
                                 B.data_ptr(), ldb, stride_b, float(beta), C.data_ptr(), ldc,
                                 stride_c, opts, h)
        _b.check(rc, "gemm_f32_batched")
        return C
    if C.dtype == torch.bfloat16:
        c_type = _b.GEMM_OUT_BF16
    elif C.dtype == torch.float32:
        c_type = _b.GEMM_OUT_F32
    else:
        raise TypeError("C must be bfloat16 or float32")
    rc = _b.gemm_bf16_batched(batch, M, N, K, float(alpha), A.data_ptr(), lda, stride_a,
                              B.data_ptr(), ldb, stride_b, float(beta), C.data_ptr(), ldc, stride_c,
                              c_type, opts, h)
    _b.check(rc, "gemm_bf16_batched")
    return C


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
    synchronising.  Host tensors go through the library's host-buffer entry
    points (gemm_f32_host / gemm_bf16_host) on ``device``: the library copies
    them in row blocks, computing each block as it lands and copying it back
    while the next computes, and the call returns once the result is in
    ``out`` (or C, or a new pinned tensor).  Pinned host tensors give the
    full copy bandwidth.
    """
    if A.is_cuda:
        return _dispatch(A, B, C, alpha, beta, out_dtype, stream)
    op, out, _keep = _host_op(A, B, C, alpha, beta, out_dtype, out)
    with torch.cuda.device(device):
        if op[0] == _b.GEMM_HOST_F32:
            rc = _b.gemm_f32_host(*op[2:5], op[5], op[7], op[8], op[9], op[10], op[6], op[11],
                                  op[12])
            _b.check(rc, "gemm_f32_host")
        else:
            rc = _b.gemm_bf16_host(*op[2:5], op[5], op[7], op[8], op[9], op[10], op[6], op[11],
                                   op[12], op[1])
            _b.check(rc, "gemm_bf16_host")
    return out


def _host_op(A, B, C, alpha, beta, out_dtype, out):
    """Checks one host-buffer product and returns (gemm_host_op_t fields,
    out, tensors to keep alive): out is the given one, C, or a new pinned
    tensor, already holding C when beta != 0."""
    if A.dtype != B.dtype or A.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("A and B must both be float32 or both bfloat16")
    if A.is_cuda or B.is_cuda or (C is not None and C.is_cuda) or (out is not None and out.is_cuda):
        raise TypeError("host-buffer call: A, B, C and out must all be host tensors")
    M, N, K = _shapes(A, B, C)
    if A.dtype == torch.float32:
        od = torch.float32
    else:
        od = out_dtype or (C.dtype if C is not None else torch.bfloat16)
    if od not in (torch.float32, torch.bfloat16):
        raise TypeError("the output must be float32 or bfloat16")
    if out is None:
        out = C if C is not None else torch.empty((M, N), dtype=od, pin_memory=True)
    if tuple(out.shape) != (M, N) or out.dtype != od:
        raise ValueError(f"out must be {(M, N)} of {od}")
    if C is not None and beta != 0.0 and out.data_ptr() != C.data_ptr():
        out.copy_(C)  # the library updates C in place
    A = A if (A.dim() == 2 and (A.size(1) <= 1 or A.stride(1) == 1)) else A.contiguous()
    B = B if (B.dim() == 2 and (B.size(1) <= 1 or B.stride(1) == 1)) else B.contiguous()
    f32 = A.dtype == torch.float32
    op = (_b.GEMM_HOST_F32 if f32 else _b.GEMM_HOST_BF16,
          _b.GEMM_OUT_F32 if od == torch.float32 else _b.GEMM_OUT_BF16,
          M, N, K, float(alpha), float(beta), A.data_ptr(), _row_major(A, "A"),
          B.data_ptr(), _row_major(B, "B"), out.data_ptr(), _row_major(out, "out"))
    return op, out, (A, B)


def gemm_many(problems, device="cuda") -> list:
    """Several host-buffer products C_i = alpha_i * A_i @ B_i + beta_i * C_i
    in one library call (gemm_host_batch): the copies of product i + 1 travel
    while product i computes, and the call returns once every result is in
    host memory.  ``problems`` is a sequence of dicts with the keys of
    :func:`gemm` (A, B and optionally C, alpha, beta, out_dtype, out), all
    host tensors.  No result may share memory with another product's
    operands or result.  Returns the outputs in order."""
    ops, outs, keep = [], [], []
    for pr in problems:
        op, out, k = _host_op(pr["A"], pr["B"], pr.get("C"), pr.get("alpha", 1.0),
                              pr.get("beta", 0.0), pr.get("out_dtype"), pr.get("out"))
        ops.append(op)
        outs.append(out)
        keep.append(k)
    arr = _b.make_host_ops(ops)
    with torch.cuda.device(device):
        _b.check(_b.gemm_host_batch(arr, len(ops)), "gemm_host_batch")
    return outs


def _dispatch(A, B, C, alpha, beta, out_dtype, stream):
    if A.dtype == torch.float32:
        return sgemm(A, B, C, alpha, beta, stream)
    if A.dtype == torch.bfloat16:
        od = out_dtype or (C.dtype if C is not None else torch.bfloat16)
        return gemm_bf16(A, B, C, alpha, beta, od, stream)
    raise TypeError(f"unsupported dtype {A.dtype}")
