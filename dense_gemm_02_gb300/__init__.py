"""Dense GEMM C = alpha * A * B + beta * C for one NVIDIA GB300 (sm_103a).

Two hand-written CUDA kernels behind a C ABI (include/gemm_gb300.h):
an FP32 SGEMM on the CUDA cores and a BF16 x BF16 -> FP32-accumulate GEMM on
the tcgen05 tensor cores, both with transposed-operand layouts and a fused
bias / activation epilogue.  This package is the thin Python binding.
"""

from . import binding
from .api import gemm, gemm_batched, gemm_bf16, gemm_ex, gemm_grouped, gemm_many, sgemm
from .binding import GemmError, get_config, set_config

__all__ = ["gemm", "gemm_batched", "gemm_bf16", "gemm_ex", "gemm_grouped", "gemm_many", "sgemm",
           "binding",
           "GemmError", "get_config", "set_config", "flops"]


def flops(M: int, N: int, K: int) -> int:
    """Floating-point operations of one GEMM, counting a multiply-add as two:
    2*M*N*K (the count of "CUDA hand-written SGEMM ..." (gtnt.cn), 1.1)."""
    return 2 * M * N * K
