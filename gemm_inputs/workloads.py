"""The benchmark workloads: shapes, operand distributions and alpha/beta.

Only descriptions and seeded draws live here (no GEMM arithmetic), so the
oracle side and the GPU side can take identical inputs.  The five workloads
are the FP32 SGEMM cases of "CUDA hand-written SGEMM: 0.4 -> 10.23 TFLOPS"
(gtnt.cn, 4096^3, section 1.1) plus a small 256^3 case, and BF16 cases in
the shapes the "Blackwell BF16 GEMM ..." page (lshu.cn) discusses: a square
4096^3 product, a transformer MLP projection (section 5.1) and a small-M
decode shape (section 5.2).
"""

from __future__ import annotations

from dataclasses import dataclass

from . import INTEGER_PASS_OFFSET, WORKLOAD_SEED_BASE, draw


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: str            # "f32" (SGEMM) or "bf16" (tensor-core GEMM)
    M: int
    N: int
    K: int
    dist: str             # "uniform" or "normal"
    sigma_a: float
    sigma_b: float
    alpha: float
    beta: float
    c_dist: str | None    # distribution of the input C (None: beta == 0)
    sigma_c: float
    out: str              # "f32" or "bf16"
    description: str

    @property
    def seed(self) -> int:
        return WORKLOAD_SEED_BASE + self.index

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def min_bytes(self) -> int:
        """A and B read once, C read if beta != 0, C written once."""
        ein = 4 if self.dtype == "f32" else 2
        eout = 4 if self.out == "f32" else 2
        c_reads = self.M * self.N * eout if self.beta != 0 else 0
        return ein * (self.M * self.K + self.K * self.N) + c_reads + self.M * self.N * eout

    def operands(self, integer: bool = False, rows: slice | None = None):
        """(A, B, C_in) as host arrays: float32 for fp32 operands, uint16
        bf16 bits for bf16 operands.  ``integer`` gives the {-2..2} pass.
        ``rows`` restricts A and C to a row range (same values as the full
        draw, since every element is a function of its index)."""
        seed = self.seed + (INTEGER_PASS_OFFSET if integer else 0)
        kind_a = "integer" if integer else self.dist
        A = _draw_rows(kind_a, seed, 0, self.M, self.K, self.sigma_a, self.dtype, rows)
        B = draw(kind_a, seed, 1, (self.K, self.N), sigma=self.sigma_b, dtype=self.dtype)
        C = None
        if self.beta != 0:
            kind_c = "integer" if integer else self.c_dist
            C = _draw_rows(kind_c, seed, 2, self.M, self.N, self.sigma_c, self.out, rows)
        return A, B, C

    def batch_operands(self, i: int, integer: bool = False):
        """(A, B, C_in) of matrix i of a strided batch of this shape: the
        elements after those of matrices 0..i-1 on the same streams (matrix
        0 is ``operands()``)."""
        seed = self.seed + (INTEGER_PASS_OFFSET if integer else 0)
        kind_a = "integer" if integer else self.dist
        A = draw(kind_a, seed, 0, (self.M, self.K), sigma=self.sigma_a, dtype=self.dtype,
                 offset=i * self.M * self.K)
        B = draw(kind_a, seed, 1, (self.K, self.N), sigma=self.sigma_b, dtype=self.dtype,
                 offset=i * self.K * self.N)
        C = None
        if self.beta != 0:
            kind_c = "integer" if integer else self.c_dist
            C = draw(kind_c, seed, 2, (self.M, self.N), sigma=self.sigma_c, dtype=self.out,
                     offset=i * self.M * self.N)
        return A, B, C


def _draw_rows(kind, seed, stream, rows_total, cols, sigma, dtype, rows):
    if rows is None:
        return draw(kind, seed, stream, (rows_total, cols), sigma=sigma, dtype=dtype)
    r0, r1 = rows.start or 0, min(rows.stop, rows_total)
    return draw(kind, seed, stream, (r1 - r0, cols), sigma=sigma, dtype=dtype, offset=r0 * cols)


WORKLOADS = {
    w.name: w for w in [
        Workload("sgemm_256", 0, "f32", 256, 256, 256, "uniform", 1.0, 1.0, 1.0, 0.0, None, 0.0,
                 "f32", "FP32 SGEMM 256^3, U[-1,1], alpha=1, beta=0"),
        Workload("sgemm_4096", 1, "f32", 4096, 4096, 4096, "uniform", 1.0, 1.0, 1.0, 0.0, None,
                 0.0, "f32", "FP32 SGEMM 4096^3, U[-1,1], alpha=1, beta=0"),
        Workload("bf16_4096", 2, "bf16", 4096, 4096, 4096, "normal", 1.0, 1.0, 1.0, 0.0, None,
                 0.0, "bf16", "BF16 GEMM 4096^3, N(0,1), fp32 accumulate, bf16 out"),
        Workload("bf16_mlp_8192x14336x4096", 3, "bf16", 8192, 14336, 4096, "normal", 0.02, 0.02,
                 0.5, 1.0, "normal", 1.0, "bf16",
                 "BF16 GEMM M=8192 N=14336 K=4096, A,B N(0,0.02^2), C N(0,1), alpha=0.5, "
                 "beta=1, bf16 out"),
        Workload("bf16_decode_64x8192x8192", 4, "bf16", 64, 8192, 8192, "normal", 1.0, 0.02, 1.0,
                 0.0, None, 0.0, "f32",
                 "BF16 GEMM M=64 N=8192 K=8192, A N(0,1), B N(0,0.02^2), fp32 out"),
    ]
}
