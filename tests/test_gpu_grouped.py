"""GPU parity of the grouped GEMMs (gemm_bf16_grouped / gemm_f32_grouped):
problems of different shapes and operands in one call, through the C ABI,
against the oracle problem by problem.

* integer operands ({-2..2}, alpha = 0.5, beta = 1 with an integer C): every
  output of every problem bit for bit, with guard bands around each C;
* normal / uniform operands: the BF16 / FP32 tolerances per problem;
* ragged shapes, all four BF16 operand layouts, problems that share a
  read-only operand, more problems than one launch carries, empty and
  degenerate problems and misaligned ones (run as single calls) mixed in;
* a withheld pipeline stage is reported and the next call is correct.
"""

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
from dense_gemm_02_gb300 import binding as b
from gpu_helpers import GuardedC, bf16_to_dev, bf16_tolerance_violations, f32_to_dev, widen

pytestmark = pytest.mark.gpu

# (M, N, K): tails in every dimension; N and K multiples of 8 so that the
# tcgen05 grouped kernel takes them.
SHAPES_BF16 = [(1, 8, 8), (7, 72, 64), (65, 264, 1000), (129, 1000, 72), (300, 520, 776),
               (128, 256, 64), (257, 1288, 2056), (1000, 1000, 1000)]
# N and K multiples of 4 for the TMA SGEMM.
SHAPES_F32 = [(1, 4, 4), (7, 68, 36), (65, 260, 1000), (129, 1000, 68), (300, 516, 772),
              (128, 128, 32), (257, 1284, 2052)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()


def _stream():
    return torch.cuda.current_stream().cuda_stream


class Problem:
    """Host operands, device copies in the stored layout, a guarded C."""

    def __init__(self, M, N, K, seed, kind, dtype, out, ta=False, tb=False, alpha=0.5, beta=1.0,
                 B_shared=None):
        self.M, self.N, self.K, self.alpha, self.beta, self.out = M, N, K, alpha, beta, out
        self.A = gi.draw(kind, seed, 0, (M, K), dtype=dtype)
        self.B = B_shared[0] if B_shared is not None else gi.draw(kind, seed, 1, (K, N), dtype=dtype)
        self.Cin = gi.draw(kind, seed, 2, (M, N), dtype=out) if beta != 0 else None
        to_dev = bf16_to_dev if dtype == "bf16" else f32_to_dev
        # stored layouts: a transposed operand is kept as its transpose, row-major
        self.dA = to_dev(np.ascontiguousarray(self.A.T)) if ta else to_dev(self.A)
        if B_shared is not None:
            self.dB = B_shared[1]
        else:
            self.dB = to_dev(np.ascontiguousarray(self.B.T)) if tb else to_dev(self.B)
        init = self.Cin
        if init is None:
            init = (np.full((M, N), 0x7FC0, np.uint16) if out == "bf16"
                    else np.full((M, N), np.nan, np.float32))
        self.C = GuardedC(M, N, N + 3, out, init)

    def entry(self):
        return (self.M, self.N, self.K, self.dA.data_ptr(), self.dA.stride(0), self.dB.data_ptr(),
                self.dB.stride(0), self.C.view.data_ptr(), self.C.ldc, self.alpha, self.beta)

    def reference(self):
        return oracle.gemm(self.A, self.B, self.Cin, alpha=self.alpha, beta=self.beta)


def _run(problems, bf16, out="f32", ta=False, tb=False):
    groups = b.make_groups([p.entry() for p in problems])
    opts = b.make_opts(trans_a=ta, trans_b=tb)
    if bf16:
        c_type = b.GEMM_OUT_F32 if out == "f32" else b.GEMM_OUT_BF16
        rc = b.gemm_bf16_grouped(groups, len(problems), c_type, opts, _stream())
    else:
        rc = b.gemm_f32_grouped(groups, len(problems), opts, _stream())
    b.check(rc, "grouped")
    torch.cuda.synchronize()
    b.check(b.get_device_status(), "device status")


def _check_exact(problems):
    for i, p in enumerate(problems):
        R = p.reference()
        want = oracle.round_bf16(R) if p.out == "bf16" else oracle.round_f32(R)
        got = p.C.result()
        assert np.array_equal(got, want), f"problem {i} {p.M}x{p.N}x{p.K}: {(got != want).sum()}"
        assert p.C.guards_intact(), f"problem {i}"


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_grouped_integer_bit_exact(out):
    probs = [Problem(M, N, K, 0x6A00 + i, "integer", "bf16", out) for i, (M, N, K) in
             enumerate(SHAPES_BF16)]
    _run(probs, True, out)
    assert b.last_kernel() == "bf16_tcgen05_grouped"
    _check_exact(probs)


@pytest.mark.parametrize("ta,tb", [(True, False), (False, True), (True, True)])
def test_bf16_grouped_layouts_integer(ta, tb):
    probs = [Problem(M, N, K, 0x6B00 + i, "integer", "bf16", "f32", ta=ta, tb=tb)
             for i, (M, N, K) in enumerate([(72, 264, 136), (264, 520, 64), (8, 1000, 1000)])]
    _run(probs, True, "f32", ta, tb)
    assert b.last_kernel() == "bf16_tcgen05_grouped"
    _check_exact(probs)


def test_bf16_grouped_normal_within_tolerance():
    probs = [Problem(M, N, K, 0x6C00 + i, "normal", "bf16", "bf16", alpha=1.0, beta=0.0)
             for i, (M, N, K) in enumerate(SHAPES_BF16)]
    _run(probs, True, "bf16")
    for i, p in enumerate(probs):
        assert bf16_tolerance_violations(widen(p.C.result(), "bf16"), p.reference()) == 0, i
        assert p.C.guards_intact()


def test_f32_grouped_integer_bit_exact_and_uniform_tolerance():
    probs = [Problem(M, N, K, 0x6D00 + i, "integer", "f32", "f32") for i, (M, N, K) in
             enumerate(SHAPES_F32)]
    _run(probs, False)
    assert b.last_kernel() == "sgemm_tma_grouped"
    _check_exact(probs)
    probs = [Problem(M, N, K, 0x6E00 + i, "uniform", "f32", "f32", alpha=1.0, beta=0.0)
             for i, (M, N, K) in enumerate(SHAPES_F32)]
    _run(probs, False)
    for i, p in enumerate(probs):
        assert np.abs(p.C.result().astype(np.float64) - p.reference()).max() <= 1e-5 * p.K, i
        assert p.C.guards_intact()


@pytest.mark.parametrize("bf16", [True, False])
def test_grouped_shared_operand_and_many_problems(bf16):
    # 130 problems (three launches of at most 64) sharing one B, as the
    # experts of a layer share nothing but here all read the same weights
    dtype = "bf16" if bf16 else "f32"
    K, N = 264, 136
    Bh = gi.draw("integer", 0x6F00, 1, (K, N), dtype=dtype)
    dB = bf16_to_dev(Bh) if bf16 else f32_to_dev(Bh)
    probs = [Problem(1 + (7 * i) % 150, N, K, 0x6F01 + i, "integer", dtype, "f32",
                     B_shared=(Bh, dB)) for i in range(130)]
    _run(probs, bf16)
    assert b.last_kernel() == ("bf16_tcgen05_grouped" if bf16 else "sgemm_tma_grouped")
    _check_exact(probs)


@pytest.mark.parametrize("bf16", [True, False])
def test_grouped_degenerate_and_misaligned_problems(bf16):
    dtype = "bf16" if bf16 else "f32"
    probs = [Problem(65, 264 if bf16 else 260, 136, 0x7000, "integer", dtype, "f32"),
             Problem(33, 72, 64, 0x7001, "integer", dtype, "f32", alpha=0.0, beta=-2.0),  # beta*C
             Problem(17, 63, 65, 0x7002, "integer", dtype, "f32"),  # pitches TMA cannot fetch
             Problem(40, 72, 136, 0x7003, "integer", dtype, "f32")]
    empty = Problem(1, 8, 8, 0x7004, "integer", dtype, "f32")
    empty.M = 0
    _run(probs + [empty], bf16)
    assert b.last_kernel() == ("bf16_grouped_mixed" if bf16 else "f32_grouped_mixed")
    _check_exact(probs)
    # K = 0: C = beta * C
    kz = Problem(9, 16, 8, 0x7005, "integer", dtype, "f32", beta=3.0)
    kz.K = 0
    _run([kz], bf16)
    assert np.array_equal(kz.C.result(), oracle.round_f32(3.0 * kz.Cin.astype(np.float64)))


@pytest.mark.parametrize("bf16", [True, False])
def test_grouped_watchdog_reports_a_withheld_stage_and_recovers(bf16):
    dtype = "bf16" if bf16 else "f32"
    probs = [Problem(M, N, K, 0x7100 + i, "integer", dtype, "f32", alpha=1.0, beta=0.0)
             for i, (M, N, K) in enumerate([(256, 512, 1024), (129, 264, 512)])]
    old = g.get_config("watchdog_ms")
    g.set_config("watchdog_ms", 200)
    g.set_config("fault_inject", 1)
    try:
        groups = b.make_groups([p.entry() for p in probs])
        rc = (b.gemm_bf16_grouped(groups, 2, b.GEMM_OUT_F32, None, _stream()) if bf16
              else b.gemm_f32_grouped(groups, 2, None, _stream()))
        assert rc == b.GEMM_OK
        status = b.get_device_status()
    finally:
        g.set_config("fault_inject", 0)
        g.set_config("watchdog_ms", old)
    assert status == b.GEMM_ERR_DEVICE_TIMEOUT
    _run(probs, bf16)
    _check_exact(probs)
