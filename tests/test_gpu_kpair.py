"""GPU parity of the CTA-pair kernel's K-pair copies.  Where K is a multiple
of 64 (and, for an operand stored MN-major, its M or N too), one TMA copy per
operand fills two consecutive ring stages: the tensor map views the K blocks
as a dimension of their own and its box spans two of them.  A column-half
tail tile's 64 B columns of both K blocks land in the first stage's B slot,
where the MMA warp reads the second block.  A pair of stages
that would wrap around the end of the ring (an odd K-block count shifts
them) falls back to one copy per K block.  "kpair_maps_off" 1 turns the
path off.

A host-side restatement of the rule picks shapes that take the path.  With
integer-valued operands every sum is exact, so both settings must match the
oracle bit for bit: whole tiles and column halves, an odd K-block count,
rows past M read through the 3-D view, padded pitches and all four operand
layouts.  The MMAs read the same shared-memory bytes in the same order either
way, so on N(0,1) data both settings must also agree bit for bit, and meet
the BF16 tolerance |C - C_ref| <= 2^-7 |C_ref| + 1e-2.
"""

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
import test_gpu_epilogue as te
import test_gpu_pair_tail as tp
from gpu_helpers import bf16_tolerance_violations, widen

pytestmark = pytest.mark.gpu

B_ = g.binding


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.init()


def kpair_applies(M, N, K, ta=0, tb=0):
    """The rule the library applies before encoding the K-pair maps: K a
    multiple of 64; M too when A is stored K x M (ta); N too when B is
    stored K x N (not tb)."""
    return K % 64 == 0 and (not ta or M % 64 == 0) and (tb or N % 64 == 0)


# (pair_limit, M, N, K):
#   whole tiles and a split partial wave, 16 K blocks;
#   17 K blocks (pairs of stages wrap around the six-stage ring), the second
#     CTA of the last row block partly past M = 704, a tile column half past N;
#   one tile on three pairs: column halves only;
#   M = 700, not a multiple of 64 (row-major A still takes the path).
CASES = [(4, 768, 512, 1024), (6, 704, 640, 1088), (3, 256, 256, 4096), (4, 700, 512, 1024)]


def test_cases_take_the_kpair_path():
    assert all(kpair_applies(M, N, K) for _, M, N, K in CASES)
    assert all(tp.tail_info(M, N, K, P)[1] for P, M, N, K in CASES)
    assert (1088 // 64) % 2 == 1
    assert not kpair_applies(700, 512, 1024, ta=1)
    assert not kpair_applies(768, 500, 1024) and kpair_applies(768, 500, 1024, tb=1)
    assert kpair_applies(4096, 4096, 4096) and kpair_applies(8192, 14336, 4096)


@pytest.mark.parametrize("off", [0, 1])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("P,M,N,K", CASES)
def test_kpair_integer_bit_exact(P, M, N, K, out, off):
    seed = 17000 + P + M + N + K + (out == "f32")
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype=out)
    with tp.config(cta_pair=2, pair_limit=P, kpair_maps_off=off):
        C = tp.run(A, B, Cin, 0.5, -1.0, out)
    assert B_.last_kernel() == "bf16_tcgen05"
    got, ref = C.result(), tp.ref_round(oracle.gemm(A, B, Cin, alpha=0.5, beta=-1.0), out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", te.TRANS)
@pytest.mark.parametrize("case", [0, 1])
def test_kpair_layouts_bias_relu_integer(case, ta, tb):
    P, M, N, K = CASES[case]
    assert kpair_applies(M, N, K, ta, tb)
    out = "bf16" if ta == tb else "f32"
    seed = 17200 + 17 * ta + 31 * tb + case
    A, B, Cin, bias = te.integer_case(seed, M, N, K, out)
    with tp.config(cta_pair=2, pair_limit=P):
        C = te.run_ex(A, B, Cin, 0.5, -1.0, bias, "relu", out, ta, tb)
    R = oracle.gemm_fused(A, B, Cin, alpha=0.5, beta=-1.0, bias=bias, act=oracle.ACT_RELU)
    got, ref = C.result(), tp.ref_round(R, out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", te.TRANS)
def test_kpair_padded_pitches_integer(ta, tb):
    """Pitches well past the stored rows: the views' strides come from the
    pitch, not from the extents."""
    P, M, N, K = CASES[1]
    seed = 17300 + 17 * ta + 31 * tb
    A, B, Cin, _ = te.integer_case(seed, M, N, K, "f32")
    with tp.config(cta_pair=2, pair_limit=P):
        C = te.run_ex(A, B, Cin, 1.0, 1.0, None, "none", "f32", ta, tb, pads=(136, 72))
    ref = oracle.round_f32(oracle.gemm(A, B, Cin, alpha=1.0, beta=1.0))
    assert np.array_equal(C.result(), ref)
    assert C.guards_intact()


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_kpair_normal_same_bits_either_way(out):
    P, M, N, K = CASES[0]
    A = gi.draw("normal", 17400, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 17400, 1, (K, N), dtype="bf16")
    res = {}
    for off in (0, 1, 0):
        with tp.config(cta_pair=2, pair_limit=P, kpair_maps_off=off):
            C = tp.run(A, B, None, 1.0, 0.0, out)
        if off in res:
            assert np.array_equal(res[off], C.result())  # repeatable
        res[off] = C.result()
    assert np.array_equal(res[0], res[1])
    assert bf16_tolerance_violations(widen(res[0], out), oracle.gemm(A, B)) == 0


def test_kpair_watchdog_and_recovery():
    """The fault-injection hook withholds the first pair of stages, which the
    K-pair copies would have filled; the waits run out and the next call is
    correct."""
    P, M, N, K = CASES[0]
    seed = 17500
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    dA, dB = te.put(A, 0, 0, "bf16"), te.put(B, 0, 0, "bf16")
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    with tp.config(cta_pair=2, pair_limit=P, watchdog_ms=200):
        g.set_config("fault_inject", 1)
        try:
            g.gemm_bf16(dA, dB, C, out_dtype=torch.float32)
            rc = B_.get_device_status()
        finally:
            g.set_config("fault_inject", 0)
        assert rc == B_.GEMM_ERR_DEVICE_TIMEOUT
        g.gemm_bf16(dA, dB, C, out_dtype=torch.float32)
        assert B_.get_device_status() == B_.GEMM_OK
    assert np.array_equal(C.cpu().numpy(), oracle.round_f32(oracle.gemm(A, B)))
