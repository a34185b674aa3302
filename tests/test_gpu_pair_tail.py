"""GPU parity of the CTA-pair kernel's partial last wave at sizes the oracle
finishes in seconds.  When the tile count leaves a partial wave, each of its
tiles is cut into two 128-column halves so that twice as many pairs share
it (a half wholly past the N edge is skipped); the halves run their K
blocks two at a time (one barrier wait and eight MMAs per pair of stages),
as every tile does ("stage_pairs" 0; 1: only the halves, 2: none).  The
"pair_limit" knob caps the pair count so that small problems reach this
path, as 4096^3 does on 76 pairs (256 tiles: 28 in the partial wave).

Integer-valued operands make every sum exact, so results must match the
oracle bit for bit with and without the split ("tail_split_off"); random
operands must meet the BF16 tolerance |C - C_ref| <= 2^-7 |C_ref| + 1e-2 and
repeat bit for bit.  The same cases run through the transposed layouts with
bias and ReLU, a strided batch, the allocation-free entry point and the
pipeline watchdog.
"""

import contextlib

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
import test_gpu_epilogue as te
from gpu_helpers import GuardedC, bf16_to_dev, bf16_tolerance_violations, widen

pytestmark = pytest.mark.gpu

B_ = g.binding


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.init()


@contextlib.contextmanager
def config(**kv):
    old = {k: g.get_config(k) for k in kv}
    for k, v in kv.items():
        g.set_config(k, v)
    try:
        yield
    finally:
        for k, v in old.items():
            g.set_config(k, v)


def tail_info(M, N, K, pairs, batch=1):
    """Host-side restatement of the partial-wave rule: (tiles in the partial
    wave, whether they are cut into column halves)."""
    tiles = -(-M // 256) * -(-N // 256) * batch
    rem = tiles % pairs
    return rem, rem > 0 and pairs // rem >= 2


# (pair_limit, M, N, K): ragged M, N and K; a CTA of the pair whose rows all
# lie past M; a tail half wholly past the N edge.
CASES = [(4, 768, 512, 1000), (7, 1280, 512, 520), (5, 700, 264, 1000), (6, 257, 1000, 4096)]


def test_cases_reach_the_split_partial_wave():
    assert all(tail_info(M, N, K, P)[1] for P, M, N, K in CASES)
    assert tail_info(4096, 4096, 4096, 76) == (28, True)


def run(A, B, Cin, alpha, beta, out):
    M, N = A.shape[0], B.shape[1]
    init = Cin if Cin is not None else (np.full((M, N), 0x7FC0, np.uint16) if out == "bf16"
                                        else np.full((M, N), np.nan, np.float32))
    C = GuardedC(M, N, N, out, init)
    g.gemm_bf16(bf16_to_dev(A), bf16_to_dev(B), C.view, alpha=alpha, beta=beta,
                out_dtype=torch.bfloat16 if out == "bf16" else torch.float32)
    torch.cuda.synchronize()
    B_.check(B_.get_device_status(), "device status")
    return C


def ref_round(R, out):
    return oracle.round_bf16(R) if out == "bf16" else oracle.round_f32(R)


# "stage_pairs": 0 every tile runs its K blocks two at a time, 1 only the
# column halves do, 2 none
@pytest.mark.parametrize("stage_pairs", [0, 1, 2])
@pytest.mark.parametrize("tail_off", [0, 1])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("P,M,N,K", CASES)
def test_partial_wave_integer_bit_exact(P, M, N, K, out, tail_off, stage_pairs):
    seed = 16000 + P + M + N + K + (out == "f32")
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype=out)
    with config(cta_pair=2, pair_limit=P, tail_split_off=tail_off, stage_pairs=stage_pairs):
        C = run(A, B, Cin, 0.5, -1.0, out)
    assert B_.last_kernel() == "bf16_tcgen05"
    got, ref = C.result(), ref_round(oracle.gemm(A, B, Cin, alpha=0.5, beta=-1.0), out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", te.TRANS)
def test_partial_wave_layouts_bias_relu_integer(ta, tb):
    P, M, N, K = CASES[1]
    out = "bf16" if ta == tb else "f32"
    seed = 16200 + 17 * ta + 31 * tb
    A, B, Cin, bias = te.integer_case(seed, M, N, K, out)
    with config(cta_pair=2, pair_limit=P):
        C = te.run_ex(A, B, Cin, 0.5, -1.0, bias, "relu", out, ta, tb)
    R = oracle.gemm_fused(A, B, Cin, alpha=0.5, beta=-1.0, bias=bias, act=oracle.ACT_RELU)
    got, ref = C.result(), ref_round(R, out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("stage_pairs", [0, 1])
def test_partial_wave_normal_tolerance_and_repeatable(out, stage_pairs):
    P, M, N, K = 7, 1280, 512, 2056
    assert tail_info(M, N, K, P)[1]
    A = gi.draw("normal", 16300, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 16300, 1, (K, N), dtype="bf16")
    with config(cta_pair=2, pair_limit=P, stage_pairs=stage_pairs):
        C1 = run(A, B, None, 1.0, 0.0, out)
        C2 = run(A, B, None, 1.0, 0.0, out)
    assert np.array_equal(C1.result(), C2.result())
    assert bf16_tolerance_violations(widen(C1.result(), out), oracle.gemm(A, B)) == 0


def test_partial_wave_batched_integer():
    P, n, M, N, K = 5, 3, 512, 512, 1024
    assert tail_info(M, N, K, P, batch=n)[1]
    seed = 16400
    As = [gi.draw("integer", seed + i, 0, (M, K), dtype="bf16") for i in range(n)]
    Bs = [gi.draw("integer", seed + i, 1, (K, N), dtype="bf16") for i in range(n)]
    dA = torch.stack([bf16_to_dev(a) for a in As])
    dB = torch.stack([bf16_to_dev(b) for b in Bs])
    C = torch.full((n, M, N), float("nan"), dtype=torch.float32, device="cuda")
    with config(cta_pair=2, pair_limit=P):
        g.gemm_batched(dA, dB, C)
        torch.cuda.synchronize()
    B_.check(B_.get_device_status(), "device status")
    got = C.cpu().numpy()
    for i in range(n):
        assert np.array_equal(got[i], oracle.round_f32(oracle.gemm(As[i], Bs[i]))), f"matrix {i}"


def test_partial_wave_through_the_allocation_free_entry():
    P, M, N, K = CASES[0]
    seed = 16500
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    dA, dB = bf16_to_dev(A), bf16_to_dev(B)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with config(cta_pair=2, pair_limit=P):
        rc = B_.gemm_bf16_noalloc(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                  C.data_ptr(), N, B_.GEMM_OUT_F32,
                                  torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    assert rc == B_.GEMM_OK
    assert np.array_equal(C.cpu().numpy(), oracle.round_f32(oracle.gemm(A, B)))


@pytest.mark.parametrize("stage_pairs", [0, 1])
def test_pair_kernel_watchdog_and_recovery(stage_pairs):
    P, M, N, K = CASES[0]
    seed = 16600
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    dA, dB = bf16_to_dev(A), bf16_to_dev(B)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    with config(cta_pair=2, pair_limit=P, watchdog_ms=200, stage_pairs=stage_pairs):
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
