"""GPU parity of the host-buffer entry points (gemm_f32_host,
gemm_bf16_host, reached through dense_gemm_02_gb300.gemm with CPU tensors):
the library copies the operands in row blocks, computes each block and
copies it back.  Checked against the oracle on the same seeded inputs:
integer-valued operands bit-exact over several row blocks with a ragged
last block, pitched host arrays, beta != 0 with C in place or a separate
``out``, alpha == 0, K == 0; random inputs within the FP32 / BF16
tolerances.
"""

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
from gpu_helpers import bf16_tolerance_violations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.init()


def host(x, dtype, pad=0, pinned=True):
    """numpy operand -> CPU tensor (bf16 from uint16 bits), optionally as a
    view with `pad` spare columns per row."""
    rows, cols = x.shape
    buf = np.zeros((rows, cols + pad), dtype=x.dtype)
    buf[:, :cols] = x
    t = torch.from_numpy(buf)
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    if pinned:
        t = t.pin_memory()
    return t[:, :cols]


def result(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()


def ref_round(R, out):
    return oracle.round_bf16(R) if out == "bf16" else oracle.round_f32(R)


@pytest.mark.parametrize("M,N,K", [(2100, 264, 520), (600, 1000, 136), (1, 72, 64),
                                   (4096, 512, 256)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_host_integer_bit_exact(M, N, K, out):
    seed = 14000 + M + N + K
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype=out)
    hC = host(Cin, out)
    res = g.gemm(host(A, "bf16", pad=3), host(B, "bf16", pad=5), hC, alpha=0.5, beta=-1.0)
    assert res.data_ptr() == hC.data_ptr()  # C updated in place
    R = oracle.gemm(A, B, Cin, alpha=0.5, beta=-1.0)
    got, ref = result(res), ref_round(R, out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"


@pytest.mark.parametrize("M,N,K", [(2100, 260, 520), (1000, 1000, 1000), (5, 7, 9)])
def test_f32_host_integer_bit_exact_pageable(M, N, K):
    seed = 14100 + M + N + K
    A = gi.draw("integer", seed, 0, (M, K))
    B = gi.draw("integer", seed, 1, (K, N))
    Cin = gi.draw("integer", seed, 2, (M, N))
    out = torch.empty((M, N), dtype=torch.float32)  # pageable, separate from C
    res = g.gemm(host(A, "f32", pinned=False), host(B, "f32", pad=1, pinned=False),
                 host(Cin, "f32", pinned=False), alpha=2.0, beta=1.0, out=out)
    assert res.data_ptr() == out.data_ptr()
    assert np.array_equal(res.numpy(), oracle.round_f32(oracle.gemm(A, B, Cin, 2.0, 1.0)))


def test_host_random_within_tolerance():
    M, N, K = 3000, 1024, 1024
    A = gi.draw("normal", 14200, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 14200, 1, (K, N), dtype="bf16")
    res = g.gemm(host(A, "bf16"), host(B, "bf16"), out_dtype=torch.float32)
    assert bf16_tolerance_violations(result(res).astype(np.float64), oracle.gemm(A, B)) == 0
    Af = gi.draw("uniform", 14201, 0, (M, K))
    Bf = gi.draw("uniform", 14201, 1, (K, N))
    resf = g.gemm(host(Af, "f32"), host(Bf, "f32"))
    assert np.abs(resf.numpy().astype(np.float64) - oracle.gemm(Af, Bf)).max() <= 1e-5 * K


def test_host_alpha_zero_and_k_zero():
    M, N, K = 700, 48, 64
    Cin = gi.draw("integer", 14300, 2, (M, N))
    nanA = np.full((M, K), np.nan, np.float32)  # alpha == 0: never read
    res = g.gemm(host(nanA, "f32"), host(np.ones((K, N), np.float32), "f32"), host(Cin, "f32"),
                 alpha=0.0, beta=-2.0)
    assert np.array_equal(res.numpy(), oracle.round_f32(oracle.gemm(
        np.zeros((M, K), np.float32), np.zeros((K, N), np.float32), Cin, 0.0, -2.0)))
    res0 = g.gemm(host(np.zeros((M, 0), np.float32), "f32"),
                  host(np.zeros((0, N), np.float32), "f32"), host(Cin, "f32"), beta=3.0)
    assert np.array_equal(res0.numpy(), oracle.round_f32(3.0 * Cin.astype(np.float64)))


def test_host_entry_rejects_overlap_and_bad_type():
    from dense_gemm_02_gb300 import binding as b

    A = torch.zeros((64, 64), dtype=torch.float32)
    # C overlapping A in host memory
    rc = b.gemm_f32_host(64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 64, 0.0,
                         A.data_ptr(), 64)
    assert rc == b.GEMM_ERR_ALIAS
    Ab = torch.zeros((64, 64), dtype=torch.bfloat16)
    Cb = torch.zeros((64, 64), dtype=torch.float32)
    rc = b.gemm_bf16_host(64, 64, 64, 1.0, Ab.data_ptr(), 64, Ab.data_ptr(), 64, 0.0,
                          Cb.data_ptr(), 64, 7)
    assert rc == b.GEMM_ERR_INVALID_ARG


def test_host_batch_mixed_products_integer_bit_exact():
    """gemm_many / gemm_host_batch: an FP32 product with several row blocks,
    a BF16 product into bf16 with beta != 0 and pitched operands, and a BF16
    product into fp32, in one pipelined call; each bit for bit against the
    oracle and equal to its single call."""
    seed = 14400
    Af = gi.draw("integer", seed, 0, (2100, 520))
    Bf = gi.draw("integer", seed, 1, (520, 264))
    Ab = gi.draw("integer", seed + 1, 0, (600, 136), dtype="bf16")
    Bb = gi.draw("integer", seed + 1, 1, (136, 1000), dtype="bf16")
    Cb = gi.draw("integer", seed + 1, 2, (600, 1000), dtype="bf16")
    Ac = gi.draw("integer", seed + 2, 0, (33, 4096), dtype="bf16")
    Bc = gi.draw("integer", seed + 2, 1, (4096, 72), dtype="bf16")
    hCb = host(Cb, "bf16")
    outs = g.gemm_many([
        dict(A=host(Af, "f32"), B=host(Bf, "f32", pad=2), alpha=2.0),
        dict(A=host(Ab, "bf16", pad=3), B=host(Bb, "bf16", pad=5), C=hCb, alpha=0.5, beta=-1.0),
        dict(A=host(Ac, "bf16"), B=host(Bc, "bf16"), out_dtype=torch.float32),
    ])
    assert outs[1].data_ptr() == hCb.data_ptr()  # C updated in place
    refs = [oracle.round_f32(oracle.gemm(Af, Bf, alpha=2.0)),
            oracle.round_bf16(oracle.gemm(Ab, Bb, Cb, alpha=0.5, beta=-1.0)),
            oracle.round_f32(oracle.gemm(Ac, Bc))]
    for i, (o, r) in enumerate(zip(outs, refs)):
        got = result(o)
        assert np.array_equal(got, r), f"product {i}: {int((got != r).sum())} mismatches"
    single = g.gemm(host(Af, "f32"), host(Bf, "f32", pad=2), alpha=2.0)
    assert np.array_equal(result(single), result(outs[0]))


def test_host_batch_of_one_and_empty():
    seed = 14500
    A = gi.draw("uniform", seed, 0, (700, 300))
    B = gi.draw("uniform", seed, 1, (300, 500))
    (one,) = g.gemm_many([dict(A=host(A, "f32"), B=host(B, "f32"))])
    ref = g.gemm(host(A, "f32"), host(B, "f32"))
    assert np.array_equal(one.numpy(), ref.numpy())  # same kernels, same order
    assert g.gemm_many([]) == []


def test_host_batch_rejects_a_result_feeding_another_product():
    """Products of one batch run overlapped, so one product's result may not
    be another's operand: the library refuses before copying anything."""
    A = host(np.ones((64, 64), np.float32), "f32")
    B = host(np.ones((64, 64), np.float32), "f32")
    C1 = torch.zeros((64, 64), dtype=torch.float32).pin_memory()
    with pytest.raises(g.GemmError) as e:
        g.gemm_many([dict(A=A, B=B, out=C1), dict(A=C1, B=B)])
    assert e.value.status == g.binding.GEMM_ERR_ALIAS
    assert float(C1.abs().max()) == 0.0  # untouched
