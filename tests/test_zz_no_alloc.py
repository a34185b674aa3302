"""The allocation-free entry point, gemm_bf16_noalloc, and its status query.

Some callers cannot call cudaMalloc at all: code running inside a host
application whose device memory is entirely owned by that application's own
arena or caching allocator (a plugin, a framework extension), or
latency-critical code that cannot take the implicit synchronisation an
allocation may cause.  For them the library offers a BF16 GEMM whose split-K
scratch is a static device array compiled into the library, and
gemm_noalloc_get_status, which reports a pipeline wait that ran out of time
without allocating either.

Checked through the C ABI:
  * on two calls in a row, bit for bit against gemm_bf16 (the same kernel
    with the same split choice), at shapes that split K;
  * bit for bit against the oracle on integer operands (with the BF16
    tolerance |C - C_ref| <= 2^-7 |C_ref| + 1e-2 on random operands);
  * the device's free memory is unchanged across the calls (after a first
    call has loaded the library's code and its static array);
  * a withheld pipeline stage is reported by gemm_noalloc_get_status, which
    then clears it, and the next call is correct;
  * a split beyond the static scratch is refused before anything runs.

This file is collected last on purpose, and every test in it works whether
it runs alone in a fresh process or after the rest of the suite.
"""

import numpy as np
import pytest
import torch

import gemm_inputs as gi
import oracle
from dense_gemm_02_gb300 import binding as b

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()
    b.lib()


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _call(fn, A, B, C, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    c_type = b.GEMM_OUT_F32 if C.dtype == torch.float32 else b.GEMM_OUT_BF16
    return fn(M, N, K, alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), beta,
              C.data_ptr(), C.stride(0), c_type, torch.cuda.current_stream().cuda_stream)


def _bits(C):
    if C.dtype == torch.float32:
        return C.cpu().numpy()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def _operands(M, N, K, out, beta, seed, integer):
    kind = "integer" if integer else "normal"
    A = gi.draw(kind, seed, 0, (M, K), dtype="bf16")
    B = gi.draw(kind, seed, 1, (K, N), sigma=0.02, dtype="bf16")
    cdt = "bf16" if out == torch.bfloat16 else "f32"
    C = gi.draw(kind, seed, 2, (M, N), dtype=cdt) if beta != 0.0 else None
    return A, B, C


def _dev_c(C, M, N, out):
    if C is None:
        return torch.full((M, N), float("nan"), device="cuda").to(out)
    return _dev_bf16(C) if out == torch.bfloat16 else torch.from_numpy(C).cuda()


# Small-M shapes, so that both entry points split K and the static scratch
# is really used: (M, N, K, alpha, beta, output dtype).
CASES = [
    (64, 2048, 4096, 1.0, 0.0, torch.float32),
    (96, 1024, 2048, 0.5, 1.0, torch.bfloat16),
]


def test_noalloc_allocates_nothing_and_matches_gemm_bf16_bit_for_bit():
    # every buffer this test uses exists before the measured calls
    runs = []
    for call, (M, N, K, alpha, beta, out) in enumerate(CASES):
        A, B, C = _operands(M, N, K, out, beta, 0x5EED0A00 + call, integer=False)
        dA, dB = _dev_bf16(A), _dev_bf16(B)
        Cin = _dev_c(C, M, N, out)
        runs.append((dA, dB, Cin, Cin.clone(), Cin.clone(), alpha, beta))
    warm = [r[2].clone() for r in runs]
    torch.cuda.synchronize()
    # A first call of each case loads the library's kernels and its static
    # array (module loading is the driver's, not a call of ours); after that
    # the device's free memory must not move.
    for (dA, dB, _c, _r, _n, alpha, beta), Cw in zip(runs, warm):
        assert _call(b.gemm_bf16_noalloc, dA, dB, Cw, alpha, beta) == b.GEMM_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for dA, dB, _Cin, _C_ref, C_new, alpha, beta in runs:  # two calls in a row
        assert _call(b.gemm_bf16_noalloc, dA, dB, C_new, alpha, beta) == b.GEMM_OK
    assert b.noalloc_get_status(torch.cuda.current_stream().cuda_stream) == (b.GEMM_OK, 0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    for dA, dB, _Cin, C_ref, C_new, alpha, beta in runs:
        assert _call(b.gemm_bf16, dA, dB, C_ref, alpha, beta) == b.GEMM_OK
    torch.cuda.synchronize()
    for i, (_a, _b, _c, C_ref, C_new, _al, _be) in enumerate(runs):
        got, want = _bits(C_new), _bits(C_ref)
        assert np.array_equal(got, want), f"call {i}: differs from gemm_bf16"
    for Cw, r in zip(warm, runs):  # the warm-up calls gave the same bits
        assert np.array_equal(_bits(Cw), _bits(r[4]))


@pytest.mark.parametrize("integer", [True, False], ids=["integer_bit_exact", "normal_tolerance"])
def test_noalloc_matches_the_oracle(integer):
    for call, (M, N, K, alpha, beta, out) in enumerate(CASES):
        A, B, C = _operands(M, N, K, out, beta, 0x5EED0B00 + call, integer=integer)
        dC = _dev_c(C, M, N, out)
        assert _call(b.gemm_bf16_noalloc, _dev_bf16(A), _dev_bf16(B), dC, alpha, beta) == b.GEMM_OK
        assert b.noalloc_get_status(torch.cuda.current_stream().cuda_stream)[0] == b.GEMM_OK
        ref = oracle.gemm(A, B, C, alpha=alpha, beta=beta)
        got = _bits(dC)
        if integer:
            want = oracle.round_bf16(ref) if out == torch.bfloat16 else oracle.round_f32(ref)
            assert np.array_equal(got, want), f"call {call}"
        else:
            gv = (gi.bf16_bits_to_f32(got) if out == torch.bfloat16 else got).astype(np.float64)
            bad = (np.abs(gv - ref) > (2.0**-7) * np.abs(ref) + 1e-2) | ~np.isfinite(gv)
            assert int(bad.sum()) == 0, f"call {call}: {int(bad.sum())} outputs out of tolerance"


def test_noalloc_status_reports_a_withheld_stage_and_clears_it():
    M, N, K = 64, 2048, 4096  # splits K
    A = gi.draw("integer", 0x5EED0C00, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", 0x5EED0C00, 1, (K, N), dtype="bf16")
    dA, dB = _dev_bf16(A), _dev_bf16(B)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert b.noalloc_get_status(stream)[0] == b.GEMM_OK
    old = b.get_config("watchdog_ms")
    b.set_config("watchdog_ms", 200)
    b.set_config("fault_inject", 1)  # the producer withholds one stage
    try:
        assert _call(b.gemm_bf16_noalloc, dA, dB, C, 1.0, 0.0) == b.GEMM_OK
        rc, info = b.noalloc_get_status(stream)
    finally:
        b.set_config("fault_inject", 0)
        b.set_config("watchdog_ms", old)
    assert rc == b.GEMM_ERR_DEVICE_TIMEOUT
    assert info & 0xFF in (1, 2, 3)  # producer, MMA issuer or epilogue
    assert b.noalloc_get_status(stream) == (b.GEMM_OK, 0)  # read once, then clear
    # the library's own status word is a different record
    assert b.get_device_status(stream) == b.GEMM_OK
    # the next call is correct
    assert _call(b.gemm_bf16_noalloc, dA, dB, C, 1.0, 0.0) == b.GEMM_OK
    assert b.noalloc_get_status(stream)[0] == b.GEMM_OK
    assert np.array_equal(C.cpu().numpy(), oracle.round_f32(oracle.gemm(A, B)))


def test_noalloc_rejects_a_split_beyond_its_scratch():
    M, N, K = 256, 4096, 2048
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    b.set_config("split_k", 16)  # 32 tiles x 16 slices of 128 KiB partials: 64 MiB
    try:
        rc = _call(b.gemm_bf16_noalloc, A, B, C, 1.0, 0.0)
    finally:
        b.set_config("split_k", 0)
    assert rc == b.GEMM_ERR_SCRATCH_LIMIT
    assert "scratch" in b.status_string(rc)
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())  # nothing was launched
