"""The allocation-free entry point, gemm_bf16_noalloc, for callers that
cannot call cudaMalloc (code running under a host application that owns all
device memory through its own allocator, or latency-critical code that
cannot take an allocation's implicit synchronisation).  It runs the same
tcgen05 kernel as gemm_bf16 but keeps its split-K scratch in a static device
array inside the library.

Checked through the C ABI against gemm_bf16 on two calls in a row, with the
BF16 tolerance the other tests use (|C - C_ref| <= 2^-7 |C_ref| + 1e-2), and
for its size limit.  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from dense_gemm_02_gb300 import binding as b

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    b.lib()


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _call(fn, A, B, C, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    c_type = b.GEMM_OUT_F32 if C.dtype == torch.float32 else b.GEMM_OUT_BF16
    return fn(M, N, K, alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), beta,
              C.data_ptr(), C.stride(0), c_type, torch.cuda.current_stream().cuda_stream)


def _as_f64(C):
    return C.float().cpu().numpy().astype(np.float64)


# Small-M shapes, so that both entry points split K and the static scratch
# is really used: (M, N, K, alpha, beta, output dtype).
CASES = [
    (64, 2048, 4096, 1.0, 0.0, torch.float32),
    (96, 1024, 2048, 0.5, 1.0, torch.bfloat16),
]


def test_noalloc_matches_gemm_bf16_on_two_calls_in_a_row():
    for call, (M, N, K, alpha, beta, out) in enumerate(CASES):
        seed = 0x5EED0A00 + call
        A = _dev_bf16(gi.draw("normal", seed, 0, (M, K), dtype="bf16"))
        B = _dev_bf16(gi.draw("normal", seed, 1, (K, N), sigma=0.02, dtype="bf16"))
        if beta != 0.0:
            c0 = gi.draw("normal", seed, 2, (M, N), dtype="bf16" if out == torch.bfloat16 else "f32")
            Cin = (_dev_bf16(c0) if out == torch.bfloat16 else torch.from_numpy(c0).cuda())
        else:
            Cin = torch.full((M, N), float("nan"), device="cuda").to(out)
        C_ref, C_new = Cin.clone(), Cin.clone()
        assert _call(b.gemm_bf16, A, B, C_ref, alpha, beta) == b.GEMM_OK
        assert _call(b.gemm_bf16_noalloc, A, B, C_new, alpha, beta) == b.GEMM_OK
        torch.cuda.synchronize()
        ref, got = _as_f64(C_ref), _as_f64(C_new)
        assert np.isfinite(got).all()
        bad = np.abs(got - ref) > (2.0**-7) * np.abs(ref) + 1e-2
        assert int(bad.sum()) == 0, f"call {call}: {int(bad.sum())} outputs out of tolerance"


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
