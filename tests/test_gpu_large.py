"""Outputs past 2^31 elements: every kernel addresses C, A and the split-K
workspace with 64-bit offsets.  Integer-valued operands, so sampled
entries (oracle.gemm_entries) must match bit for bit, including entries
in the last rows and columns."""

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.init()


def sample_rows_cols(M, N, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rng.integers(0, M, n), [0, M - 1, M - 1, M // 2]])
    cols = np.concatenate([rng.integers(0, N, n), [0, N - 1, 0, N - 1]])
    return rows.astype(np.int64), cols.astype(np.int64)


@pytest.mark.parametrize("dtype,out", [("f32", "f32"), ("bf16", "f32"), ("bf16", "bf16")])
def test_output_beyond_2_31_elements(dtype, out):
    M, N, K = 65600, 32800, 72  # M * N = 2.15e9 > 2^31
    seed = 15000 + (dtype == "bf16") + 2 * (out == "bf16")
    A = gi.draw("integer", seed, 0, (M, K), dtype=dtype)
    B = gi.draw("integer", seed, 1, (K, N), dtype=dtype)
    if dtype == "f32":
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = g.sgemm(dA, dB)
        want = "sgemm_tma"
    else:
        dA = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
        dB = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)
        C = g.gemm_bf16(dA, dB, out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
        want = "bf16_tcgen05"
    torch.cuda.synchronize()
    g.binding.check(g.binding.get_device_status(), "device status")
    assert g.binding.last_kernel() == want
    rows, cols = sample_rows_cols(M, N, 2000, seed)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    got = got.float().cpu().numpy() if out == "f32" else got.view(torch.int16).cpu().numpy()
    ref = oracle.gemm_entries(A, B, rows, cols)
    if out == "f32":
        assert np.array_equal(got, oracle.round_f32(ref))
    else:
        assert np.array_equal(got.view(np.uint16), oracle.round_bf16(ref))
    del C
    torch.cuda.empty_cache()
