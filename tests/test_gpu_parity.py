"""GPU parity: the CUDA kernels, called through the C ABI, against the CPU
oracle on the same seeded inputs.

* integer-valued inputs in {-2..2}: every product and partial sum is an
  integer (or half-integer when alpha = 0.5) far below 2^24, so fp32 and the
  tensor cores' fp32 accumulation are exact in any order and the single final
  rounding is the same on both sides: results must match bit for bit;
* random inputs: FP32 max |C - C_ref| <= 1e-5 * K; BF16 elementwise
  |C - C_ref| <= 2^-7 |C_ref| + 1e-2, C_ref from the same bf16 operands;
* shapes that are not tile multiples, pitches larger than the row length
  (odd ones take the generic kernels), guard bands around C, NaN-filled C
  when beta == 0, and run-to-run determinism.
"""

import itertools

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
from gpu_helpers import (GuardedC, bf16_from_dev, bf16_to_dev, bf16_tolerance_violations,
                         f32_to_dev, widen)

pytestmark = pytest.mark.gpu

# Ragged shapes from the tail set {1, 7, 63, 65, 127, 129, 1000, 1001}.
SHAPES = sorted(set(itertools.product((1, 7, 65, 129), (1, 63, 127, 1001), (1, 65, 1000)))
                | {(1000, 1000, 1000), (1001, 1001, 1001), (256, 256, 256), (300, 520, 777)})
# Shapes whose rows TMA can fetch (N, K multiples of 8) but that are not
# multiples of the tcgen05 tiles (128 x 128/256 x 64).
SHAPES_TC = sorted(set(itertools.product((1, 7, 65, 129, 257), (8, 72, 264, 1000), (8, 72, 1000)))
                   | {(1000, 1000, 1000), (1024, 1024, 1024), (128, 256, 64), (383, 1288, 2056)})


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_02_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.init()


def _status_ok():
    g.binding.check(g.binding.get_device_status(), "device status")


def run_f32(A, B, Cin, alpha, beta, lda=None, ldb=None, ldc=None):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = f32_to_dev(A, lda), f32_to_dev(B, ldb)
    init = Cin if Cin is not None else np.full((M, N), np.nan, np.float32)
    C = GuardedC(M, N, ldc or N, "f32", init)
    g.sgemm(dA, dB, C.view, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    _status_ok()
    return C


def run_bf16(A, B, Cin, alpha, beta, out, lda=None, ldb=None, ldc=None):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = bf16_to_dev(A, lda), bf16_to_dev(B, ldb)
    if Cin is None:
        init = (np.full((M, N), 0x7FC0, np.uint16) if out == "bf16"
                else np.full((M, N), np.nan, np.float32))
    else:
        init = Cin
    C = GuardedC(M, N, ldc or N, out, init)
    g.gemm_bf16(dA, dB, C.view, alpha=alpha, beta=beta,
                out_dtype=torch.bfloat16 if out == "bf16" else torch.float32)
    torch.cuda.synchronize()
    _status_ok()
    return C


# ------------------------------------------------------------------ FP32

@pytest.mark.parametrize("M,N,K", SHAPES)
def test_f32_integer_bit_exact(M, N, K):
    seed = gi.WORKLOAD_SEED_BASE + gi.INTEGER_PASS_OFFSET + M * 7 + N * 13 + K
    A = gi.draw("integer", seed, 0, (M, K))
    B = gi.draw("integer", seed, 1, (K, N))
    Cin = gi.draw("integer", seed, 2, (M, N))
    C = run_f32(A, B, Cin, 1.0, -1.0)
    # rows TMA can fetch (pitches multiples of 4 floats) take the TMA kernel
    want = "sgemm_tma" if (K % 4 == 0 and N % 4 == 0) else "sgemm_simt"
    assert g.binding.last_kernel() == want
    ref = oracle.round_f32(oracle.gemm(A, B, Cin, alpha=1.0, beta=-1.0))
    assert np.array_equal(C.result(), ref)
    assert C.guards_intact()


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_f32_uniform_within_tolerance(M, N, K):
    seed = gi.WORKLOAD_SEED_BASE + M * 7 + N * 13 + K
    A = gi.draw("uniform", seed, 0, (M, K))
    B = gi.draw("uniform", seed, 1, (K, N))
    C = run_f32(A, B, None, 1.0, 0.0)  # C pre-filled with NaN: must not be read
    ref = oracle.gemm(A, B)
    err = np.abs(C.result().astype(np.float64) - ref)
    assert np.isfinite(C.result()).all()
    assert err.max() <= 1e-5 * K
    assert C.guards_intact()


@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad", [(3, 5, 7), (4, 4, 4), (1, 0, 2), (0, 1, 0)])
def test_f32_pitched_operands(lda_pad, ldb_pad, ldc_pad):
    M, N, K = 129, 127, 1001
    seed = 777 + lda_pad
    A = gi.draw("integer", seed, 0, (M, K))
    B = gi.draw("integer", seed, 1, (K, N))
    Cin = gi.draw("integer", seed, 2, (M, N))
    C = run_f32(A, B, Cin, 2.0, 0.5, lda=K + lda_pad, ldb=N + ldb_pad, ldc=N + ldc_pad)
    ref = oracle.round_f32(oracle.gemm(A, B, Cin, alpha=2.0, beta=0.5))
    assert np.array_equal(C.result(), ref)
    assert C.guards_intact()


@pytest.mark.parametrize("force", [0, 1])
def test_f32_tma_and_cp_async_kernels_agree_exactly(force):
    M, N, K = 300, 520, 776
    A = gi.draw("integer", 2024, 0, (M, K))
    B = gi.draw("integer", 2024, 1, (K, N))
    g.set_config("force_path", force)
    try:
        C = run_f32(A, B, None, 1.0, 0.0)
    finally:
        g.set_config("force_path", 0)
    assert g.binding.last_kernel() == ("sgemm_simt" if force else "sgemm_tma")
    assert np.array_equal(C.result(), oracle.round_f32(oracle.gemm(A, B)))
    assert C.guards_intact()


# Shapes whose tile count leaves a remainder over the SM count, so the
# FP32 kernel splits the remaining tiles along K (on 152 SMs: 2304^2 has 324
# tiles, 20 past two full rounds, split 4 ways at K = 520; 1000^2 has 64,
# all split; 4096 x 4096 has 1024, 112 split 4 ways).  tail_split_off = 1
# runs the same shapes unsplit.
@pytest.mark.parametrize("M,N,K", [(2304, 2304, 520), (1000, 1000, 1000), (4096, 4096, 520),
                                   (1001, 1003, 999)])
@pytest.mark.parametrize("tail_off", [0, 1])
def test_f32_partial_wave_k_split_integer(M, N, K, tail_off):
    seed = 8800 + M + N + K
    A = gi.draw("integer", seed, 0, (M, K))
    B = gi.draw("integer", seed, 1, (K, N))
    Cin = gi.draw("integer", seed, 2, (M, N))
    g.set_config("tail_split_off", tail_off)
    try:
        C = run_f32(A, B, Cin, 0.5, -1.0, lda=K + (-K) % 4, ldb=N + (-N) % 4)
    finally:
        g.set_config("tail_split_off", 0)
    assert g.binding.last_kernel() == "sgemm_tma"
    ref = oracle.round_f32(oracle.gemm(A, B, Cin, alpha=0.5, beta=-1.0))
    got = C.result()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


def test_f32_partial_wave_k_split_uniform_tolerance_and_repeatable():
    M, N, K = 2304, 2304, 1032
    A = gi.draw("uniform", 8900, 0, (M, K))
    B = gi.draw("uniform", 8900, 1, (K, N))
    C1 = run_f32(A, B, None, 1.0, 0.0)
    C2 = run_f32(A, B, None, 1.0, 0.0)
    assert np.array_equal(C1.result(), C2.result())
    ref = oracle.gemm(A, B)
    assert np.abs(C1.result().astype(np.float64) - ref).max() <= 1e-5 * K


def test_f32_alpha_zero_and_k_zero_scale_c():
    M, N, K = 70, 90, 33
    A = np.full((M, K), np.nan, np.float32)
    B = np.full((K, N), np.nan, np.float32)
    Cin = gi.draw("integer", 5, 2, (M, N))
    C = run_f32(A, B, Cin, 0.0, 3.0)
    assert g.binding.last_kernel() == "scale_c"
    assert np.array_equal(C.result(), 3.0 * Cin)
    C0 = GuardedC(M, N, N + 3, "f32", Cin)
    g.sgemm(torch.zeros((M, 0), device="cuda"), torch.zeros((0, N), device="cuda"), C0.view,
            alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert (C0.result() == 0).all() and C0.guards_intact()


# ------------------------------------------------------------------ BF16

@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("M,N,K", SHAPES_TC + SHAPES)
def test_bf16_integer_bit_exact(M, N, K, out):
    seed = gi.WORKLOAD_SEED_BASE + gi.INTEGER_PASS_OFFSET + M * 5 + N * 11 + K
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype=out)
    C = run_bf16(A, B, Cin, 0.5, 1.0, out)
    # K % 8 == 0 and N % 8 == 0 rows are TMA-able; the rest go generic.
    want = "bf16_tcgen05" if (K % 8 == 0 and N % 8 == 0) else "bf16_simt"
    assert g.binding.last_kernel() == want
    R = oracle.gemm(A, B, Cin, alpha=0.5, beta=1.0)
    ref = oracle.round_bf16(R) if out == "bf16" else oracle.round_f32(R)
    got = C.result()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("M,N,K", SHAPES_TC + [(7, 63, 65), (129, 1001, 1000), (1001, 1001, 1001)])
def test_bf16_normal_within_tolerance(M, N, K, out):
    seed = gi.WORKLOAD_SEED_BASE + M * 5 + N * 11 + K
    A = gi.draw("normal", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", seed, 1, (K, N), dtype="bf16")
    C = run_bf16(A, B, None, 1.0, 0.0, out)  # NaN-filled C, beta = 0
    ref = oracle.gemm(A, B)
    assert bf16_tolerance_violations(widen(C.result(), out), ref) == 0
    assert C.guards_intact()


@pytest.mark.parametrize("pads", [(8, 8, 8), (8, 16, 3), (1, 8, 0), (8, 1, 5), (3, 3, 3)])
def test_bf16_pitched_operands(pads):
    lda_pad, ldb_pad, ldc_pad = pads
    M, N, K = 200, 264, 320
    seed = 4242 + sum(pads)
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype="bf16")
    C = run_bf16(A, B, Cin, 1.0, -2.0, "bf16", lda=K + lda_pad, ldb=N + ldb_pad, ldc=N + ldc_pad)
    tma = (K + lda_pad) % 8 == 0 and (N + ldb_pad) % 8 == 0
    assert g.binding.last_kernel() == ("bf16_tcgen05" if tma else "bf16_simt")
    ref = oracle.round_bf16(oracle.gemm(A, B, Cin, alpha=1.0, beta=-2.0))
    assert np.array_equal(C.result(), ref)
    assert C.guards_intact()


# stage_pairs 0 (default): K blocks two at a time where the ring is deep
# enough (the 128-wide tiles' six stages, the slices' odd block counts
# ending on a single stage); 2: one at a time
@pytest.mark.parametrize("stage_pairs", [0, 2])
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("split_k", [1, 2, 3, 5])
def test_bf16_tiles_and_split_k_integer(tile_n, split_k, stage_pairs):
    M, N, K = 192, 640, 1536
    seed = 99 + tile_n + split_k
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype="f32")
    g.set_config("bf16_tile_n", tile_n)
    g.set_config("split_k", split_k)
    g.set_config("stage_pairs", stage_pairs)
    try:
        C = run_bf16(A, B, Cin, 1.0, 1.0, "f32")
    finally:
        g.set_config("bf16_tile_n", 0)
        g.set_config("split_k", 0)
        g.set_config("stage_pairs", 0)
    ref = oracle.round_f32(oracle.gemm(A, B, Cin, alpha=1.0, beta=1.0))
    assert np.array_equal(C.result(), ref)
    assert C.guards_intact()


# Few tiles and a long K: with stream_k = 1 the K iterations of all tiles
# are dealt out to the SMs in equal ranges (tiles shared by 2-4 CTAs, summed
# in K order); stream_k = 0 (default) runs equal K slices per tile.
@pytest.mark.parametrize("M,N,K", [(64, 8192, 2048), (1, 1000, 4096), (200, 520, 3000),
                                   (129, 264, 1000), (7, 72, 8192), (64, 2048, 8200)])
@pytest.mark.parametrize("stream_k", [0, 1])
def test_bf16_stream_k_integer(M, N, K, stream_k):
    seed = 6600 + M + N + K
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype="f32")
    g.set_config("stream_k", stream_k)
    try:
        C = run_bf16(A, B, Cin, 0.5, 1.0, "f32")
    finally:
        g.set_config("stream_k", 0)
    assert g.binding.last_kernel() == "bf16_tcgen05"
    ref = oracle.round_f32(oracle.gemm(A, B, Cin, alpha=0.5, beta=1.0))
    got = C.result()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


def test_bf16_stream_k_normal_tolerance_and_repeatable():
    M, N, K = 64, 8192, 8192
    A = gi.draw("normal", 6700, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 6700, 1, (K, N), sigma=0.02, dtype="bf16")
    g.set_config("stream_k", 1)
    try:
        C1 = run_bf16(A, B, None, 1.0, 0.0, "f32")
        C2 = run_bf16(A, B, None, 1.0, 0.0, "f32")
    finally:
        g.set_config("stream_k", 0)
    assert np.array_equal(C1.result(), C2.result())
    assert bf16_tolerance_violations(widen(C1.result(), "f32"), oracle.gemm(A, B)) == 0


# Tile counts that leave a partial last wave on a 152-SM part, so the tail
# tiles are cut into 2 or 4 narrower sub-tiles; the ragged-N shape puts
# sub-tiles wholly past the N edge.
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 256), (1792, 3328, 256), (1792, 3144, 200),
                                   (1000, 2056, 72)])
@pytest.mark.parametrize("tail_off", [0, 1])
def test_bf16_partial_wave_tail_split_integer(M, N, K, tail_off):
    seed = 555 + M + N + K
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype="bf16")
    g.set_config("tail_split_off", tail_off)
    try:
        C = run_bf16(A, B, Cin, 1.0, 1.0, "bf16")
    finally:
        g.set_config("tail_split_off", 0)
    assert g.binding.last_kernel() == "bf16_tcgen05"
    ref = oracle.round_bf16(oracle.gemm(A, B, Cin, alpha=1.0, beta=1.0))
    got = C.result()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


PAIR_SHAPES = [(1, 8, 8), (7, 72, 72), (129, 264, 1000), (257, 1000, 72), (300, 520, 776),
               (1000, 1000, 1000), (2048, 2048, 512), (4096, 4096, 256), (1792, 3144, 200)]


@pytest.mark.parametrize("cta_pair", [1, 2])
@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
def test_bf16_single_and_pair_kernels_integer(M, N, K, cta_pair):
    seed = 777 + M * 3 + N * 5 + K
    A = gi.draw("integer", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", seed, 1, (K, N), dtype="bf16")
    Cin = gi.draw("integer", seed, 2, (M, N), dtype="bf16")
    g.set_config("cta_pair", cta_pair)
    try:
        C = run_bf16(A, B, Cin, 0.5, 1.0, "bf16")
    finally:
        g.set_config("cta_pair", 0)
    assert g.binding.last_kernel() == "bf16_tcgen05"
    ref = oracle.round_bf16(oracle.gemm(A, B, Cin, alpha=0.5, beta=1.0))
    got = C.result()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_pair_kernel_normal_tolerance(out):
    M, N, K = 1000, 1288, 2056
    A = gi.draw("normal", 4321, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 4321, 1, (K, N), dtype="bf16")
    g.set_config("cta_pair", 2)
    try:
        C = run_bf16(A, B, None, 1.0, 0.0, out)
    finally:
        g.set_config("cta_pair", 0)
    ref = oracle.gemm(A, B)
    assert bf16_tolerance_violations(widen(C.result(), out), ref) == 0
    assert C.guards_intact()


def test_bf16_forced_generic_matches_tcgen05_on_integers():
    M, N, K = 257, 384, 512
    A = gi.draw("integer", 31337, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", 31337, 1, (K, N), dtype="bf16")
    C1 = run_bf16(A, B, None, 1.0, 0.0, "bf16")
    assert g.binding.last_kernel() == "bf16_tcgen05"
    g.set_config("force_path", 1)
    try:
        C2 = run_bf16(A, B, None, 1.0, 0.0, "bf16")
        assert g.binding.last_kernel() == "bf16_simt"
    finally:
        g.set_config("force_path", 0)
    assert np.array_equal(C1.result(), C2.result())


def test_bf16_alpha_zero_scales_c():
    M, N, K = 33, 48, 64
    A = np.full((M, K), 0x7FC0, np.uint16)
    B = np.full((K, N), 0x7FC0, np.uint16)
    Cin = gi.draw("integer", 8, 2, (M, N), dtype="bf16")
    C = run_bf16(A, B, Cin, 0.0, -1.0, "bf16")
    assert g.binding.last_kernel() == "scale_c"
    assert np.array_equal(C.result(), oracle.round_bf16(-oracle.widen_bf16(Cin)))


def test_bf16_nan_and_inf_propagate():
    M, N, K = 128, 256, 128
    A = gi.draw("integer", 9, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", 9, 1, (K, N), dtype="bf16")
    A[3, 5] = 0x7F80   # +inf
    A[7, 9] = 0x7FC0   # NaN
    C = run_bf16(A, B, None, 1.0, 0.0, "f32")
    ref = oracle.gemm(A, B)
    got = C.result().astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_determinism_two_runs_bit_identical(dtype):
    M, N, K = 64, 1024, 4096  # small M: the tcgen05 kernel splits K here
    if dtype == "f32":
        A = gi.draw("uniform", 1, 0, (M, K))
        B = gi.draw("uniform", 1, 1, (K, N))
        r1 = run_f32(A, B, None, 1.0, 0.0).result()
        r2 = run_f32(A, B, None, 1.0, 0.0).result()
    else:
        A = gi.draw("normal", 1, 0, (M, K), dtype="bf16")
        B = gi.draw("normal", 1, 1, (K, N), sigma=0.02, dtype="bf16")
        r1 = run_bf16(A, B, None, 1.0, 0.0, "f32").result()
        r2 = run_bf16(A, B, None, 1.0, 0.0, "f32").result()
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))


def test_host_buffer_entry_point_matches_device_path():
    M, N, K = 300, 200, 136
    A = gi.draw("normal", 3, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 3, 1, (K, N), dtype="bf16")
    hA = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).pin_memory()
    hB = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).pin_memory()
    out = g.gemm(hA, hB)
    assert not out.is_cuda
    dev = g.gemm_bf16(bf16_to_dev(A), bf16_to_dev(B))
    torch.cuda.synchronize()
    assert np.array_equal(out.view(torch.int16).numpy().view(np.uint16), bf16_from_dev(dev))


def test_watchdog_reports_a_withheld_stage_and_recovers():
    M, N, K = 512, 512, 1024
    A = gi.draw("integer", 17, 0, (M, K), dtype="bf16")
    B = gi.draw("integer", 17, 1, (K, N), dtype="bf16")
    dA, dB = bf16_to_dev(A), bf16_to_dev(B)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    old = g.get_config("watchdog_ms")
    g.set_config("watchdog_ms", 200)
    g.set_config("fault_inject", 1)
    try:
        g.gemm_bf16(dA, dB, C, out_dtype=torch.float32)
        rc = g.binding.get_device_status()
    finally:
        g.set_config("fault_inject", 0)
        g.set_config("watchdog_ms", old)
    assert rc == g.binding.GEMM_ERR_DEVICE_TIMEOUT
    info = g.binding.get_device_fault_info()
    assert info & 0xFF in (1, 2, 3)
    # the context is still usable and the next call is correct
    g.gemm_bf16(dA, dB, C, out_dtype=torch.float32)
    assert g.binding.get_device_status() == g.binding.GEMM_OK
    ref = oracle.round_f32(oracle.gemm(A, B))
    assert np.array_equal(C.cpu().numpy(), ref)


def test_sgemm_watchdog_reports_a_withheld_stage_and_recovers():
    M, N, K = 512, 512, 1024
    A = gi.draw("integer", 18, 0, (M, K))
    B = gi.draw("integer", 18, 1, (K, N))
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    old = g.get_config("watchdog_ms")
    g.set_config("watchdog_ms", 200)
    g.set_config("fault_inject", 1)
    try:
        g.sgemm(dA, dB, C)
        rc = g.binding.get_device_status()
    finally:
        g.set_config("fault_inject", 0)
        g.set_config("watchdog_ms", old)
    assert g.binding.last_kernel() == "sgemm_tma"
    assert rc == g.binding.GEMM_ERR_DEVICE_TIMEOUT
    assert g.binding.get_device_fault_info() & 0xFF == 4  # the SGEMM's role code
    g.sgemm(dA, dB, C)
    assert g.binding.get_device_status() == g.binding.GEMM_OK
    assert np.array_equal(C.cpu().numpy(), oracle.round_f32(oracle.gemm(A, B)))


def test_tensor_map_reuse_across_calls_integer():
    """Calls that repeat, or only partly repeat, an earlier call's base
    addresses, shapes and pitches: the encoded tensor maps a call reuses must
    match its own arguments exactly (more distinct operands than the
    per-thread cache holds, the same buffers with a different M, N, pitch
    or output type, and repeats)."""
    M, N, K = 384, 520, 264
    bufs = []
    for i in range(14):
        A = gi.draw("integer", 19000 + i, 0, (M, K), dtype="bf16")
        B = gi.draw("integer", 19000 + i, 1, (K, N), dtype="bf16")
        bufs.append((A, B, bf16_to_dev(A), bf16_to_dev(B)))
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    Cb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for rnd in range(2):
        for A, B, dA, dB in bufs:
            g.gemm_bf16(dA, dB, C, out_dtype=torch.float32)
            assert np.array_equal(C.cpu().numpy(), oracle.round_f32(oracle.gemm(A, B)))
    A, B, dA, dB = bufs[0]
    # same base addresses, fewer rows / columns (views), other pitches
    g.gemm_bf16(dA[:200], dB, C[:200], out_dtype=torch.float32)
    assert np.array_equal(C[:200].cpu().numpy(), oracle.round_f32(oracle.gemm(A[:200], B)))
    sub = C[:, :256]
    g.gemm_bf16(dA, dB[:, :256], sub, out_dtype=torch.float32)
    assert np.array_equal(sub.cpu().numpy(), oracle.round_f32(oracle.gemm(A, B[:, :256])))
    g.gemm_bf16(dA, dB, Cb)
    assert np.array_equal(bf16_from_dev(Cb), oracle.round_bf16(oracle.gemm(A, B)))
    # FP32 path through the same cache
    Af = gi.draw("integer", 19100, 0, (M, K))
    Bf = gi.draw("integer", 19100, 1, (K, N))
    dAf, dBf = torch.from_numpy(Af).cuda(), torch.from_numpy(Bf).cuda()
    for _ in range(2):
        g.sgemm(dAf, dBf, C)
        assert np.array_equal(C.cpu().numpy(), oracle.round_f32(oracle.gemm(Af, Bf)))
    g.sgemm(dAf[:100], dBf, C[:100])
    assert np.array_equal(C[:100].cpu().numpy(), oracle.round_f32(oracle.gemm(Af[:100], Bf)))
    _status_ok()
