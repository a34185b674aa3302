"""The seeded input generator: published splitmix64 outputs, determinism,
value sets and moments of each distribution, and bf16 rounding of operands."""

import numpy as np
import pytest

import gemm_inputs as gi


def test_splitmix64_published_first_outputs():
    # splitmix64 started from state 0: the first output is the widely quoted
    # 0xE220A8397B1DCDAF (Steele, Lea, Flood 2014 reference sequence).
    x = gi.splitmix64_from_state(0, 0, 1)
    assert int(x[0]) == 0xE220A8397B1DCDAF


def test_counter_based_any_order():
    full = gi.splitmix64_stream(123, 2, 0, 1000)
    part = gi.splitmix64_stream(123, 2, 600, 400)
    assert np.array_equal(full[600:], part)
    other = gi.splitmix64_stream(123, 3, 0, 1000)
    assert not np.array_equal(full, other)


def test_uniform_exact_grid_and_range():
    u = gi.uniform_f32(7, 0, 1 << 18)
    assert u.dtype == np.float32
    assert u.min() >= -1.0 and u.max() < 1.0
    k = (u.astype(np.float64) + 1.0) * 2.0**23
    assert np.array_equal(k, np.round(k))
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01


def test_normal_moments_and_sigma():
    z = gi.normal_f32(9, 1, 1 << 18)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    z2 = gi.normal_f32(9, 1, 1 << 18, sigma=0.02)
    assert np.allclose(z2, (z.astype(np.float64) * 0.02).astype(np.float32), rtol=1e-6)


def test_integer_values():
    v = gi.integer_f32(5, 2, 100000)
    assert set(np.unique(v).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_deterministic_and_chunk_independent():
    a = gi.draw("normal", 0x5EED0003, 0, (3000, 2000), dtype="bf16")
    b = gi.draw("normal", 0x5EED0003, 0, (3000, 2000), dtype="bf16")
    assert np.array_equal(a, b)
    flat = gi.normal_f32(0x5EED0003, 0, 3000 * 2000)
    assert np.array_equal(gi.f32_to_bf16_bits(flat).reshape(3000, 2000), a)


def test_bf16_operand_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = gi.normal_f32(77, 0, 1 << 16) * np.float32(1000.0)
    ours = gi.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = gi.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_batch_operands_continue_the_streams():
    from gemm_inputs.workloads import WORKLOADS

    w = WORKLOADS["bf16_mlp_8192x14336x4096"]
    import dataclasses

    small = dataclasses.replace(w, M=6, N=5, K=4)
    A0, B0, C0 = small.operands()
    a0, b0, c0 = small.batch_operands(0)
    assert np.array_equal(A0, a0) and np.array_equal(B0, b0) and np.array_equal(C0, c0)
    a1, b1, c1 = small.batch_operands(1)
    # matrix 1 holds the next elements of each stream
    big_a = gi.draw(small.dist, small.seed, 0, (12, 4), sigma=small.sigma_a, dtype=small.dtype)
    assert np.array_equal(big_a[6:], a1)
    assert not np.array_equal(b0, b1) and not np.array_equal(c0, c1)
