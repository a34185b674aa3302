"""Pins for the CPU oracle, each fixed by the mathematics rather than by the
oracle itself: identity and permutation products, a rank-1 closed form, the
alpha/beta conventions, brute force against exact Python integers and
fractions on every tiny shape, a library special case (numpy float64
matmul), and the bf16 / fp32 rounding rules.  No GPU involved.
"""

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import gemm_inputs as gi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- products

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identity_left_and_right(oracle, dtype):
    M, K, N = 37, 37, 53
    B = gi.draw("normal", 11, 1, (K, N), dtype=dtype)
    eye = np.eye(K, dtype=np.float32)
    eye = eye if dtype == "f32" else gi.f32_to_bf16_bits(eye)
    R = oracle.gemm(eye, B)
    Bd = B.astype(np.float64) if dtype == "f32" else oracle.widen_bf16(B)
    assert np.array_equal(R, Bd)
    # right identity: A @ I = A
    A = gi.draw("uniform", 12, 0, (M, K), dtype=dtype)
    R2 = oracle.gemm(A, eye)
    Ad = A.astype(np.float64) if dtype == "f32" else oracle.widen_bf16(A)
    assert np.array_equal(R2, Ad)


def test_permutation_rows_and_columns(oracle):
    M, K, N = 41, 41, 29
    perm = _rng(3).permutation(M)
    P = np.zeros((M, K), dtype=np.float32)
    P[np.arange(M), perm] = 1.0
    B = gi.draw("uniform", 13, 1, (K, N))
    R = oracle.gemm(P, B)
    assert np.array_equal(R, B[perm].astype(np.float64))
    # right multiplication by a permutation permutes columns
    qperm = _rng(4).permutation(N)
    Q = np.zeros((N, N), dtype=np.float32)
    Q[qperm, np.arange(N)] = 1.0
    R2 = oracle.gemm(B, Q)
    assert np.array_equal(R2, B[:, qperm].astype(np.float64))


def test_non_square_permutation_detects_transpose(oracle):
    # A selects rows of B; a transposed or swapped operand cannot give this.
    K, N = 6, 4
    B = np.arange(K * N, dtype=np.float32).reshape(K, N)
    A = np.zeros((2, K), dtype=np.float32)
    A[0, 5] = 1.0
    A[1, 2] = 1.0
    R = oracle.gemm(A, B)
    assert R.tolist() == [[20, 21, 22, 23], [8, 9, 10, 11]]


def test_rank1_closed_form(oracle):
    # A[i][k] = u_i x_k, B[k][j] = y_k v_j  =>  C[i][j] = u_i v_j (x . y)
    M, K, N = 19, 23, 17
    r = _rng(5)
    u, x = r.integers(-3, 4, M), r.integers(-3, 4, K)
    y, v = r.integers(-3, 4, K), r.integers(-3, 4, N)
    A = np.outer(u, x).astype(np.float32)
    B = np.outer(y, v).astype(np.float32)
    dot = int(np.dot(x, y))
    expect = np.outer(u, v).astype(np.int64) * dot
    R = oracle.gemm(A, B)
    assert np.array_equal(R, expect.astype(np.float64))


def test_alpha_beta_conventions(oracle):
    M, K, N = 9, 7, 5
    A = gi.draw("integer", 21, 0, (M, K))
    B = gi.draw("integer", 21, 1, (K, N))
    C = gi.draw("integer", 21, 2, (M, N))
    # alpha = 0: A and B are not read (NaN operands must not leak)
    nanA = np.full((M, K), np.nan, np.float32)
    nanB = np.full((K, N), np.nan, np.float32)
    assert np.array_equal(oracle.gemm(nanA, nanB, C, alpha=0.0, beta=1.0),
                          C.astype(np.float64))
    assert np.array_equal(oracle.gemm(nanA, nanB, C, alpha=0.0, beta=0.0),
                          np.zeros((M, N)))
    # beta = 0: C is not read
    nanC = np.full((M, N), np.nan, np.float32)
    R = oracle.gemm(A, B, nanC, alpha=1.0, beta=0.0)
    assert np.isfinite(R).all()
    # K = 0: empty sum, only beta*C remains
    R0 = oracle.gemm(np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32),
                     C, alpha=3.0, beta=-2.0)
    assert np.array_equal(R0, -2.0 * C.astype(np.float64))
    # general alpha, beta against exact integers
    Ai, Bi, Ci = A.astype(np.int64), B.astype(np.int64), C.astype(np.int64)
    expect = 2 * (Ai @ Bi) - 3 * Ci
    assert np.array_equal(oracle.gemm(A, B, C, alpha=2.0, beta=-3.0),
                          expect.astype(np.float64))
    # alpha = 0.5 gives exact half-integers
    expect_half = (Ai @ Bi).astype(np.float64) * 0.5 + Ci
    assert np.array_equal(oracle.gemm(A, B, C, alpha=0.5, beta=1.0), expect_half)


def test_alpha_zero_result_is_beta_c_including_its_sign_of_zero(oracle):
    # BLAS reading: alpha == 0 (or K == 0) gives beta*C itself, so a zero
    # of C scaled by a negative beta is -0; beta == 0 gives alpha*A*B itself,
    # so an exact zero product scaled by a negative alpha is -0.
    M, K, N = 3, 4, 2
    C = np.zeros((M, N), np.float32)
    R = oracle.gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32), C,
                    alpha=0.0, beta=-2.0)
    assert np.signbit(R).all() and (R == 0).all()
    R0 = oracle.gemm(np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), C,
                     alpha=1.0, beta=-2.0)
    assert np.signbit(R0).all()
    Z = oracle.gemm(np.zeros((M, K), np.float32), np.ones((K, N), np.float32), None,
                    alpha=-1.0, beta=0.0)
    assert np.signbit(Z).all() and (Z == 0).all()
    # both terms present: IEEE sum of (-0) + (+0) is +0
    P = oracle.gemm(np.zeros((M, K), np.float32), np.ones((K, N), np.float32), C,
                    alpha=-1.0, beta=1.0)
    assert not np.signbit(P).any()
    E = oracle.gemm_entries(np.zeros((M, K), np.float32), np.ones((K, N), np.float32),
                            np.array([0, 2]), np.array([1, 0]), C=C, alpha=0.0, beta=-3.0)
    assert np.signbit(E).all()


def _exact_product(A, B, C, alpha, beta):
    """Independent exact evaluation with Fractions, column-major loop order."""
    M, K = len(A), len(A[0]) if A else 0
    N = len(B[0]) if B else 0
    out = [[None] * N for _ in range(M)]
    for j in range(N):
        for i in range(M):
            s = sum((A[i][k] * B[k][j] for k in range(K)), Fraction(0))
            out[i][j] = alpha * s + beta * C[i][j]
    return out


def test_bruteforce_all_tiny_shapes_integer(oracle):
    for M, N, K in itertools.product(range(1, 10), repeat=3):
        seed = 1000 + 100 * M + 10 * N + K
        A = gi.draw("integer", seed, 0, (M, K))
        B = gi.draw("integer", seed, 1, (K, N))
        C = gi.draw("integer", seed, 2, (M, N))
        R = oracle.gemm(A, B, C, alpha=1.0, beta=1.0)
        Af = [[Fraction(int(v)) for v in row] for row in A]
        Bf = [[Fraction(int(v)) for v in row] for row in B]
        Cf = [[Fraction(int(v)) for v in row] for row in C]
        E = _exact_product(Af, Bf, Cf, 1, 1)
        assert R.tolist() == [[float(e) for e in row] for row in E], (M, N, K)


def test_bruteforce_tiny_shapes_random_within_double_rounding(oracle):
    for M, N, K in itertools.product((1, 2, 5, 9), repeat=3):
        seed = 5000 + 100 * M + 10 * N + K
        A = gi.draw("uniform", seed, 0, (M, K))
        B = gi.draw("uniform", seed, 1, (K, N))
        C = gi.draw("uniform", seed, 2, (M, N))
        R = oracle.gemm(A, B, C, alpha=0.75, beta=-1.25)
        Af = [[Fraction(float(v)) for v in row] for row in A]
        Bf = [[Fraction(float(v)) for v in row] for row in B]
        Cf = [[Fraction(float(v)) for v in row] for row in C]
        E = _exact_product(Af, Bf, Cf, Fraction(3, 4), Fraction(-5, 4))
        for i in range(M):
            for j in range(N):
                # K+2 roundings of double sums, each <= 2^-53 relative to a
                # partial sum bounded by sum |terms| <= K + 2.
                bound = (K + 3) * 2.0**-52 * (K + 2)
                assert abs(Fraction(R[i, j]) - E[i][j]) <= bound, (M, N, K, i, j)


def test_numpy_float64_matmul_special_case(oracle):
    M, K, N = 200, 300, 150
    A = gi.draw("uniform", 31, 0, (M, K))
    B = gi.draw("uniform", 31, 1, (K, N))
    C = gi.draw("uniform", 31, 2, (M, N))
    R = oracle.gemm(A, B, C, alpha=1.5, beta=0.25)
    ref = 1.5 * (A.astype(np.float64) @ B.astype(np.float64)) + 0.25 * C.astype(np.float64)
    assert np.max(np.abs(R - ref)) <= 1e-12 * K


def test_strided_operands_and_threads_agree(oracle):
    M, K, N = 33, 45, 27
    big = gi.draw("uniform", 41, 0, (M, K + 7))
    A = big[:, 3:3 + K]
    Bbig = gi.draw("uniform", 41, 1, (K, N + 5))
    B = Bbig[:, :N]
    R1 = oracle.gemm(A, B, threads=1)
    R8 = oracle.gemm(A, B, threads=8)
    assert np.array_equal(R1, R8)
    R = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), threads=3)
    assert np.array_equal(R, R1)


def test_entries_match_full_product(oracle):
    M, K, N = 40, 64, 50
    A = gi.draw("normal", 51, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 51, 1, (K, N), sigma=0.02, dtype="bf16")
    C = gi.draw("normal", 51, 2, (M, N), dtype="bf16")
    R = oracle.gemm(A, B, C, alpha=0.5, beta=1.0)
    rows = np.array([0, 5, 39, 17, 39])
    cols = np.array([0, 49, 0, 23, 49])
    e = oracle.gemm_entries(A, B, rows, cols, C, alpha=0.5, beta=1.0)
    assert np.array_equal(e, R[rows, cols])


def test_mixed_input_types_widen_exactly(oracle):
    # bf16 bits widen to the same double as the fp32 value they round to.
    x = gi.draw("normal", 61, 0, (16, 16))
    xb = gi.f32_to_bf16_bits(x)
    wide = oracle.widen_bf16(xb)
    assert np.array_equal(wide, gi.bf16_bits_to_f32(xb).astype(np.float64))
    R1 = oracle.gemm(xb, xb)
    R2 = oracle.gemm(gi.bf16_bits_to_f32(xb), gi.bf16_bits_to_f32(xb))
    assert np.array_equal(R1, R2)


# ---------------------------------------------------------------- rounding

def test_bf16_round_ties_to_even(oracle):
    one = 1.0
    ulp = 2.0**-7
    cases = [
        (one, 0x3F80),
        (one + ulp / 2, 0x3F80),            # tie, 1.0 has even mantissa
        (one + 3 * ulp / 2, 0x3F82),        # tie, rounds up to even
        (one + ulp / 2 + 2.0**-40, 0x3F81),  # just above the tie
        (-(one + 3 * ulp / 2), 0xBF82),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0**-133, 0x0001),                # smallest subnormal
        (1.5 * 2.0**-133, 0x0002),          # tie between 1 and 2 quanta -> even
        (0.5 * 2.0**-133, 0x0000),          # tie between 0 and 1 quantum -> 0
        (0.75 * 2.0**-133, 0x0001),
        (2.0**-126, 0x0080),                # smallest normal
        ((2 - 2.0**-7) * 2.0**127, 0x7F7F),  # largest finite
        ((2 - 2.0**-8) * 2.0**127, 0x7F80),  # midpoint to 2^128: even -> inf
        ((2 - 2.0**-8 - 2.0**-30) * 2.0**127, 0x7F7F),
        (1e300, 0x7F80),
        (-1e300, 0xFF80),
        (math.inf, 0x7F80),
        (-math.inf, 0xFF80),
        (1e-300, 0x0000),
    ]
    got = oracle.round_bf16(np.array([v for v, _ in cases], dtype=np.float64))
    assert [int(g) for g in got] == [w for _, w in cases]
    nan = oracle.round_bf16(np.array([math.nan]))[0]
    assert (int(nan) & 0x7F80) == 0x7F80 and (int(nan) & 0x7F) != 0


def test_bf16_round_matches_torch_on_fp32_values(oracle):
    torch = pytest.importorskip("torch")
    bits = _rng(7).integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ours = oracle.round_bf16(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_matches_exact_nearest_on_doubles(oracle):
    # Values with more bits than fp32: compare against exact nearest-even
    # selection among bf16 neighbours, done with Fractions.
    vals = gi.normal_f32(71, 0, 300).astype(np.float64) * (1 + 2.0**-30)
    got = oracle.round_bf16(vals)
    for v, g in zip(vals, got):
        fv = Fraction(float(v))
        e = math.frexp(abs(float(v)))[1]
        q = Fraction(2) ** (max(e - 8, -133))
        lo = (fv / q).__floor__()
        cand = [lo, lo + 1]
        best = min(cand, key=lambda c: (abs(fv - c * q), c % 2))
        want = gi.f32_to_bf16_bits(np.array([float(best * q)], np.float32))[0]
        assert int(g) == int(want)


def test_f32_round_matches_numpy(oracle):
    x = _rng(8).standard_normal(10000) * 10.0 ** _rng(9).integers(-40, 40, 10000)
    assert np.array_equal(oracle.round_f32(x), x.astype(np.float32))


# ---------------------------------------------------------------- page facts

def test_page_facts_bf16_format(oracle):
    facts = json.load(open(GOLDEN))["bf16_format"]
    assert facts["sign_bits"] + facts["exponent_bits"] + facts["mantissa_bits"] == 16
    # same exponent width as fp32: the largest finite bf16 is close to fp32 max
    largest = oracle.widen_bf16(np.array([0x7F7F], np.uint16))[0]
    assert largest == (2 - 2.0 ** -facts["mantissa_bits"]) * 2.0 ** (2 ** (facts["exponent_bits"] - 1) - 1)
    assert largest / float(np.finfo(np.float32).max) > 0.99
    # one bf16 ulp at 1.0 is 2^-mantissa_bits
    assert oracle.widen_bf16(np.array([0x3F81], np.uint16))[0] - 1.0 == 2.0 ** -facts["mantissa_bits"]


def test_page_facts_fp16_is_not_bf16(oracle):
    facts = json.load(open(GOLDEN))["fp16_max"]
    # 65504 fits in bf16's range with room to spare, but is not exact in bf16
    b = oracle.round_bf16(np.array([facts["printed_max"]], dtype=np.float64))
    assert oracle.widen_bf16(b)[0] == 65536.0


# ---------------------------------------------------------------- fused epilogue

def test_gelu_tanh_constant_is_the_printed_one(oracle):
    # "Z-Turbo" page, section 2.1 prints the constant as 0.79788456
    assert abs(math.sqrt(2 / math.pi) - 0.79788456) < 5e-9


def test_gelu_odd_part_identity_and_limits(oracle):
    x = np.linspace(-8, 8, 2001)
    g = oracle.act_values(x, oracle.ACT_GELU)
    gm = oracle.act_values(-x, oracle.ACT_GELU)
    # 0.5x(1+tanh(u)) - 0.5(-x)(1+tanh(-u)) = x for the tanh form
    assert np.max(np.abs((g - gm) - x)) < 1e-12
    assert oracle.act_values([0.0], oracle.ACT_GELU)[0] == 0.0
    big = oracle.act_values([30.0, -30.0], oracle.ACT_GELU)
    assert big[0] == 30.0 and abs(big[1]) < 1e-300 + 1e-12


def test_gelu_tanh_close_to_erf_gelu(oracle):
    # the tanh form approximates x * Phi(x) to a few 1e-4
    x = np.linspace(-6, 6, 4001)
    g = oracle.act_values(x, oracle.ACT_GELU)
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in x])
    assert np.max(np.abs(g - exact)) < 5e-4


def test_relu_and_none(oracle):
    x = np.array([-2.5, -0.0, 0.0, 1e-300, 3.0])
    assert oracle.act_values(x, oracle.ACT_RELU).tolist() == [0.0, 0.0, 0.0, 1e-300, 3.0]
    assert np.array_equal(oracle.act_values(x, oracle.ACT_NONE), x)


def test_fused_epilogue_order_bias_act_then_residual(oracle):
    M, K, N = 6, 5, 7
    A = gi.draw("integer", 91, 0, (M, K))
    B = gi.draw("integer", 91, 1, (K, N))
    C = gi.draw("integer", 91, 2, (M, N))
    bias = gi.draw("integer", 91, 3, (1, N)).reshape(-1)
    R = oracle.gemm_fused(A, B, C, alpha=0.5, beta=2.0, bias=bias, act=oracle.ACT_RELU)
    lin = 0.5 * (A.astype(np.int64) @ B.astype(np.int64)) + bias.astype(np.float64)
    expect = np.maximum(lin, 0.0) + 2.0 * C.astype(np.float64)
    assert np.array_equal(R, expect)
    # no bias, no activation: the plain GEMM
    assert np.array_equal(oracle.gemm_fused(A, B, C, alpha=0.5, beta=2.0),
                          oracle.gemm(A, B, C, alpha=0.5, beta=2.0))
    # bf16 bias widens exactly
    bb = gi.f32_to_bf16_bits(bias.astype(np.float32))
    assert np.array_equal(oracle.gemm_fused(A, B, bias=bb), oracle.gemm_fused(A, B, bias=bias))


# The tanh-form GELU the "Z-Turbo" page prints in its section 2.1,
# 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), evaluated here in 40-digit
# decimal arithmetic from nothing but that formula: pi from Machin's
# arctangent series, tanh from exp.  These values tell the tanh form apart
# from the erf form x * Phi(x) (at x = 1 they differ by 1.5e-4, at x = 2 by
# 1e-4), which the identity and closeness pins above cannot.
def _gelu_tanh_decimal(x):
    from decimal import Decimal, localcontext

    with localcontext() as ctx:
        ctx.prec = 40

        def atan_inv(n):  # arctan(1/n) by its Taylor series
            n = Decimal(n)
            term = total = 1 / n
            k, sign, n2 = 1, -1, n * n
            while True:
                term /= n2
                nxt = total + sign * term / (2 * k + 1)
                if nxt == total:
                    return total
                total, k, sign = nxt, k + 1, -sign

        pi = 16 * atan_inv(5) - 4 * atan_inv(239)
        xd = Decimal(repr(float(x)))
        u = (2 / pi).sqrt() * (xd + Decimal("0.044715") * xd ** 3)
        e = (2 * u).exp()
        return float(Decimal("0.5") * xd * (1 + (e - 1) / (e + 1)))


def test_gelu_is_the_printed_tanh_form_not_the_erf_form(oracle):
    xs = [1.0, 2.0, -1.0, -2.0, 0.5, 3.0, -0.25, 1.5]
    got = oracle.act_values(xs, oracle.ACT_GELU)
    for x, g in zip(xs, got):
        want = _gelu_tanh_decimal(x)
        assert abs(g - want) <= 1e-13 * max(1.0, abs(want)), (x, g, want)
    # hand-checked values at 1 and 2 (tanh form), and the erf form's values,
    # which must fail the comparison above
    assert abs(_gelu_tanh_decimal(1.0) - 0.8411919906082768) < 1e-15
    assert abs(_gelu_tanh_decimal(2.0) - 1.954597694087775) < 1e-14
    for x, erf_form in [(1.0, 0.8413447460685429), (2.0, 1.9544997361036416)]:
        assert abs(erf_form - 0.5 * x * (1 + math.erf(x / math.sqrt(2)))) < 1e-15
        assert abs(erf_form - _gelu_tanh_decimal(x)) > 1e-5
