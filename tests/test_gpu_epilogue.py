"""GPU parity of the extended entry points: transposed operand layouts and
the fused epilogue C = act(alpha * op(A) * op(B) + bias) + beta * C,
against the oracle (oracle.gemm_fused) on the same seeded inputs.

* integer-valued operands, bias and C with ReLU (or no activation): every
  step is exact in fp32 in any order, so results match bit for bit on every
  kernel path (1-CTA tiles of 128 and 256 columns, CTA pairs, split-K, the
  generic SIMT kernel, the FP32 TMA kernel) and for all four layouts;
* GELU (tanh form): the activation alone checked against the oracle's
  double-precision GELU to within fp32 evaluation error, then whole GEMMs
  with normal inputs within the BF16 tolerance |C - C_ref| <= 2^-7 |C_ref|
  + 1e-2 (FP32 path: max |C - C_ref| <= 1.2e-5 K + 2e-6 |C_ref|);
* opts NULL / all-zero reproduce the plain entry points exactly; alpha == 0
  gives act(bias) + beta * C without reading A or B.
"""

import contextlib

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
from gpu_helpers import (GuardedC, bf16_to_dev, bf16_tolerance_violations, f32_to_dev,
                         widen)

pytestmark = pytest.mark.gpu

B_ = g.binding
TRANS = [(0, 0), (1, 0), (0, 1), (1, 1)]


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


def _status_ok():
    B_.check(B_.get_device_status(), "device status")


def put(X, trans, pad, dtype):
    """Logical operand X (rows x cols) on the device in the stored layout:
    row-major with pitch cols + pad, or (trans) stored transposed, cols x
    rows with pitch rows + pad, returned as the logical (transposed) view."""
    up = bf16_to_dev if dtype == "bf16" else f32_to_dev
    if trans:
        st = np.ascontiguousarray(X.T)
        return up(st, st.shape[1] + pad).t()
    return up(X, X.shape[1] + pad)


def tma_pad(n, dtype):
    """Padding that makes a row of n elements a multiple of 16 bytes."""
    q = 8 if dtype == "bf16" else 4
    return (-n) % q


def run_ex(A, B, Cin, alpha, beta, bias, act, out, ta, tb, pads=None, ldc=None, dtype="bf16"):
    """One gemm_ex call through the tensor API; A, B logical numpy operands."""
    M, K = A.shape
    N = B.shape[1]
    if pads is None:  # TMA-able pitches for the stored layout
        pads = (tma_pad(M if ta else K, dtype), tma_pad(K if tb else N, dtype))
    dA, dB = put(A, ta, pads[0], dtype), put(B, tb, pads[1], dtype)
    if Cin is None:
        init = (np.full((M, N), 0x7FC0, np.uint16) if out == "bf16"
                else np.full((M, N), np.nan, np.float32))
    else:
        init = Cin
    C = GuardedC(M, N, ldc or N, out, init)
    dbias = None
    if bias is not None:
        dbias = (torch.from_numpy(bias.view(np.int16)).cuda().view(torch.bfloat16)
                 if bias.dtype == np.uint16 else torch.from_numpy(bias).cuda())
    g.gemm_ex(dA, dB, C.view, alpha=alpha, beta=beta, bias=dbias, act=act)
    torch.cuda.synchronize()
    _status_ok()
    return C


def integer_case(seed, M, N, K, out, bias_dtype="f32", dtype="bf16"):
    A = gi.draw("integer", seed, 0, (M, K), dtype=dtype)
    B = gi.draw("integer", seed, 1, (K, N), dtype=dtype)
    Cin = gi.draw("integer", seed, 2, (M, N), dtype=out)
    bias = gi.draw("integer", seed, 3, (N,), dtype=bias_dtype)
    return A, B, Cin, bias


def ref_round(R, out):
    return oracle.round_bf16(R) if out == "bf16" else oracle.round_f32(R)


# --------------------------------------------------------------- BF16 paths

PATHS = {
    "tile256": dict(cta_pair=1, bf16_tile_n=256),
    "tile128": dict(cta_pair=1, bf16_tile_n=128),
    "pair": dict(cta_pair=2),
    "split_k3": dict(cta_pair=1, split_k=3),
}
SHAPES = [(129, 264, 1000), (257, 1000, 72), (300, 520, 776), (7, 72, 1000)]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_bf16_layouts_bias_relu_integer_bit_exact(M, N, K, ta, tb, path):
    out = "bf16" if (M + N) % 2 else "f32"
    seed = 9100 + M * 3 + N * 5 + K + 17 * ta + 31 * tb
    A, B, Cin, bias = integer_case(seed, M, N, K, out, bias_dtype="bf16" if K % 2 else "f32")
    with config(**PATHS[path]):
        C = run_ex(A, B, Cin, 0.5, -1.0, bias, "relu", out, ta, tb)
    assert B_.last_kernel() == "bf16_tcgen05"
    R = oracle.gemm_fused(A, B, Cin, alpha=0.5, beta=-1.0, bias=bias, act=oracle.ACT_RELU)
    got, ref = C.result(), ref_round(R, out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("ldc_pad", [0, 3])
def test_bf16_layouts_auto_path_and_c_store_modes(ta, tb, ldc_pad):
    # ldc_pad 0: C rows 16-byte aligned, stored by TMA; 3: direct stores.
    M, N, K = 1000, 1288, 520
    seed = 9200 + ta * 2 + tb + ldc_pad
    A, B, Cin, bias = integer_case(seed, M, N, K, "bf16")
    C = run_ex(A, B, Cin, 1.0, 1.0, bias, "none", "bf16", ta, tb, ldc=N + ldc_pad)
    assert B_.last_kernel() == "bf16_tcgen05"
    R = oracle.gemm_fused(A, B, Cin, alpha=1.0, beta=1.0, bias=bias)
    got, ref = C.result(), ref_round(R, "bf16")
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} mismatches"
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("pads", [(3, 5), (1, 0), (0, 1)])
def test_bf16_layouts_generic_kernel_integer(ta, tb, pads):
    # Pitches that TMA cannot fetch take the generic SIMT kernel.
    M, N, K = 65, 127, 200
    seed = 9300 + ta * 2 + tb + 7 * sum(pads)
    A, B, Cin, bias = integer_case(seed, M, N, K, "f32")
    pa = pads[0] + tma_pad(M if ta else K, "bf16")
    pb = pads[1] + tma_pad(K if tb else N, "bf16")
    C = run_ex(A, B, Cin, 2.0, 0.5, bias, "relu", "f32", ta, tb, pads=(pa, pb))
    tma = (pads[0] == 0 and pads[1] == 0)
    assert B_.last_kernel() == ("bf16_tcgen05" if tma else "bf16_simt")
    R = oracle.gemm_fused(A, B, Cin, alpha=2.0, beta=0.5, bias=bias, act=oracle.ACT_RELU)
    assert np.array_equal(C.result(), ref_round(R, "f32"))
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_layouts_gelu_normal_within_tolerance(ta, tb, out):
    M, N, K = 383, 1288, 1032
    seed = 9400 + ta * 2 + tb
    A = gi.draw("normal", seed, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", seed, 1, (K, N), sigma=1.0 / 32, dtype="bf16")
    Cin = gi.draw("normal", seed, 2, (M, N), dtype=out)
    bias = gi.draw("normal", seed, 3, (N,))
    C = run_ex(A, B, Cin, 1.0, 1.0, bias, "gelu", out, ta, tb)
    R = oracle.gemm_fused(A, B, Cin, alpha=1.0, beta=1.0, bias=bias, act=oracle.ACT_GELU)
    assert bf16_tolerance_violations(widen(C.result(), out), R) == 0
    assert C.guards_intact()


def test_bf16_gelu_on_the_decode_shape_split_k():
    # 64 x 8192 x 8192 runs split-K: the epilogue sits in the reduction.
    M, N, K = 64, 8192, 8192
    A = gi.draw("normal", 9450, 0, (M, K), dtype="bf16")
    B = gi.draw("normal", 9450, 1, (K, N), sigma=1.0 / 64, dtype="bf16")
    bias = gi.draw("normal", 9450, 3, (N,), dtype="bf16")
    C = run_ex(A, B, None, 1.0, 0.0, bias, "gelu", "f32", 0, 1)
    R = oracle.gemm_fused(A, B, None, bias=bias, act=oracle.ACT_GELU)
    assert bf16_tolerance_violations(widen(C.result(), "f32"), R) == 0


# ------------------------------------------------------------ activations

def _gelu_probe_values():
    x = np.concatenate([np.linspace(-10.0, 10.0, 2001), [0.0, -0.0, 1e-30, -1e-30, 3.5, -3.5],
                        gi.draw("normal", 9500, 0, (1017,), sigma=3.0).astype(np.float64)])
    return x.astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gelu_activation_against_double(dtype):
    # K = 8, A = e_1 rows, B row 0 = x: every output is exactly act(x) of
    # one probe value, so this isolates the activation.  N = 3024 (a
    # multiple of 8): the bf16 case runs on the tcgen05 kernel.
    x = _gelu_probe_values()
    if dtype == "bf16":
        xb = gi.f32_to_bf16_bits(x)
        x = gi.bf16_bits_to_f32(xb)
    N, K, M = x.size, 8, 4
    A = np.zeros((M, K), np.float32)
    A[:, 0] = 1.0
    Bm = np.zeros((K, N), np.float32)
    Bm[0] = x
    if dtype == "bf16":
        A, Bm = gi.f32_to_bf16_bits(A), gi.f32_to_bf16_bits(Bm)
    C = run_ex(A, Bm, None, 1.0, 0.0, None, "gelu", "f32", 0, 0, dtype=dtype)
    want = oracle.act_values(x.astype(np.float64), oracle.ACT_GELU)
    got = C.result().astype(np.float64)
    tol = 1e-6 * np.abs(want) + 2.0**-22 * np.abs(x.astype(np.float64)) + 1e-30
    for r in range(M):
        err = np.abs(got[r] - want)
        assert (err <= tol).all(), f"max excess {float((err - tol).max())}"


def test_relu_activation_signs_exact():
    x = np.array([-3.0, -0.0, 0.0, 1e-38, -1e-38, 2.5, -2.5, 65504.0], np.float32)
    N, K, M = x.size, 4, 2
    A = np.zeros((M, K), np.float32)
    A[:, 0] = 1.0
    Bm = np.zeros((K, N), np.float32)
    Bm[0] = x
    C = run_ex(A, Bm, None, 1.0, 0.0, None, "relu", "f32", 0, 0, dtype="f32")
    want = oracle.round_f32(oracle.act_values(x.astype(np.float64), oracle.ACT_RELU))
    got = C.result()
    assert np.array_equal(got.view(np.uint32), np.broadcast_to(want, got.shape).view(np.uint32))


# --------------------------------------------------------------- FP32 paths

@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", [(129, 264, 1000), (65, 127, 200), (300, 520, 776)])
def test_f32_layouts_bias_relu_integer_bit_exact(M, N, K, ta, tb):
    seed = 9600 + M + N + K + 17 * ta + 31 * tb
    A, B, Cin, bias = integer_case(seed, M, N, K, "f32", dtype="f32",
                                   bias_dtype="bf16" if ta else "f32")
    C = run_ex(A, B, Cin, 1.0, -1.0, bias, "relu", "f32", ta, tb, dtype="f32")
    # run_ex pads the pitches to multiples of 16 bytes: row-major operands
    # take the TMA kernel, transposed ones the generic kernel.
    assert B_.last_kernel() == ("sgemm_tma" if not ta and not tb else "f32_simt")
    R = oracle.gemm_fused(A, B, Cin, alpha=1.0, beta=-1.0, bias=bias, act=oracle.ACT_RELU)
    assert np.array_equal(C.result(), oracle.round_f32(R))
    assert C.guards_intact()


@pytest.mark.parametrize("ta,tb", TRANS)
def test_f32_layouts_gelu_uniform_within_tolerance(ta, tb):
    M, N, K = 300, 520, 776
    seed = 9700 + 2 * ta + tb
    A = gi.draw("uniform", seed, 0, (M, K))
    B = gi.draw("uniform", seed, 1, (K, N))
    Cin = gi.draw("uniform", seed, 2, (M, N))
    bias = gi.draw("uniform", seed, 3, (N,))
    C = run_ex(A, B, Cin, 1.0 / 64, 0.5, bias, "gelu", "f32", ta, tb, dtype="f32")
    R = oracle.gemm_fused(A, B, Cin, alpha=1.0 / 64, beta=0.5, bias=bias, act=oracle.ACT_GELU)
    err = np.abs(C.result().astype(np.float64) - R)
    assert (err <= 1.2e-5 * K + 2e-6 * np.abs(R)).all()


# ------------------------------------------------------- special cases

def _raw_bf16_ex(A, B, C, M, N, K, alpha, beta, opts, c_type):
    return B_.gemm_bf16_ex(M, N, K, alpha, A.data_ptr() if A is not None else None,
                           A.stride(0) if A is not None else max(1, K),
                           B.data_ptr() if B is not None else None,
                           B.stride(0) if B is not None else max(1, N), beta, C.data_ptr(),
                           C.stride(0), c_type, opts,
                           int(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("opts_kind", ["null", "zero"])
def test_ex_without_options_reproduces_plain_entry_point(opts_kind):
    M, N, K = 1000, 1288, 520
    A = bf16_to_dev(gi.draw("normal", 9800, 0, (M, K), dtype="bf16"))
    Bd = bf16_to_dev(gi.draw("normal", 9800, 1, (K, N), dtype="bf16"))
    C1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C2 = torch.empty_like(C1)
    g.gemm_bf16(A, Bd, C1, out_dtype=torch.float32)
    opts = None if opts_kind == "null" else B_.make_opts()
    B_.check(_raw_bf16_ex(A, Bd, C2, M, N, K, 1.0, 0.0, opts, B_.GEMM_OUT_F32), "gemm_bf16_ex")
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_alpha_zero_gives_activation_of_bias_plus_beta_c(out):
    M, N, K = 33, 48, 64
    Cin = gi.draw("integer", 9900, 2, (M, N), dtype=out)
    bias = gi.draw("integer", 9900, 3, (N,))
    # A and B hold NaN: with alpha == 0 they must not be read.
    A = np.full((M, K), 0x7FC0, np.uint16)
    Bm = np.full((K, N), 0x7FC0, np.uint16)
    C = run_ex(A, Bm, Cin, 0.0, 2.0, bias, "relu", out, 0, 0)
    assert B_.last_kernel() == "bf16_simt"
    Z = np.zeros((M, K), np.uint16)
    R = oracle.gemm_fused(Z, np.zeros((K, N), np.uint16), Cin, alpha=0.0, beta=2.0, bias=bias,
                          act=oracle.ACT_RELU)
    assert np.array_equal(C.result(), ref_round(R, out))
    assert C.guards_intact()


def test_k_zero_with_bias_and_null_operands():
    M, N = 17, 40
    bias = gi.draw("integer", 9950, 3, (N,))
    Cin = gi.draw("integer", 9950, 2, (M, N))
    dbias = torch.from_numpy(bias).cuda()
    C = torch.from_numpy(Cin).cuda()
    opts = B_.make_opts(bias=dbias.data_ptr(), bias_type=B_.GEMM_OUT_F32, act=B_.GEMM_ACT_RELU)
    rc = B_.gemm_f32_ex(M, N, 0, 1.0, None, 1, None, N, 1.0, C.data_ptr(), N, opts,
                        int(torch.cuda.current_stream().cuda_stream))
    B_.check(rc, "gemm_f32_ex")
    torch.cuda.synchronize()
    assert B_.last_kernel() == "f32_simt"
    R = oracle.gemm_fused(np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), Cin,
                          alpha=1.0, beta=1.0, bias=bias, act=oracle.ACT_RELU)
    assert np.array_equal(C.cpu().numpy(), oracle.round_f32(R))
