"""GPU parity of the strided batched GEMMs (gemm_bf16_batched,
gemm_f32_batched): every matrix of the batch against the oracle on the same
seeded inputs.

* integer-valued operands, bias and C: bit-exact on every kernel path (CTA
  pairs, 1-CTA tiles of 128 and 256 columns, split-K, stream-K, the TMA
  SGEMM with its K split, the generic kernels), for contiguous batches,
  batch strides with gaps, operands shared by the whole batch (stride 0)
  and transposed layouts;
* normal inputs within the BF16 tolerance; guard sentinels after the last
  C matrix and in the gaps between C matrices must survive.
"""

import contextlib

import numpy as np
import pytest
import torch

import dense_gemm_02_gb300 as g
import gemm_inputs as gi
import oracle
from gpu_helpers import SENTINEL_BF16, SENTINEL_F32, bf16_tolerance_violations

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


def to_dev(mats, trans, gap, dtype, shared=False):
    """Logical matrices (list of rows x cols numpy arrays) stored on the
    device as a strided batch: each matrix row-major (or, with trans, its
    transpose row-major), `gap` spare elements between matrices.  Returns
    (3-D logical view, element stride between matrices)."""
    st = [np.ascontiguousarray(m.T if trans else m) for m in mats]
    r, c = st[0].shape
    span = r * c
    stride = 0 if shared else span + gap
    n = 1 if shared else len(st)
    tdt = torch.int16 if dtype == "bf16" else torch.float32
    buf = torch.zeros(max(1, (n - 1) * stride + span), dtype=tdt, device="cuda")
    for i in range(n):
        src = st[i].view(np.int16) if dtype == "bf16" else st[i]
        buf[i * stride:i * stride + span] = torch.from_numpy(src.reshape(-1)).cuda()
    if dtype == "bf16":
        buf = buf.view(torch.bfloat16)
    v = torch.as_strided(buf, (len(mats), r, c), (stride, c, 1))
    return (v.transpose(1, 2) if trans else v), stride


class GuardedBatch:
    """C matrices (M x N, contiguous rows) `gap` elements apart in a buffer
    whose gaps and tail hold a sentinel."""

    def __init__(self, inits, gap, out):
        self.out, self.gap = out, gap
        self.n = len(inits)
        self.M, self.N = inits[0].shape
        self.span = self.M * self.N
        self.stride = self.span + gap
        total = self.n * self.stride + 64
        if out == "bf16":
            self.buf = torch.full((total,), SENTINEL_BF16, dtype=torch.int16, device="cuda")
        else:
            self.buf = torch.full((total,), float(SENTINEL_F32), dtype=torch.float32,
                                  device="cuda")
        for i, m in enumerate(inits):
            src = m.view(np.int16) if out == "bf16" else m
            self.buf[i * self.stride:i * self.stride + self.span] = torch.from_numpy(
                np.ascontiguousarray(src).reshape(-1)).cuda()
        base = self.buf.view(torch.bfloat16) if out == "bf16" else self.buf
        self.view = torch.as_strided(base, (self.n, self.M, self.N), (self.stride, self.N, 1))

    def results(self):
        b = self.buf.cpu().numpy()
        if self.out == "bf16":
            b = b.view(np.uint16)
        return [b[i * self.stride:i * self.stride + self.span].reshape(self.M, self.N)
                for i in range(self.n)]

    def guards_intact(self):
        b = self.buf.cpu().numpy()
        s = SENTINEL_BF16 if self.out == "bf16" else SENTINEL_F32
        if self.out == "bf16":
            b = b.view(np.uint16)
        ok = (b[self.n * self.stride:] == s).all()
        for i in range(self.n):
            ok &= (b[i * self.stride + self.span:(i + 1) * self.stride] == s).all()
        return bool(ok)


def run_batch(As, Bs, Cins, alpha, beta, out, dtype="bf16", ta=0, tb=0, gaps=(0, 0, 0),
              share=(False, False), bias=None, act="none"):
    dA, _ = to_dev(As, ta, gaps[0], dtype, shared=share[0])
    dB, _ = to_dev(Bs, tb, gaps[1], dtype, shared=share[1])
    M, N = As[0].shape[0], Bs[0].shape[1]
    inits = Cins if Cins is not None else [
        np.full((M, N), 0x7FC0, np.uint16) if out == "bf16" else
        np.full((M, N), np.nan, np.float32) for _ in As]
    C = GuardedBatch(inits, gaps[2], out)
    dbias = None
    if bias is not None:
        dbias = (torch.from_numpy(bias.view(np.int16)).cuda().view(torch.bfloat16)
                 if bias.dtype == np.uint16 else torch.from_numpy(bias).cuda())
    g.gemm_batched(dA, dB, C.view, alpha=alpha, beta=beta, bias=dbias, act=act)
    torch.cuda.synchronize()
    B_.check(B_.get_device_status(), "device status")
    return C


def integer_batch(seed, n, M, N, K, out, dtype="bf16", share=(False, False)):
    As = [gi.draw("integer", seed + 31 * i, 0, (M, K), dtype=dtype) for i in range(n)]
    Bs = [gi.draw("integer", seed + 31 * i, 1, (K, N), dtype=dtype) for i in range(n)]
    if share[0]:
        As = [As[0]] * n
    if share[1]:
        Bs = [Bs[0]] * n
    Cs = [gi.draw("integer", seed + 31 * i, 2, (M, N), dtype=out) for i in range(n)]
    return As, Bs, Cs


def ref_round(R, out):
    return oracle.round_bf16(R) if out == "bf16" else oracle.round_f32(R)


def check_all(C, As, Bs, Cins, alpha, beta, out, bias=None, act=oracle.ACT_NONE):
    for i, got in enumerate(C.results()):
        R = oracle.gemm_fused(As[i], Bs[i], Cins[i] if Cins is not None else None, alpha=alpha,
                              beta=beta, bias=bias, act=act)
        ref = ref_round(R, out)
        assert np.array_equal(got, ref), f"matrix {i}: {int((got != ref).sum())} mismatches"
    assert C.guards_intact()


# --------------------------------------------------------------- BF16

PATHS = {
    "auto": {},
    "pair": dict(cta_pair=2),
    "tile256": dict(cta_pair=1, bf16_tile_n=256),
    "tile128": dict(cta_pair=1, bf16_tile_n=128),
    "split_k3": dict(cta_pair=1, split_k=3),
}


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("n,M,N,K", [(3, 129, 264, 1000), (2, 300, 520, 776), (5, 7, 72, 200)])
def test_bf16_batched_integer_bit_exact(n, M, N, K, path):
    out = "f32" if M % 2 else "bf16"
    seed = 12000 + n + M + N + K
    As, Bs, Cs = integer_batch(seed, n, M, N, K, out)
    with config(**PATHS[path]):
        C = run_batch(As, Bs, Cs, 0.5, -1.0, out)
    assert B_.last_kernel() == "bf16_tcgen05"
    check_all(C, As, Bs, Cs, 0.5, -1.0, out)


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("share", [(False, False), (True, False), (False, True)])
def test_bf16_batched_layouts_gaps_and_shared_operands(ta, tb, share):
    n, M, N, K = 4, 200, 264, 328
    seed = 12100 + 2 * ta + tb + 7 * share[0] + 13 * share[1]
    As, Bs, Cs = integer_batch(seed, n, M, N, K, "bf16", share=share)
    bias = gi.draw("integer", seed, 3, (N,))
    # gaps keep every batch stride a multiple of 16 bytes (TMA path)
    C = run_batch(As, Bs, Cs, 1.0, 1.0, "bf16", ta=ta, tb=tb, gaps=(64, 128, 8), share=share,
                  bias=bias, act="relu")
    assert B_.last_kernel() == "bf16_tcgen05"
    check_all(C, As, Bs, Cs, 1.0, 1.0, "bf16", bias=bias, act=oracle.ACT_RELU)


@pytest.mark.parametrize("gaps", [(3, 0, 0), (0, 5, 0), (0, 0, 3)])
def test_bf16_batched_odd_strides(gaps):
    # A or B batch strides that are not multiples of 16 bytes take the
    # generic kernel; an odd C stride keeps the tensor cores but stores C
    # directly.
    n, M, N, K = 3, 65, 136, 200
    seed = 12200 + sum(gaps)
    As, Bs, Cs = integer_batch(seed, n, M, N, K, "bf16")
    C = run_batch(As, Bs, Cs, 2.0, 0.5, "bf16", gaps=gaps)
    want = "bf16_simt" if (gaps[0] or gaps[1]) else "bf16_tcgen05"
    assert B_.last_kernel() == want
    check_all(C, As, Bs, Cs, 2.0, 0.5, "bf16")


@pytest.mark.parametrize("stream_k", [0, 1])
def test_bf16_batched_small_m_long_k(stream_k):
    # Few tiles per matrix and a long K: split K (or stream-K) over the
    # whole batch.
    n, M, N, K = 3, 64, 512, 4096
    As, Bs, Cs = integer_batch(12300, n, M, N, K, "f32")
    with config(stream_k=stream_k):
        C = run_batch(As, Bs, Cs, 1.0, 1.0, "f32")
    assert B_.last_kernel() == "bf16_tcgen05"
    check_all(C, As, Bs, Cs, 1.0, 1.0, "f32")


def test_bf16_batched_normal_tolerance():
    n, M, N, K = 6, 512, 768, 1024
    As = [gi.draw("normal", 12400 + i, 0, (M, K), dtype="bf16") for i in range(n)]
    Bs = [gi.draw("normal", 12400 + i, 1, (K, N), dtype="bf16") for i in range(n)]
    C = run_batch(As, Bs, None, 1.0, 0.0, "bf16")
    for i, got in enumerate(C.results()):
        ref = oracle.gemm(As[i], Bs[i])
        assert bf16_tolerance_violations(gi.bf16_bits_to_f32(got).astype(np.float64), ref) == 0
    assert C.guards_intact()


def test_bf16_batched_alpha_zero_scales_every_c():
    n, M, N, K = 4, 33, 48, 64
    As = [np.full((M, K), 0x7FC0, np.uint16)] * n  # NaN: must not be read
    Bs = [np.full((K, N), 0x7FC0, np.uint16)] * n
    Cs = [gi.draw("integer", 12500 + i, 2, (M, N), dtype="bf16") for i in range(n)]
    C = run_batch(As, Bs, Cs, 0.0, -2.0, "bf16", gaps=(0, 0, 16))
    assert B_.last_kernel() == "scale_c"
    Z = [np.zeros((M, K), np.uint16)] * n
    check_all(C, Z, [np.zeros((K, N), np.uint16)] * n, Cs, 0.0, -2.0, "bf16")


def test_batch_of_one_matches_the_single_call():
    M, N, K = 300, 520, 776
    A = gi.draw("normal", 12600, 0, (M, K), dtype="bf16")
    Bm = gi.draw("normal", 12600, 1, (K, N), dtype="bf16")
    C1 = run_batch([A], [Bm], None, 1.0, 0.0, "f32")
    dA = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
    dB = torch.from_numpy(Bm.view(np.int16)).cuda().view(torch.bfloat16)
    C2 = g.gemm_bf16(dA, dB, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(C1.results()[0].view(np.uint32), C2.cpu().numpy().view(np.uint32))


# --------------------------------------------------------------- FP32

@pytest.mark.parametrize("n,M,N,K", [(3, 129, 264, 1000), (4, 1000, 1000, 136), (2, 65, 127, 200)])
def test_f32_batched_tma_integer_bit_exact(n, M, N, K):
    seed = 12700 + n + M + N + K
    As, Bs, Cs = integer_batch(seed, n, M, N, K, "f32", dtype="f32")
    # K, N padding gaps keep the strides multiples of 16 bytes
    C = run_batch(As, Bs, Cs, 1.0, -1.0, "f32", dtype="f32",
                  gaps=((-M * K) % 4, (-K * N) % 4, 0))
    want = "sgemm_tma" if (K % 4 == 0 and N % 4 == 0) else "f32_simt"
    assert B_.last_kernel() == want
    check_all(C, As, Bs, Cs, 1.0, -1.0, "f32")


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1)])
def test_f32_batched_transposed_generic(ta, tb):
    n, M, N, K = 3, 100, 72, 96
    As, Bs, Cs = integer_batch(12800 + ta, n, M, N, K, "f32", dtype="f32")
    bias = gi.draw("integer", 12800, 3, (N,))
    C = run_batch(As, Bs, Cs, 0.5, 1.0, "f32", dtype="f32", ta=ta, tb=tb, bias=bias, act="relu")
    assert B_.last_kernel() == "f32_simt"
    check_all(C, As, Bs, Cs, 0.5, 1.0, "f32", bias=bias, act=oracle.ACT_RELU)


def test_f32_batched_uniform_tolerance_shared_b():
    n, M, N, K = 5, 512, 512, 1024
    As = [gi.draw("uniform", 12900 + i, 0, (M, K)) for i in range(n)]
    Bs = [gi.draw("uniform", 12900, 1, (K, N))] * n
    C = run_batch(As, Bs, None, 1.0, 0.0, "f32", dtype="f32", share=(False, True))
    assert B_.last_kernel() == "sgemm_tma"
    for i, got in enumerate(C.results()):
        assert np.abs(got.astype(np.float64) - oracle.gemm(As[i], Bs[i])).max() <= 1e-5 * K
    assert C.guards_intact()
