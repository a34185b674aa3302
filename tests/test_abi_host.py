"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function the public header declares, and rejects bad
arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_02_gb300 import _build, binding

    _build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:GEMM_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(gemm_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("gemm_f32", "gemm_bf16", "gemm_get_device_status", "gemm_status_string",
                 "gemm_set_config", "gemm_shutdown"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from dense_gemm_02_gb300 import binding

    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"
        assert name in binding.SIGNATURES, f"{name} has no binding signature"


def test_only_declared_symbols_are_exported(lib):
    # The library is built with hidden visibility; its dynamic symbol table
    # should hold the C ABI and nothing else of ours.
    import subprocess

    from dense_gemm_02_gb300 import _build

    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    ours = {ln.split()[-1] for ln in out.stdout.splitlines() if " T gemm_" in ln}
    assert ours == set(declared_functions())


def test_release_and_debug_builds_report_their_variant(lib):
    """The debug build (GEMM_DEBUG=1) builds from the same sources, exports
    the same C ABI and says it is the debug build; the release build says it
    is not.  Loading needs no GPU."""
    from dense_gemm_02_gb300 import _build, binding

    assert lib.gemm_debug_checks() == 0
    assert not binding.debug_build_requested() or binding.library_path() == _build.DEBUG_LIB_PATH
    path = _build.build(debug=True)
    assert path == _build.DEBUG_LIB_PATH and path != _build.LIB_PATH
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), f"{name} declared but not exported by the debug build"
    dbg.gemm_debug_checks.restype = ctypes.c_int
    assert dbg.gemm_debug_checks() == 1
    dbg.gemm_status_string.restype = ctypes.c_char_p
    assert dbg.gemm_status_string(-10).decode().startswith("GEMM_ERR_DEVICE_CHECK")


def test_status_strings_and_version(lib):
    from dense_gemm_02_gb300 import binding as b

    assert b.abi_version() == 2
    for code in range(-8, 1):
        assert b.status_string(code).startswith("GEMM_")
    assert "unknown" in b.status_string(42)


def test_argument_errors_are_reported_before_any_cuda_call(lib):
    from dense_gemm_02_gb300 import binding as b

    f = b.gemm_f32
    fake = 1 << 20  # never dereferenced: every call below fails validation
    assert f(-1, 4, 4, 1.0, fake, 4, fake, 4, 0.0, fake, 4, None) == b.GEMM_ERR_INVALID_ARG
    assert f(4, 4, 4, 1.0, fake, 3, fake, 4, 0.0, fake, 4, None) == b.GEMM_ERR_BAD_LD
    assert f(4, 4, 4, 1.0, fake, 4, fake, 3, 0.0, fake, 4, None) == b.GEMM_ERR_BAD_LD
    assert f(4, 4, 4, 1.0, fake, 4, fake, 4, 0.0, fake, 3, None) == b.GEMM_ERR_BAD_LD
    assert f(4, 4, 4, 1.0, None, 4, fake, 4, 0.0, fake + 4096, 4, None) == b.GEMM_ERR_NULLPTR
    assert f(4, 4, 4, 1.0, fake, 4, fake + 4096, 4, 0.0, None, 4, None) == b.GEMM_ERR_NULLPTR
    assert f(1 << 31, 4, 4, 1.0, fake, 4, fake, 4, 0.0, fake, 4, None) == b.GEMM_ERR_TOO_LARGE
    # C overlapping A or B
    assert f(4, 4, 4, 1.0, fake, 4, fake + 4096, 4, 0.0, fake + 16, 4, None) == b.GEMM_ERR_ALIAS
    assert f(4, 4, 4, 1.0, fake, 4, fake + 4096, 4, 0.0, fake + 4096 + 60, 4,
             None) == b.GEMM_ERR_ALIAS
    # empty problems are a no-op with no pointer needed
    assert f(0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, None) == b.GEMM_OK
    assert f(4, 0, 4, 1.0, None, 4, None, 1, 0.0, None, 1, None) == b.GEMM_OK
    g = b.gemm_bf16
    assert g(4, 4, 4, 1.0, fake, 4, fake, 4, 0.0, fake, 4, 7, None) == b.GEMM_ERR_INVALID_ARG
    assert g(4, 4, 4, 1.0, fake, 2, fake, 4, 0.0, fake, 4, 0, None) == b.GEMM_ERR_BAD_LD
    assert g(4, 4, 4, 1.0, fake, 4, fake + 4096, 4, 0.0, fake + 8, 4, 1,
             None) == b.GEMM_ERR_ALIAS


def test_extended_entry_point_errors(lib):
    """gemm_bf16_ex / gemm_f32_ex: option and layout checks run before any
    CUDA call (the stored shapes of transposed operands set the pitch
    minimums, and the bias may not overlap C)."""
    from dense_gemm_02_gb300 import binding as b

    fake = 1 << 20
    for f, extra in ((b.gemm_bf16_ex, (b.GEMM_OUT_F32,)), (b.gemm_f32_ex, ())):
        def call(M, N, K, lda, ldb, ldc, opts, A=fake, B=fake + 65536, C=fake + 131072):
            return f(M, N, K, 1.0, A, lda, B, ldb, 0.0, C, ldc, *extra, opts, None)

        # unknown activation, bias type or transpose flag
        assert call(4, 4, 4, 4, 4, 4, b.make_opts(act=3)) == b.GEMM_ERR_INVALID_ARG
        assert call(4, 4, 4, 4, 4, 4, b.make_opts(act=-1)) == b.GEMM_ERR_INVALID_ARG
        assert call(4, 4, 4, 4, 4, 4, b.make_opts(bias_type=5)) == b.GEMM_ERR_INVALID_ARG
        bad = b.make_opts()
        bad.trans_a = 2
        assert call(4, 4, 4, 4, 4, 4, bad) == b.GEMM_ERR_INVALID_ARG
        # trans_a: A stored K x M needs lda >= M; trans_b: B stored N x K
        # needs ldb >= K
        ta, tb = b.make_opts(trans_a=True), b.make_opts(trans_b=True)
        assert call(8, 4, 2, 4, 4, 4, ta) == b.GEMM_ERR_BAD_LD      # lda 4 < M 8
        assert call(2, 4, 8, 4, 4, 4, tb) == b.GEMM_ERR_BAD_LD      # ldb 4 < K 8
        # C overlapping a transposed A (stored K x M = 16 x 4, pitch 4: at
        # least 128 bytes; row-major it would be rejected as lda < K)
        assert call(4, 4, 16, 4, 4, 4, ta, A=fake, C=fake + 100) == b.GEMM_ERR_ALIAS
        # bias overlapping C
        ob = b.make_opts(bias=fake + 131072 + 8)
        assert call(4, 4, 4, 4, 4, 4, ob) == b.GEMM_ERR_ALIAS
        # empty output: nothing to do, no pointer needed
        assert f(0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, *extra, ta, None) == b.GEMM_OK


def test_batched_entry_point_errors(lib):
    """gemm_bf16_batched / gemm_f32_batched: batch and stride checks run
    before any CUDA call."""
    from dense_gemm_02_gb300 import binding as b

    fake = 1 << 20
    for f, extra in ((b.gemm_bf16_batched, (b.GEMM_OUT_F32,)), (b.gemm_f32_batched, ())):
        def call(batch, sa, sb, sc, A=fake, B=fake + (1 << 16), C=fake + (1 << 18), opts=None):
            return f(batch, 4, 4, 4, 1.0, A, 4, sa, B, 4, sb, 0.0, C, 4, sc, *extra, opts, None)

        assert call(-1, 16, 16, 16) == b.GEMM_ERR_INVALID_ARG
        assert call(0, 16, 16, 16, A=None, B=None, C=None) == b.GEMM_OK  # empty batch
        assert call(2, -16, 16, 16) == b.GEMM_ERR_INVALID_ARG
        assert call(2, 16, 16, -16) == b.GEMM_ERR_INVALID_ARG
        # C matrices 8 elements apart overlap (one 4 x 4 C spans 16)
        assert call(2, 16, 16, 8) == b.GEMM_ERR_ALIAS
        assert call(3, 16, 16, 0) == b.GEMM_ERR_ALIAS
        # the third C lands on B's first matrix
        assert call(3, 0, 0, 1 << 14, C=fake + (1 << 16) - 2 * (1 << 14) * 4) == b.GEMM_ERR_ALIAS
        # unknown option still reported first
        assert call(2, 16, 16, 16, opts=b.make_opts(act=9)) == b.GEMM_ERR_INVALID_ARG


def test_config_keys(lib):
    from dense_gemm_02_gb300 import binding as b

    old = b.get_config("watchdog_ms")
    b.set_config("watchdog_ms", 250)
    assert b.get_config("watchdog_ms") == 250
    b.set_config("watchdog_ms", old)
    with pytest.raises(b.GemmError):
        b.set_config("no_such_key", 1)
    with pytest.raises(b.GemmError):
        b.set_config("bf16_tile_n", 96)
    # every documented key round-trips its default and rejects a bad value
    for key, bad in (("force_path", 3), ("fault_inject", 2), ("split_k", 65), ("bf16_tile_n", 64),
                     ("tail_split_off", 2), ("stream_k", 2), ("raster_group", -1),
                     ("cta_pair", 3), ("pair_limit", -1), ("stage_pairs", 3),
                     ("kpair_maps_off", 2)):
        v = b.get_config(key)
        b.set_config(key, v)
        with pytest.raises(b.GemmError):
            b.set_config(key, bad)
        assert b.get_config(key) == v
    b.set_config("pair_limit", 4)
    assert b.get_config("pair_limit") == 4
    b.set_config("pair_limit", 0)
    assert b.last_kernel() in {"none", "sgemm_simt", "sgemm_tma", "bf16_tcgen05", "bf16_simt",
                                "f32_simt", "scale_c"}


def test_package_fails_loudly_without_library(tmp_path, monkeypatch):
    from dense_gemm_02_gb300 import _build, binding

    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_ctypes_signatures_match_header_arity(lib):
    from dense_gemm_02_gb300 import binding

    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for name, (_res, args) in binding.SIGNATURES.items():
        m = re.search(name + r"\s*\(([^)]*)\)", text)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), name
    assert isinstance(lib, ctypes.CDLL)


def test_grouped_entry_point_errors(lib):
    """gemm_bf16_grouped / gemm_f32_grouped: every problem's checks and the
    cross-problem overlap check run before any CUDA call."""
    from dense_gemm_02_gb300 import binding as b

    fake = 1 << 24

    def prob(A, B, C, M=4, N=4, K=4, lda=4, ldb=4, ldc=4, alpha=1.0, beta=0.0):
        return (M, N, K, A, lda, B, ldb, C, ldc, alpha, beta)

    for grouped, esz in ((lambda g, n, o=None: b.gemm_bf16_grouped(g, n, b.GEMM_OUT_F32, o, None), 2),
                         (lambda g, n, o=None: b.gemm_f32_grouped(g, n, o, None), 4)):
        A0, B0, C0 = fake, fake + 4096, fake + 8192
        A1, B1, C1 = fake + 12288, fake + 16384, fake + 20480
        ok = [prob(A0, B0, C0), prob(A1, B1, C1)]
        assert grouped(b.make_groups([]), -1) == b.GEMM_ERR_INVALID_ARG
        assert grouped(None, 0) == b.GEMM_OK  # nothing to do
        assert grouped(None, 2) == b.GEMM_ERR_NULLPTR
        # a bad pitch in the second problem
        assert grouped(b.make_groups([ok[0], prob(A1, B1, C1, lda=2)]), 2) == b.GEMM_ERR_BAD_LD
        # a missing operand
        assert grouped(b.make_groups([ok[0], prob(None, B1, C1)]), 2) == b.GEMM_ERR_NULLPTR
        # no epilogue in grouped calls
        assert grouped(b.make_groups(ok), 2, b.make_opts(act=b.GEMM_ACT_RELU)) == \
            b.GEMM_ERR_INVALID_ARG
        # problem 1 writes into problem 0's A, B or C
        for target in (A0, B0, C0 + 8):
            bad = [ok[0], prob(A1, B1, target)]
            assert grouped(b.make_groups(bad), 2) == b.GEMM_ERR_ALIAS, target
        # problem 1 reads problem 0's C
        assert grouped(b.make_groups([ok[0], prob(C0, B1, C1)]), 2) == b.GEMM_ERR_ALIAS
        # (shared read-only operands are allowed: tested on the GPU with
        # real buffers, since a call that passes the checks launches)


def test_host_batch_entry_point_errors(lib):
    """gemm_host_batch: the count, every product's checks and the
    cross-product overlap check run before any CUDA call."""
    from dense_gemm_02_gb300 import binding as b

    fake = 1 << 24
    F32, BF = b.GEMM_HOST_F32, b.GEMM_HOST_BF16

    def op(A, B, C, dtype=F32, c_type=b.GEMM_OUT_F32, M=4, N=4, K=4, lda=4, ldb=4, ldc=4,
           alpha=1.0, beta=0.0):
        return (dtype, c_type, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc)

    A0, B0, C0 = fake, fake + 4096, fake + 8192
    A1, B1, C1 = fake + 12288, fake + 16384, fake + 20480
    ok = [op(A0, B0, C0), op(A1, B1, C1, dtype=BF)]
    assert b.gemm_host_batch(b.make_host_ops([]), -1) == b.GEMM_ERR_INVALID_ARG
    assert b.gemm_host_batch(b.make_host_ops(ok), b.GEMM_HOST_BATCH_MAX + 1) == \
        b.GEMM_ERR_INVALID_ARG
    assert b.gemm_host_batch(None, 0) == b.GEMM_OK  # nothing to do
    assert b.gemm_host_batch(None, 2) == b.GEMM_ERR_NULLPTR
    # products with M == 0 or N == 0 are skipped: a batch of them does nothing
    assert b.gemm_host_batch(b.make_host_ops([op(A0, B0, C0, M=0), op(A1, B1, C1, N=0)]), 2) == \
        b.GEMM_OK
    # an unknown element type, a bad output type for a bf16 product
    assert b.gemm_host_batch(b.make_host_ops([ok[0], op(A1, B1, C1, dtype=7)]), 2) == \
        b.GEMM_ERR_INVALID_ARG
    assert b.gemm_host_batch(b.make_host_ops([ok[0], op(A1, B1, C1, dtype=BF, c_type=5)]), 2) == \
        b.GEMM_ERR_INVALID_ARG
    # a bad pitch or a missing operand in the second product
    assert b.gemm_host_batch(b.make_host_ops([ok[0], op(A1, B1, C1, ldb=2)]), 2) == \
        b.GEMM_ERR_BAD_LD
    assert b.gemm_host_batch(b.make_host_ops([ok[0], op(A1, None, C1)]), 2) == \
        b.GEMM_ERR_NULLPTR
    # C overlapping its own A (the single-product rule)
    assert b.gemm_host_batch(b.make_host_ops([op(A0, B0, A0 + 4)]), 1) == b.GEMM_ERR_ALIAS
    # product 1 writes into product 0's A, B or C, or reads product 0's C
    for target in (A0, B0, C0 + 8):
        assert b.gemm_host_batch(b.make_host_ops([ok[0], op(A1, B1, target)]), 2) == \
            b.GEMM_ERR_ALIAS, target
    assert b.gemm_host_batch(b.make_host_ops([ok[0], op(C0, B1, C1)]), 2) == b.GEMM_ERR_ALIAS
