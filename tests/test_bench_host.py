"""Host logic of bench.py that needs no GPU: when recorded ncu DRAM traffic
may be attached to a kernel (only while the kernel's code is the captured
one), the variant parser, workload selection and the peak table."""

import json
import os
import shutil

import pytest

import bench
from gemm_inputs.workloads import WORKLOADS


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    """A copy of the kernel sources under a scratch root with a traffic
    record made for them, so edits do not touch the tree."""
    csrc = tmp_path / "dense_gemm_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("sgemm_tma.cu", "gemm_bf16_tc.cu"):
        shutil.copy(os.path.join(bench.ROOT, "dense_gemm_02_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {name: {"kernel": bench.kernel_name(w), "source_sha256_16": bench.kernel_source_hash(w),
                  "dram_bytes_per_launch": 1000.0 + w.index}
           for name, w in WORKLOADS.items() if name != "sgemm_256"}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    return tmp_path


def test_recorded_traffic_follows_the_code_not_its_comments(fake_root):
    w = WORKLOADS["sgemm_4096"]
    assert bench.recorded_traffic(w) == 1000.0 + w.index
    src = fake_root / "dense_gemm_02_gb300" / "csrc" / "sgemm_tma.cu"
    text = src.read_text()
    # comments and whitespace runs: still the captured kernel
    src.write_text("// a new comment\n/* and a\n   block comment */\n" +
                   text.replace(";\n", ";   \n", 3))
    assert bench.recorded_traffic(w) == 1000.0 + w.index
    # a code change: the record no longer applies
    edited = text.replace("TBK = 32", "TBK = 16", 1)
    assert edited != text
    src.write_text(edited)
    assert bench.recorded_traffic(w) is None
    # the BF16 records follow their own source
    assert bench.recorded_traffic(WORKLOADS["bf16_4096"]) == 1000.0 + WORKLOADS["bf16_4096"].index


def test_recorded_traffic_absent_or_unknown(fake_root):
    os.remove(fake_root / "profiles" / "traffic.json")
    assert bench.recorded_traffic(WORKLOADS["bf16_4096"]) is None


def test_committed_records_are_well_formed():
    # (whether they are current is the bench's decision at run time: a
    # stale record reads as null, it is not an error)
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert set(rec) <= set(WORKLOADS)
    for name, r in rec.items():
        assert len(r["source_sha256_16"]) == 16 and r["dram_bytes_per_launch"] > 0, name
        assert r["kernel"].split("<")[0] == bench.kernel_name(WORKLOADS[name]), name


@pytest.mark.parametrize("spec,want", [
    ("plain", (False, False, False, "none")),
    ("tn", (True, False, False, "none")),
    ("nt,bias", (False, True, True, "none")),
    ("tt,bias,gelu", (True, True, True, "gelu")),
    ("relu", (False, False, False, "relu")),
])
def test_parse_variant(spec, want):
    assert bench.parse_variant(spec) == want


def test_parse_variant_rejects_unknown_items():
    with pytest.raises(SystemExit):
        bench.parse_variant("nn,swish")


def test_workload_selection():
    step = bench.workloads_for("step")
    assert [w.name for w in step] == ["bf16_4096", "sgemm_4096"]
    assert bench.workloads_for("bf16_decode_64x8192x8192")[0].M == 64
    with pytest.raises(SystemExit):
        bench.workloads_for("no_such_workload")


def test_peaks_table_has_the_denominators():
    peaks, source = bench.load_peaks()
    assert source in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 0 and peaks["bf16_tflops"] > 0


def test_parity_records_count_violations_and_mismatches(oracle):
    import numpy as np

    import gemm_inputs as gi

    w32 = WORKLOADS["sgemm_256"]
    ref = np.linspace(-3, 3, 12, dtype=np.float64).reshape(3, 4)
    got = ref.astype(np.float32)
    rec = bench.parity_random(w32, got, ref)
    assert rec["violations"] == 0 and rec["compared"] == 12 and rec["rows"] == 3
    got2 = got.copy()
    got2[1, 2] += 1e-5 * w32.K * 2  # beyond 1e-5 K
    got2[2, 3] = np.nan
    assert bench.parity_random(w32, got2, ref)["violations"] == 2
    # bf16 tolerance: 2^-7 |ref| + 1e-2, elementwise
    wb = WORKLOADS["bf16_4096"]
    refb = np.array([[100.0, -100.0, 0.0, 1.0]])
    ok = gi.f32_to_bf16_bits(np.array([[100.5, -100.5, 0.009, 1.0]], np.float32))
    assert bench.parity_random(wb, ok, refb)["violations"] == 0
    bad = gi.f32_to_bf16_bits(np.array([[102.0, -100.0, 0.02, 1.0]], np.float32))
    assert bench.parity_random(wb, bad, refb)["violations"] == 2
    # integer pass: bit-exact after one rounding of the double result
    refi = np.array([[3.0, -5.0, 257.0]])  # 257 rounds to 256 in bf16 (ties to even)
    assert bench.parity_integer(wb, oracle.round_bf16(refi), refi)["mismatches"] == 0
    off = oracle.round_bf16(refi)
    off[0, 2] += 1
    assert bench.parity_integer(wb, off, refi)["mismatches"] == 1


def test_oracle_sample_keeps_products_of_given_operands(oracle):
    import numpy as np

    w = WORKLOADS["sgemm_256"]
    A, B, C = w.operands()
    flops, dt, rows, threads, res = bench.oracle_sample_time([w], 0.01, operands={w.name: (A, B, C)},
                                                            keep=True)
    assert rows >= 1 and flops == 2 * rows * w.N * w.K and dt > 0
    assert np.array_equal(res[w.name], oracle.gemm(A[:rows], B, None))


def test_cpu_model_is_a_name():
    name = bench.cpu_model()
    assert isinstance(name, str) and name
