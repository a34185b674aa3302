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
    assert [w.name for w in step] == ["sgemm_4096", "bf16_4096"]
    assert bench.workloads_for("bf16_decode_64x8192x8192")[0].M == 64
    with pytest.raises(SystemExit):
        bench.workloads_for("no_such_workload")


def test_peaks_table_has_the_denominators():
    peaks, source = bench.load_peaks()
    assert source in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 0 and peaks["bf16_tflops"] > 0
