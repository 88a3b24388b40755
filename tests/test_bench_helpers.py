"""The benchmark's roofline bookkeeping on CPU: the ncu traffic of a kernel is
reported only while its source is the one the capture measured, and the
roofline object takes the longest kernel of the step's bound against the
measured peak."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_table_entries_match_current_sources():
    """Every entry with bytes names a source file that exists; an entry whose
    hash matches that file is reported, any other is withheld (None)."""
    table = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert table
    for kernel, entry in table.items():
        src = os.path.join(ROOT, entry["source"])
        assert os.path.exists(src), kernel
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        got = bench.traffic_for(kernel)
        if digest == entry["source_sha256_16"]:
            assert got == entry["dram_bytes_per_launch"], kernel
            units = entry.get("algorithmic_per_launch")
            if got is not None and units:
                # traffic of a launch with twice the work: twice the bytes
                assert bench.traffic_for(kernel, 2 * units) == pytest.approx(2 * got, rel=1e-9)
        else:
            assert got is None, kernel


def test_traffic_withheld_for_a_changed_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (prof / "traffic.json").write_text(json.dumps(
        {"k": {"source": "k.cu", "source_sha256_16": digest, "dram_bytes_per_launch": 123,
               "algorithmic_per_launch": 100}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k") == 123
    assert bench.traffic_for("k", 1000) == 1230     # another launch of the kernel, 10x the work
    src.write_text("kernel v2\n")
    assert bench.traffic_for("k") is None
    assert bench.traffic_for("unknown") is None


class _Work:
    bound = "hbm"


def test_roofline_takes_the_longest_kernel_of_the_bound(monkeypatch):
    monkeypatch.setattr(bench, "peaks", lambda bound="hbm": (
        (2000.0, "TFLOP/s", "test") if bound == "tensor" else (8000.0, "GB/s", "test")))
    monkeypatch.setattr(bench, "traffic_for", lambda k, units=None: None)
    kern = [("small", 0.01, 4e7, "hbm"), ("big", 2.0, 16e9, "hbm"), ("mma", 3.0, 3e12, "tensor")]
    r = bench.roofline(_Work(), kern)
    assert r["kernel"] == "big"
    assert r["achieved"] == pytest.approx(16e9 / 2e-3 / 1e9)
    assert r["frac"] == pytest.approx(8000.0 / 8000.0)
    assert r["algorithmic_bytes_per_launch"] == 16e9
    assert set(r["other_kernels"]) == {"small", "mma"}
    assert r["other_kernels"]["mma"]["unit"] == "TFLOP/s"
    assert r["other_kernels"]["mma"]["frac"] == pytest.approx((3e12 / 3e-3 / 1e12) / 2000.0)
