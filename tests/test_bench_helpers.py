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


# ---------------------------------------------------------------------------
# The oracle leg of every workload (cpu_baseline), on tiny CPU-resident inputs
# set on bare instances (the constructors allocate on the GPU).
# ---------------------------------------------------------------------------
import numpy as np  # noqa: E402
import torch  # noqa: E402

import mla_inputs as mi  # noqa: E402
import oracle  # noqa: E402
from mla_family_attention_gb300 import accounting as acc  # noqa: E402


def _bare(cls, **kw):
    o = object.__new__(cls)
    o.__dict__.update(kw)
    return o


def _check(res, unit, extrapolated=False):
    assert res["unit"] == unit and res["kind"] == "oracle"
    assert res["value"] > 0 and res["cores"] >= 1
    assert ("extrapolated" in res["sample"]) == extrapolated


def test_cpu_sample_decode_kinds():
    dec = mi.make_decode([300, 40], 4, True, config=71)
    _check(_bare(bench.DecodeWork, dec=dec, lengths=dec.lengths, H=4, B=2).cpu_sample(0.01),
           "GB/s")
    cd = mi.make_capacity_decode([99, 99], 4, 100, True, config=72)
    w = _bare(bench.DecodeCachedWork, cd=cd, T=100, H=4, B=2)
    _check(w.cpu_sample(0.01), "GB/s")


def test_cpu_sample_prefill_kinds():
    pf = mi.make_prefill(1, 3, 64, 64, True, config=73)
    w = _bare(bench.PrefillWork, pf=pf, T=64, H=3, work=acc.prefill_flops(1, 3, 64, 64))
    _check(w.cpu_sample(0.01), "TFLOP/s")
    pf = mi.make_prefill(1, 2, 1280, 1280, False, config=74)
    w = _bare(bench.PrefillWork, pf=pf, T=1280, H=2, work=acc.prefill_flops(1, 2, 1280, 1280))
    _check(w.cpu_sample(0.01), "TFLOP/s", extrapolated=True)
    c, n = 256, 3
    pf = mi.make_prefill(1, 2, c * n, c * n, True, config=75)
    sl = [slice(i * c, (i + 1) * c) for i in range(n)]
    w = _bare(bench.ChunkedPrefillWork, q=[pf.q[:, :, s] for s in sl],
              kn=[pf.k[:, :, s] for s in sl], vn=[pf.v[:, :, s] for s in sl],
              g=[pf.gate[:, s] for s in sl], c=c, T=c * n, H=2, scale=pf.scale)
    _check(w.cpu_sample(0.01), "TFLOP/s", extrapolated=True)


def test_cpu_sample_dsa_kinds():
    lengths = [3000, 500]
    d = mi.make_dsa(lengths, H=2, config=76)
    _check(_bare(bench.DsaWork, d=d, lengths=lengths, H=2, B=2, topk=256).cpu_sample(0.01),
           "GB/s")
    _check(_bare(bench.IndexWork, d=d, lengths=lengths, B=2, topk=256).cpu_sample(0.01), "GB/s")
    codes, sc = oracle.quantize_e4m3_rows(d.index_k)
    w = _bare(bench.IndexFp8Work, d=d, lengths=lengths, B=2, topk=256,
              k8=torch.from_numpy(codes), ks=torch.from_numpy(sc))
    _check(w.cpu_sample(0.01), "GB/s")


def test_cpu_sample_latent_kinds():
    lat = mi.make_latent_decode([200, 30], 16, True, config=77)
    w = _bare(bench.LatentDecodeWork, d=lat, lengths=lat.lengths, H=16, B=2)
    _check(w.cpu_sample(0.01), "GB/s", extrapolated=True)
    rec = torch.from_numpy(oracle.quantize_latent_records(lat.ckv))
    w = _bare(bench.LatentDecodeFp8Work, d=lat, lengths=lat.lengths, H=16, B=2, rec=rec)
    _check(w.cpu_sample(0.01), "GB/s", extrapolated=True)
    dp = mi.make_dsa_prefill(300, 300, 8, config=78)
    w = _bare(bench.DsaPrefillWork, d=dp, T=300, K=64, H=8)
    _check(w.cpu_sample(0.01), "TFLOP/s", extrapolated=True)


def test_compact_keeps_the_summary_figures():
    entry = {"value": 1.5, "unit": "GB/s", "ms_per_step": 2.0, "steps": 3,
             "roofline": {"frac": 0.5, "kernel_ms": 1.9, "other_kernels": {}},
             "cpu_baseline": {"value": 0.01}}
    got = bench._compact(entry)
    assert dict(zip(bench.ALSO_FIELDS, got)) == {
        "value": 1.5, "unit": "GB/s", "ms_per_step": 2.0, "roofline.frac": 0.5,
        "roofline.kernel_ms": 1.9, "cpu_baseline.value": 0.01,
        "latency_after_l2_flush_ms": None}
    entry["latency_after_l2_flush_ms"] = 0.0146
    assert bench._compact(entry)[-1] == 0.0146
