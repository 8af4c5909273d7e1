"""The bench's host-side bookkeeping (CPU only): the algorithmic byte and
flop counts per GEMM, and the DRAM-traffic record that the roofline object
carries only while the profiled kernel source is unchanged."""
import hashlib
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_counts_of_the_sweep_shape():
    N, K = bench.N, bench.K
    assert (N, K) == (8192, 21760)
    assert bench.weight_bytes() == 89_128_960 + 4 * 8192    # packed int4 + fp32 channel scales
    # M=1024: weights + int8 activations + token scales + fp16 output
    assert bench.algo_bytes(1024) == bench.weight_bytes() + 1024 * K + 4 * 1024 + 2 * 1024 * N
    assert bench.flops(1024) == 2 * 1024 * N * K


def test_traffic_records_point_at_their_sources_and_match():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    assert recs, "no traffic records"
    for kernel, rec in recs.items():
        src = os.path.join(ROOT, rec["src"])
        assert os.path.exists(src), (kernel, rec["src"])
        assert os.path.exists(os.path.join(ROOT, rec["from"])), (kernel, rec["from"])
        assert rec["dram_bytes_per_launch"] > 0
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
        got = bench.measured_traffic(kernel, rec["M"])
        # a record whose source changed since the capture reports no traffic
        assert got == (rec["dram_bytes_per_launch"] if sha.startswith(rec["src_sha1_prefix"]) else None)
        assert bench.measured_traffic(kernel, rec["M"] + 1) is None  # another M: no record


def test_traffic_is_dropped_when_the_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = hashlib.sha1(src.read_bytes()).hexdigest()
    (prof / "traffic.json").write_text(json.dumps({"k": {"M": 4, "src": "k.cu", "src_sha1_prefix": sha[:12],
                                                         "dram_bytes_per_launch": 123, "from": "x"}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("k", 4) == 123
    src.write_text("kernel v2\n")
    assert bench.measured_traffic("k", 4) is None
    assert bench.measured_traffic("missing", 4) is None
