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


def test_rotation_reads_a_different_copy_every_gemm():
    nper, R = len(bench.M_SWEEP), bench.ROTATE
    seq = [bench.rotation(i, j) for i in range(3 * R) for j in range(nper)]
    assert all(0 <= c < R for c in seq)
    # consecutive GEMMs (also across steps) read different copies, and a copy
    # comes back only after R - 1 others
    for g in range(len(seq) - R):
        assert seq[g + R] == seq[g]
        assert len(set(seq[g:g + R])) == R
    # the step graphs repeat with the rotation period
    P = bench.rotation_period()
    for i in range(2 * P):
        assert [bench.rotation(i, j) for j in range(nper)] == \
            [bench.rotation(i + P, j) for j in range(nper)]
    # (R - 1) 89 MB weight copies between two reads of one copy exceed 2x L2
    assert (R - 1) * bench.weight_bytes() > 2 * bench.L2_BYTES


def test_copies_for_exceeds_twice_l2():
    for nb in (1, 9_000_000, 62_000_000, 200_000_000, 10 ** 9):
        R = bench.copies_for(nb)
        assert R >= 2 and (R - 1) * nb > 2 * bench.L2_BYTES


def test_parse_clocks_window_and_reasons():
    text = "\n".join([
        "2026/01/01 00:00:00.000, 1500, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/01 00:00:01.000, 2070, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/01/01 00:00:01.100, 2060, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/01/01 00:00:05.000, 1000, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    import datetime
    t = lambda s: datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    c = bench.parse_clocks(text, t("2026/01/01 00:00:00.500"), t("2026/01/01 00:00:02.000"))
    assert c["samples"] == 2 and c["sm_mhz"] == 2065 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 950.0
    assert bench.parse_clocks(text)["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.parse_clocks("") is None


def test_roofline_entry_picks_the_binding_limit():
    pk = dict(hbm=6758.2, bf16=1888.6, bf16_sus=1710.5, src="measured")
    # M=1: HBM-bound; at the floor time the fraction is 1
    t = bench.algo_bytes(1) / (pk["hbm"] * 1e9) * 1e6
    e = bench.roofline_entry(t, bench.flops(1), bench.algo_bytes(1), pk)
    assert e["bound"] == "hbm" and abs(e["roofline_frac"] - 1) < 1e-3
    # M=1024: tensor-bound against the burst peak
    t = bench.flops(1024) / (pk["bf16"] * 1e12) * 1e6 * 2
    e = bench.roofline_entry(t, bench.flops(1024), bench.algo_bytes(1024), pk)
    assert e["bound"] == "tensor" and abs(e["roofline_frac"] - 0.5) < 1e-3
