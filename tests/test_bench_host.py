"""The bench's host-side reporting: the clock-normalised tensor peak, the CPU
baseline record (threads, extrapolation, ring-simulation timings) and the DRAM
traffic figure read from the committed ncu summary.  No GPU is needed."""

import dataclasses

import pytest

import bench
from context_ring_attention_gb300 import workloads


def test_clock_peak():
    # 152 SMs x 8192 dense bf16 FLOP per SM per clock at 2070 MHz
    assert bench.clock_peak(152, 2070.0) == pytest.approx(152 * 8192 * 2070e6 / 1e12)
    assert bench.clock_peak(152, 2070.0) == pytest.approx(2577.5, abs=0.1)
    assert bench.clock_peak(152, None) is None          # no clock sample: no fraction


def test_cpu_baseline_record_fields():
    # a small workload so the sample takes a moment: 8 rows of one 4k head
    wl = workloads.WORKLOADS["noncausal_4k_n8"]
    rec = bench.cpu_baseline_record(wl, rows=8, with_ring_sim=True)
    assert rec["kind"] == "oracle" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["cores"] >= 1
    assert rec["blas_threads"] is None or rec["blas_threads"] >= 1
    # the extrapolation is the whole workload at the measured rate, and says so
    assert rec["extrapolated_full_s"] == pytest.approx(wl.flops() / (rec["value"] * 1e12))
    assert "extrapolated" in rec["extrapolated_note"]
    rs = rec["ring_sim"]
    assert set(rs) == {"toy_ring_4x3_d8", "noncausal_4k_n8"}
    assert rs["noncausal_4k_n8"]["extrapolated_full_s"] == pytest.approx(rs["noncausal_4k_n8"]["seconds"] * 64)


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    got = bench.measured_traffic("zigzag_1m_n8")
    assert got is None or got > 21.6e9           # at least the compulsory bytes of the 1M launch
    monkeypatch.setattr(bench, "fwd_source_digest", lambda: "0" * 64)
    assert bench.measured_traffic("zigzag_1m_n8") is None   # sources changed since the capture
    assert bench.measured_traffic("no_such_workload") is None


def test_config_names_the_workload():
    wl = dataclasses.replace(workloads.WORKLOADS["causal_32k_n8"], layouts=("zigzag",))
    cfg = bench.config_of(wl)
    assert cfg["workload"] == "causal_32k_n8" and cfg["layout"] == "zigzag" and cfg["seq"] == 32768


def test_exp_rate():
    # 1M causal zigzag: 9.007e15 FLOP -> 1.759e13 exponentials; over 5.18 s at 1845 MHz
    r = bench.exp_rate(9007207844675584, 128, 5.18, 152, 1845.0)
    assert abs(r["achieved_per_s"] - 9007207844675584 / 512 / 5.18) < 1e3
    assert abs(r["peak_per_s"] - 152 * 32 * 1845e6) < 1.0
    assert 0.37 < r["frac"] < 0.39
    assert bench.exp_rate(1e12, 128, 1.0, 152, None)["frac"] is None
