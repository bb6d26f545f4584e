"""Host logic of bench.py that needs no GPU: the FLOP count of the metric,
the clock record kept beside each number, and the traffic record's link to
the kernel source it was captured from."""
import hashlib
import json

import pytest

import bench


def test_prefill_flops():
    # causal counts half of 4 B H N^2 D
    assert bench.prefill_flops(1, 32, 16384, 128) == pytest.approx(2.19902e12, rel=1e-5)
    assert bench.prefill_flops(4, 16, 2048, 128, causal=False) == 4.0 * 4 * 16 * 2048 ** 2 * 128
    assert bench.prefill_flops(4, 16, 2048, 128) == 2.0 * 4 * 16 * 2048 ** 2 * 128


def test_clock_summary_keeps_the_timed_window():
    s = bench.ClockSampler(0)
    s.max_mhz = 2070.0
    s.samples = [(0.5, 900.0, 0x8),      # before the timed region: ignored
                 (1.0, 2070.0, 0x0),
                 (1.5, 2000.0, 0x4),     # power cap inside the region
                 (2.0, 1980.0, 0x0),
                 (3.5, 500.0, 0x40)]     # after it: ignored
    s.t0, s.t1 = 1.0, 2.0
    r = s.summary()
    assert r["sm_mhz"] == 2000.0
    assert r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] == 3


def test_clock_summary_names_every_reason():
    s = bench.ClockSampler(0)
    s.samples = [(None, 1500.0, 0x8 | 0x20 | 0x40 | 0x4)]  # nvidia-smi samples carry no time
    r = s.summary()
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                            "sw_thermal_slowdown"]
    assert r["sm_mhz"] == 1500.0


def test_traffic_record_follows_the_source(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"bytes_per_launch": 123.0,
                 "source_sha256": hashlib.sha256(src.read_bytes()).hexdigest()}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("k", "k.cu") == 123.0
    assert bench.load_traffic("other", "k.cu") is None
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.load_traffic("k", "k.cu") is None
