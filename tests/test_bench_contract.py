"""Host logic of bench.py that needs no GPU: the reference arm's JSON line
(the oracle timed on a bounded sample) and the clock sampler's reading of
nvidia-smi output (median SM clock under load, throttle reasons)."""
import argparse
import json
import os
import stat

import pytest

import bench


def _run_reference(monkeypatch, capsys, rank=0, world=1):
    small = dict(bench.WORKLOAD, prefill=600)        # a short prefix keeps it to ~1 s
    monkeypatch.setattr(bench, "WORKLOAD", small)
    args = argparse.Namespace(steps=3, warmup=3)
    bench.reference_arm(args, rank, world)
    return capsys.readouterr().out.strip()


def test_reference_line_carries_the_contract_keys(monkeypatch, capsys):
    line = json.loads(_run_reference(monkeypatch, capsys))
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 3 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert cb["cpu"]                            # the host CPU model is named
    assert "600-token prefill" in cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the value is the sample's algorithmic bytes over its time
    nbytes, _ = bench.kv_bytes(1, bench.WORKLOAD["n_kv_heads"], bench.WORKLOAD["head_dim"], 601,
                               max(1, 600 * bench.WORKLOAD["budget"] // 600))
    assert line["value"] == pytest.approx(nbytes / (line["ms_per_step"] * 1e-3) / 1e9, rel=2e-3)


def test_reference_arm_prints_on_rank_0_only(monkeypatch, capsys):
    assert _run_reference(monkeypatch, capsys, rank=1, world=2) == ""


def _fake_smi(tmp_path, lines):
    """An nvidia-smi stand-in that prints canned query lines, then waits."""
    script = tmp_path / "nvidia-smi"
    body = "\n".join(f"echo '{x}'" for x in lines)
    script.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    script.chmod(script.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def test_clock_sampler_takes_the_loaded_median_and_the_reasons(tmp_path, monkeypatch):
    rows = ["0, 1980, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2070, 2070, 700.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2040, 2070, 710.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2055, 2070, 705.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    res = s.stop()
    assert res["samples"] == 4 and res["sm_max_mhz"] == 2070.0
    assert res["sm_mhz"] == 2055.0             # median of the three samples under load
    assert res["reasons"] == ["sw_power_cap"] and res["power_w_max"] == 710.0


def test_clock_sampler_reports_thermal_slowdown(tmp_path, monkeypatch):
    rows = ["0, 1500, 2070, 900.0, 0x40, Not Active, Active, Not Active, Not Active"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    res = s.stop()
    assert res["reasons"] == ["hw_thermal_slowdown"] and res["sm_mhz"] == 1500.0


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))          # an empty directory
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_cpu_baseline_repeats_the_oracle_step_to_a_bounded_sample():
    from workloads import llama8b_workload
    wl = llama8b_workload(0, prefill_len=400, n_layers=2)
    val, secs, sample = bench.cpu_baseline(wl, 2, min_seconds=0.2, max_reps=3)
    reps = int(sample.split("timed ")[1].split()[0])
    assert 1 <= reps <= 3 and secs > 0
    assert "first 2 of 32 layers (all 401 tokens)" in sample
    nbytes, _ = bench.kv_bytes(2, bench.WORKLOAD["n_kv_heads"], bench.WORKLOAD["head_dim"], 401,
                               bench.WORKLOAD["budget"])
    assert val == pytest.approx(nbytes * reps / secs / 1e9)
