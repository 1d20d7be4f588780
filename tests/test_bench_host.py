"""Host-side logic of bench.py (no GPU): the clock-sample summary, the
per-stage algorithmic accounting, the workload overrides and the recorded
DRAM-traffic lookup."""
import json

import pytest

import bench
import synth


def _sampler(lines):
    c = bench.ClockSampler(0)
    c.lines = lines
    return c.summary()


def test_clock_summary_takes_the_loaded_samples_and_the_active_reasons():
    s = _sampler([
        "0, 2070, 2070, 1250.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1950, 2070, 1380.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1500, 2070, 140.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # idle: left out
        "garbage line",
    ])
    assert s["samples"] == 3 and s["samples_under_load"] == 2
    assert s["sm_mhz"] == pytest.approx((2070 + 1950) / 2)
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_and_hw_slowdown():
    s = _sampler(["0, 1200, 2070, 1300.0, 0x8, Active, Not Active, Active, Not Active"])
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    assert _sampler([])["samples"] == 0


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen2", "skew", "deepseek", "mixtral22b"])
def test_stage_flops_add_up_to_the_layer(name):
    wl = synth.workload(name, T=512)
    alg = bench.stage_algorithmic(wl, wl.E)
    total = sum(f for f, _ in alg.values())
    extra_gate = 2.0 * wl.T * wl.H if wl.shared_gate else 0.0  # the shared gate rides in the router GEMM
    assert total + extra_gate == pytest.approx(wl.flops(), rel=1e-12)
    # every stage moves at least its inputs once
    assert all(b > 0 for _, b in alg.values())
    f, b = alg["gate_up_gemm"]
    assert b >= wl.E * 4.0 * wl.H * wl.F  # the gate and up weights of the active experts


def test_job_throughput_counts_every_replica():
    assert bench.job_tokens_per_s(4, 1000, 10, 20.0) == pytest.approx(4 * 1000 * 10 / 0.020)


def test_workload_overrides():
    class A:
        workload, alpha, activation, experts = "deepseek", None, "gelu", 32
    kw = bench.workload_overrides(A)
    assert kw == {"activation": "gelu", "E": 32}
    wl = synth.workload("deepseek", T=64, **kw)
    assert wl.E == 32 and wl.n_group == 8 and "E=32" in wl.label and "act=gelu" in wl.label

    class B:
        workload, alpha, activation, experts = "deepseek", None, None, 12  # not a multiple of 8 groups
    with pytest.raises(SystemExit):
        bench.workload_overrides(B)


def test_recorded_traffic_only_for_the_current_sources_and_workload(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"gate_up_gemm": {"workload": "w", "sources_sha": bench.sources_sha(), "dram_bytes_per_launch": 123},
           "down_gemm": {"workload": "w", "sources_sha": "0000000000000000", "dram_bytes_per_launch": 456}}
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "sources_sha", lambda: rec["gate_up_gemm"]["sources_sha"])
    assert bench.recorded_traffic("gate_up_gemm", "w") == 123
    assert bench.recorded_traffic("gate_up_gemm", "other workload") is None
    assert bench.recorded_traffic("down_gemm", "w") is None  # counters taken on other kernel sources
    assert bench.recorded_traffic("combine", "w") is None
