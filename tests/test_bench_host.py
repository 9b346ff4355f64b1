"""Host logic of the bench (no GPU): the clock record that decides whether a
timed run stands, the traffic record's source-hash gate, and the algorithmic
byte counts behind the roofline numbers."""
import json

import numpy as np
import pytest

import bench
import oracle


def _row(sm, sm_max, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", power="Not Active"):
    return ["0", str(sm), str(sm_max), "900.0", "0x0", hw, thermal, sw_thermal, power]


def test_clock_summary_takes_the_timed_window():
    cs = bench.ClockSampler(0)
    cs.samples = [(0.0, _row(1000, 2070)), (1.0, _row(2070, 2070)), (1.1, _row(2060, 2070)),
                  (1.2, _row(2070, 2070, power="Active")), (5.0, _row(900, 2070, thermal="Active"))]
    s = cs.summary(0.9, 1.3)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]          # kept and noted
    s = cs.summary(4.9, 5.1)
    assert s["reasons"] == ["hw_thermal_slowdown"]   # a run that must be re-measured


def test_clock_summary_short_window_and_no_samples():
    cs = bench.ClockSampler(0)
    cs.samples = [(1.0, _row(2070, 2070)), (1.25, _row(2065, 2070))]
    s = cs.summary(1.05, 1.06)                     # shorter than the sampling period
    assert s["samples"] == 2 and s["sm_mhz"] == pytest.approx(2067.5)
    cs.samples = []
    assert cs.summary(0, 1) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}


def test_traffic_record_is_gated_by_the_kernel_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic_record("a" * 64) is None                  # no record at all
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(
        json.dumps({"dram_bytes_per_launch": 123.0, "kernel_source_sha256": "a" * 64}))
    assert bench._traffic_record("a" * 64)["dram_bytes_per_launch"] == 123.0
    assert bench._traffic_record("b" * 64) is None                  # taken on other code: not reported


def test_algorithmic_bytes():
    # int4 weights, fp16 scale and zero per 128 inputs, bf16 x in and y out
    assert bench._gemm_bytes(5, 4608, 3584) == 4608 * 3584 // 2 + 4 * 4608 * 28 + 2 * 5 * 3584 + 2 * 5 * 4608
    # verify: fp32 draft rows (gamma) and target rows (gamma + 1) per batch element
    assert bench._verify_bytes(1, 4, 152064) == 4 * 9 * 152064


def test_step_weight_bytes():
    from quantized_speculative_decoding_gb300 import spec_step
    assert spec_step.weight_bytes("bf16", 10, 128) == 2560
    assert spec_step.weight_bytes("int8", 10, 128) == 1280 + 20
    assert spec_step.weight_bytes("int4-tiled", 10, 256) == 1280 + 4 * 10 * 2


def test_traffic_json_is_well_formed():
    import os
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert set(rec) >= {"kernel", "workload", "dram_bytes_per_launch", "command", "kernel_source_sha256"}
    assert "--clock-control none" in rec["command"]


def test_sweep_rows_option():
    assert set(bench.parse_args(["--sweep"]).rows.split(",")) == {
        "a2", "a3", "a4", "a5-a9", "next-1", "next-2", "next-3", "next-4"}
    assert bench.parse_args(["--sweep", "--rows", "next-1"]).rows == "next-1"
    assert bench.parse_args(["--warmup", "1"]).warmup == 3  # at least three warm-up steps


def test_cpu_baseline_all_cores_runs_spawned_workers():
    out = bench.cpu_baseline_all_cores(budget_s=0.2, cores=2, rows=2)
    assert out["cores"] == 2 and out["kind"] == "oracle" and out["unit"] == "GB/s"
    assert out["value"] > 0 and "2 processes" in out["sample"]


def test_acceptance_summary_agrees_with_oracle_trials():
    """The bench's acceptance summary on accept lengths drawn by the oracle's
    verify (independent draft tokens and seeds per trial): the measured mean
    lies within a few standard errors of the closed form."""
    from quantized_speculative_decoding_gb300 import synth
    dl, tl = synth.logits(2, 4, 64, 0.8, 5)
    lens = []
    for trial in range(400):
        dt = synth.draft_tokens(dl, 1.0, 700 + trial)
        lens.append(oracle.verify(dl, tl, dt, 4, 1.0, trial)[1])
    out = bench._acceptance_summary(np.array(lens), dl, tl, 1.0)
    assert out["trials"] == 400
    assert abs(out["closed_form"]["z"]) < 4.5
    beta = out["closed_form"]["beta"]
    assert all(0 < b < 1 for b in beta)
    # conditional acceptance estimates beta, the unconditional one its running product
    assert abs(out["conditional_acceptance"][0] - beta[0]) < 0.1
    assert out["position_acceptance"] == sorted(out["position_acceptance"], reverse=True)


def test_acceptance_summary_at_zero_temperature_has_no_closed_form():
    lens = np.array([[4], [4], [2]])
    dl = np.zeros((1, 4, 8), np.float32)
    out = bench._acceptance_summary(lens, dl, np.zeros((1, 5, 8), np.float32), 0.0)
    assert "closed_form" not in out
    assert out["mean_emitted_tokens"] == (5 + 5 + 3) / 3
    assert out["position_acceptance"] == [1.0, 1.0, 2 / 3, 2 / 3]


def test_oracle_step_extrapolation_counts_every_row():
    per_row = {name: 1e-6 * (i + 1) for i, (name, K, N) in enumerate(bench._layer())}
    got = bench._oracle_step_seconds(per_row, 0.5)
    want = 28 * sum(N * 1e-6 * (i + 1) for i, (_, K, N) in enumerate(bench._layer())) + 0.5
    assert abs(got - want) < 1e-12
    assert bench._step_bytes() > 28 * sum(N * K // 2 for _, K, N in bench._layer())
