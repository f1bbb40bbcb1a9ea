"""Host-side pieces of bench.py that need no GPU: the clock record taken during the timed region
(median SM clock, the maximum, and which throttle reasons were active), its behaviour when
nvidia-smi is absent, the peaks' source, and the workload description."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import configs  # noqa: E402


def _sampler_over(tmp_path, lines):
    s = bench.ClockSampler(0, str(tmp_path))
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = object()  # as if nvidia-smi had been started
    return s


def _row(sm, smax, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {smax}, 812.4, 0x0000000000000000, {hw}, {hwt}, {swt}, {cap}"


def test_clock_summary_median_max_and_reasons(tmp_path):
    s = _sampler_over(tmp_path, [_row(2070, 2070), _row(1980, 2070, cap="Active"),
                                 _row(2040, 2070), "garbage line", _row("[N/A]", 2070)])
    c = s.summary()
    assert c["sm_mhz"] == 2040 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_each_slowdown_reason(tmp_path):
    s = _sampler_over(tmp_path, [_row(1500, 2070, hw="Active"), _row(1400, 2070, hwt="Active"),
                                 _row(1600, 2070, swt="Active")])
    assert s.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown",
                                      "sw_thermal_slowdown"]


def test_clock_summary_without_samples_is_none(tmp_path):
    assert _sampler_over(tmp_path, ["", "not,a,row"]).summary() is None
    s = bench.ClockSampler(0, str(tmp_path))
    assert s.summary() is None  # never started


def test_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi on the path
    with bench.ClockSampler(0, str(tmp_path)) as s:
        pass
    assert s.proc is None and s.summary() is None


def test_measured_peaks_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks()[2] == "fallback"
    with open(os.path.join(tmp_path, "MEASURED_PEAKS.json"), "w") as f:
        json.dump({"hbm_gbs": 6794.8, "bf16_tflops": 1896.2}, f)
    assert bench.measured_peaks() == (6794.8, 1896.2, "measured")


def test_workload_config_names_the_workload():
    cfg = configs.get(1)
    c = bench.workload_config(cfg, {"extra": 1})
    assert c["vocab"] == cfg.V and c["hidden"] == cfg.d and c["verify_rows"] == cfg.k + 1
    assert str(cfg.V) in c["workload"] and c["extra"] == 1
    assert not any(k in c for k in ("model", "global_batch", "seq_len"))
