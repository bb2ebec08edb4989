"""Host-side pieces of the benchmark, checked on CPU: the roofline rows, the peak
fallback, the clock sampler's parsing of nvidia-smi lines, and the e2e/launch
fields' arithmetic."""
import os

import pytest

import bench


def test_rows_divide_work_by_time_and_peak():
    pk = {"hbm": 6000.0, "bf16": 2000.0}
    r = bench._hbm_row(6e9, 1.0, pk, "x")        # 6 GB in 1 ms = 6000 GB/s
    assert r["GB/s"] == 6000.0 and r["frac"] == 1.0
    t = bench._tc_row(2e12, 2.0, pk, "g")        # 2 TFLOP in 2 ms = 1000 TFLOP/s
    assert t["TOPS"] == 1000.0 and t["frac"] == 0.5


def test_peaks_fall_back_when_the_measurement_is_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()
    assert pk["source"] == "fallback" and pk["hbm"] == 6800.0 and pk["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6786.9, "bf16_tflops": 1873.6}')
    pk = bench.peaks()
    assert pk["source"] == "measured" and pk["hbm"] == 6786.9 and pk["bf16_sustained"] == 1873.6


def test_clock_sampler_parses_reasons_and_median(tmp_path):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc, s.nvml = None, None
    f = open(tmp_path / "c.csv", "w+")
    lines = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    f.write("\n".join(lines) + "\n")
    f.flush()
    s.file = f
    out = s.stop()
    assert out["samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(tmp_path / "c.csv")


def test_nvml_sampler_is_absent_without_a_driver():
    s = bench.NvmlSampler(None, 0)
    if s.lib is None:
        assert s.stop() is None
    else:  # a machine with a driver: the sampler runs and stops cleanly
        assert isinstance(s.stop()["samples"], list)


@pytest.mark.parametrize("world,steps,ms", [(1, 20, 73.5), (8, 20, 80.0)])
def test_weak_scaling_value(world, steps, ms):
    ops = 4.0 * 20480 * 16384 * 4096
    v = bench.weak_scaling_value(world, ops, steps, ms)
    assert v == pytest.approx(world * ops * steps / (ms * 1e-3) / 1e12)
