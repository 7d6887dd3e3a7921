"""bench.py's clock record, on CPU: the summary of nvidia-smi samples that
goes into the JSON line (median SM clock under load, the throttle reasons
seen, the hottest sample), parsed from a file of samples as nvidia-smi
writes them (csv, no header, no units)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _sampler_with(lines, tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(line + "\n" for line in lines))
    s = bench.ClockSampler(0)
    s.path = str(path)
    return s


def test_summary_of_samples(tmp_path):
    # index, sm, max sm, power, active, hw, hw thermal, sw thermal, sw power cap, temp, mem
    rows = ["0, 2070, 2070, 1002.5, 0x4, Not Active, Not Active, Not Active, Active, 45, 3996",
            "0, 2010, 2070, 1180.0, 0x4, Not Active, Not Active, Not Active, Active, 49, 3996",
            "0, 1995, 2070, 990.1, 0x0, Not Active, Not Active, Not Active, Not Active, 47, 3996"]
    summ = _sampler_with(rows, tmp_path).summary()
    assert summ["sm_mhz"] == 2010
    assert summ["sm_max_mhz"] == 2070
    assert summ["power_w_max"] == 1180.0
    assert summ["temp_c_max"] == 49
    assert summ["mem_mhz"] == 3996
    assert summ["samples"] == 3
    assert summ["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(tmp_path / "clocks.csv")  # the sample file is removed


def test_slowdown_reasons_are_reported(tmp_path):
    rows = ["0, 1500, 2070, 700.0, 0x8, Active, Not Active, Active, Not Active, 88, 3996"]
    summ = _sampler_with(rows, tmp_path).summary()
    assert summ["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_samples_without_the_newer_fields(tmp_path):
    # nine fields (an older field list): the summary still forms, without temperature
    rows = ["0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    summ = _sampler_with(rows, tmp_path).summary()
    assert summ["sm_mhz"] == 2070 and summ["temp_c_max"] is None and summ["mem_mhz"] is None


def test_no_samples(tmp_path):
    summ = _sampler_with([], tmp_path).summary()
    assert summ["sm_mhz"] is None and summ["reasons"] == ["no nvidia-smi samples"]
