"""Host logic of bench.py's evidence fields, on CPU: the clock record taken
during the timed region and the ncu traffic record of the dominant kernel."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _row(sm, smax, power, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    active = "0x0000000000000000"
    return ", ".join(["0", str(sm), str(smax), str(power), active, hw, hwt, swt, cap]) + "\n"


def test_clock_summary_takes_the_median_and_every_active_reason():
    lines = [_row(2070, 2070, 800.0), _row(2055, 2070, 1390.5, cap="Active"), _row(2070, 2070, 900.0)]
    c = bench.summarize_clocks(lines)
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert c["power_w_max"] == 1390.5
    c = bench.summarize_clocks([_row(1500, 2070, 700.0, hwt="Active"), _row(1480, 2070, 700.0, hw="Active")])
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"] and c["sm_mhz"] == 1490


def test_clock_summary_skips_rows_that_do_not_parse():
    lines = ["\n", "0, [N/A], 2070, 10.0, 0x0, Not Active, Not Active, Not Active, Not Active\n", "garbage\n",
             _row(2070, 2070, 500.0)]
    c = bench.summarize_clocks(lines)
    assert c["samples"] == 1 and c["sm_mhz"] == 2070
    assert bench.summarize_clocks([])["reasons"] == ["no samples"]


def test_traffic_record_is_withheld_once_the_kernel_source_changes(monkeypatch):
    monkeypatch.setattr(bench, "filter_source_sha", lambda: "0" * 16)
    assert bench.recorded_traffic("single_row_2p28_pareto15_k1024", 1 << 28) is None


def test_traffic_record_scales_the_captured_bytes_per_element():
    row = bench.recorded_traffic("single_row_2p28_pareto15_k1024", 1 << 28)
    if row is None:
        pytest.skip("the committed capture predates the current filter source")
    # one read of 4-byte elements plus the survivors and stray dirty lines: no re-reads
    assert 4.0 * (1 << 28) <= row <= 4.05 * (1 << 28)
    batch = bench.recorded_traffic("batchtopk_4096x65536_relu_bf16_k131072", 1 << 28)
    assert batch is not None and 2.0 * (1 << 28) <= batch <= 2.05 * (1 << 28)
    assert bench.recorded_traffic("no_such_workload", 1 << 28) is None
