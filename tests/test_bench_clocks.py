"""The clock record of the benchmark's timed region: nvidia-smi rows are parsed, only the
rows inside the timed window count, and every throttle reason seen there is reported
(a run that saw a hardware or thermal slowdown is rejected on that record)."""
import datetime

import bench


def _row(ts, sm, reasons=(), smax=2070):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ", ".join("Active" if n in reasons else "Not Active" for n in names)
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, 0, {sm}, {smax}, 700.00, 0x0000000000000000, {flags}\n"


T0 = datetime.datetime(2026, 12, 2, 13, 0, 0).timestamp()


def test_only_rows_inside_the_timed_window_count():
    lines = [_row(T0 - 2.0, 900, ("hw_slowdown",)),          # before the timed region
             _row(T0 + 0.1, 2070), _row(T0 + 0.2, 2055), _row(T0 + 0.3, 2070),
             _row(T0 + 5.0, 1200, ("sw_thermal_slowdown",))]  # after it
    got = bench.summarize_clock_samples(lines, T0, T0 + 0.35)
    assert got["samples_in_timed_region"] == 3 and got["samples"] == 3
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == []


def test_reasons_inside_the_window_are_reported():
    lines = [_row(T0 + 0.1, 2070), _row(T0 + 0.2, 1980, ("sw_power_cap",)),
             _row(T0 + 0.3, 1500, ("hw_slowdown", "sw_power_cap"))]
    got = bench.summarize_clock_samples(lines, T0, T0 + 1.0)
    assert got["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert got["sm_mhz"] == 1980


def test_no_row_in_the_window_falls_back_to_every_row():
    lines = [_row(T0 - 3.0, 2070), _row(T0 + 9.0, 2040)]
    got = bench.summarize_clock_samples(lines, T0, T0 + 1.0)
    assert got["samples_in_timed_region"] == 0 and got["samples"] == 2
    assert got["sm_mhz"] == 2055


def test_malformed_rows_are_skipped():
    lines = ["", "garbage\n", "a, b, c, d, e, f, g, h, i, j\n", _row(T0 + 0.1, 2070)]
    got = bench.summarize_clock_samples(lines, T0, T0 + 1.0)
    assert got["samples"] == 1 and got["sm_mhz"] == 2070


def test_the_record_of_a_real_sample_row_parses():
    line = ("2026/12/02 13:41:52.852, 0, 2070, 2070, 222.99, 0x0000000000000000, "
            "Not Active, Not Active, Not Active, Not Active\n")
    got = bench.summarize_clock_samples([line])
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 1,
                   "samples_in_timed_region": 0}
