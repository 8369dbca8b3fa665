"""Host-side logic of bench.py: the clock record is taken from the samples
inside the timed region."""
import datetime
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _line(t, mhz, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, {thermal}, {power_cap}"


def test_clock_summary_keeps_samples_inside_the_timed_region():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.5, 2070), _line(t0 + 0.01, 1900, power_cap="Active"), _line(t0 + 0.03, 1880),
             _line(t0 + 0.05, 1890), _line(t0 + 1.0, 2070, thermal="Active")]
    c = bench.summarize_clocks(lines, [t0, t0 + 0.06], 20)
    assert c["samples"] == 3 and c["sm_mhz"] == 1890
    assert c["reasons"] == ["sw_power_cap"] and c["from"] == "timed region"
    assert c["sm_max_mhz"] == 2070


def test_clock_summary_short_region_takes_the_nearest_sample():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.2, 2070), _line(t0 + 0.15, 1950), _line(t0 + 0.4, 2070)]
    c = bench.summarize_clocks(lines, [t0 + 0.1, t0 + 0.101], 20)
    assert c["samples"] == 1 and c["sm_mhz"] == 1950 and c["from"].startswith("nearest")


def test_clock_summary_ignores_malformed_lines():
    assert bench.summarize_clocks(["", "garbage", "a, b"], [0.0, 1.0], 20) is None


def test_kernel_hash_ignores_comments_only():
    code = "int a = 1; // a comment\n/* block\n comment */ float b;"
    assert bench._code_only(code) == bench._code_only("int a = 1;\nfloat   b;")
    assert bench._code_only(code) != bench._code_only("int a = 2; float b;")
