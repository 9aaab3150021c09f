"""bench.py's clock record keeps only the nvidia-smi rows taken during the
timed region (host time stamps), so that an idle sample before or after the
timed steps can neither stand in for the clock under load nor hide a
throttle reason seen during them."""
import datetime
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(spec)
spec.loader.exec_module(bench)

BASE = datetime.datetime(2026, 1, 2, 3, 4, 5).timestamp()


def row(dt, mhz, hw_slow="Not Active", power_cap="Not Active"):
    ts = datetime.datetime.fromtimestamp(BASE + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return "%s, 0, %d, 2070, 900.00, 0x0, %s, Not Active, Not Active, %s\n" % (
        ts, mhz, hw_slow, power_cap)


def test_only_rows_inside_the_timed_region_count():
    lines = [row(0.00, 345, hw_slow="Active"),            # idle, before the region
             row(0.10, 2070), row(0.12, 2055, power_cap="Active"), row(0.14, 2070),
             row(0.30, 1200, hw_slow="Active")]            # after the region
    clk = bench.summarize_clock_rows(lines, BASE + 0.09, BASE + 0.15)
    assert clk["samples"] == 3 and clk["window"] == "timed region"
    assert clk["sm_mhz"] == 2070 and clk["sm_max_mhz"] == 2070
    assert clk["reasons"] == ["sw_power_cap"]


def test_a_region_shorter_than_the_sampling_period_uses_the_nearest_rows():
    lines = [row(0.00, 2070), row(0.02, 2040), row(0.50, 2070, hw_slow="Active")]
    clk = bench.summarize_clock_rows(lines, BASE + 0.005, BASE + 0.015)
    assert clk["window"] == "within 0.1 s of the timed region"
    assert clk["samples"] == 2 and clk["reasons"] == []
    assert bench.summarize_clock_rows(lines, BASE + 5.0, BASE + 5.01) is None


def test_malformed_rows_are_skipped():
    lines = ["", "garbage\n", row(0.1, 2070).replace("2026", "20x6"), row(0.1, 2070)]
    clk = bench.summarize_clock_rows(lines, BASE, BASE + 1.0)
    assert clk["samples"] == 1 and clk["sm_mhz"] == 2070
