"""Host-side check of bench.py's clock summary: only samples inside the
timed region count, and a region shorter than the sampling interval takes
the next sample (no GPU needed)."""
import datetime
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _line(ts, mhz, cap="Not Active", therm="Not Active"):
    return (f"{ts.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, {mhz}, 2032, 900.0, 0x0, "
            f"Not Active, Not Active, {therm}, {cap}\n")


def test_samples_outside_the_timed_region_are_ignored():
    b = _bench()
    clk = b.ClockSampler(0)
    t = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    clk.lines = [_line(t, 1000, cap="Active"),           # before the region
                 _line(t + 200 * ms, 2000),
                 _line(t + 220 * ms, 2010),
                 _line(t + 240 * ms, 2020),
                 _line(t + 900 * ms, 1100, therm="Active")]  # after it
    clk.t0, clk.t1 = t + 190 * ms, t + 250 * ms
    s = clk.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2010
    assert s["reasons"] == []


def test_short_region_takes_the_next_sample():
    b = _bench()
    clk = b.ClockSampler(0)
    t = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    clk.lines = [_line(t, 1500), _line(t + 100 * ms, 1990, cap="Active")]
    clk.t0, clk.t1 = t + 30 * ms, t + 40 * ms
    s = clk.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 1990 and s["reasons"] == ["sw_power_cap"]
