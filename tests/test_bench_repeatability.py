"""The benchmark's repeatability summary (pure host arithmetic): the timed
steps cut into consecutive runs, the median run mean and the slowest / fastest
run ratio, flagged when above 1.05."""
import importlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    return importlib.import_module("bench")


def test_steady_times_are_reportable():
    r = _bench().repeatability([0.066] * 400)
    assert r == {"repeats": 5, "median_ms": 0.066, "spread": 1.0, "reportable": True}


def test_a_slow_run_is_flagged():
    times = [0.066] * 320 + [0.080] * 80  # the last fifth 21 % slower
    r = _bench().repeatability(times)
    assert r["repeats"] == 5 and r["median_ms"] == 0.066
    assert abs(r["spread"] - 0.080 / 0.066) < 1e-3 and r["reportable"] is False


def test_few_steps_and_no_steps():
    b = _bench()
    assert b.repeatability([0.05, 0.07])["repeats"] == 2
    assert b.repeatability([0.05])["spread"] == 1.0
    assert b.repeatability([]) == {"repeats": 0, "median_ms": None, "spread": None, "reportable": False}
    r = b.repeatability([0.05] * 7)  # 7 steps into 5 runs: the last run takes the remainder
    assert r["repeats"] == 5 and r["spread"] == 1.0
