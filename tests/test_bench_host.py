"""Host-side arithmetic of bench.py, without a GPU."""
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_projection_closed_forms():
    import bench
    # free drafts and a verify as costly as a dense step: the speedup is the
    # number of tokens committed per iteration
    p = bench.speedup_projection(0.7, 5, 0.0, 80.0, 20.0, 100.0)
    assert p["gamma"] == 0.0
    assert math.isclose(p["S_formula"], 0.7 * 5 + 1)
    tokens = sum(0.7 ** i for i in range(6))          # E[a + 1] under the prefix rule
    assert math.isclose(p["tokens_per_iteration_prefix_rule"], tokens)
    assert math.isclose(p["S_measured_prefix_rule"], tokens)
    # every draft accepted
    p = bench.speedup_projection(1.0, 4, 10.0, 30.0, 10.0, 40.0)
    assert p["tokens_per_iteration_prefix_rule"] == 5
    assert math.isclose(p["gamma"], 0.25)
    assert math.isclose(p["S_formula"], 5 / 2)
    assert math.isclose(p["S_measured_prefix_rule"], 5 * 40.0 / (4 * 10.0 + 40.0))
