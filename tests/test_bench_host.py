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


def test_algorithmic_bytes_hand_count():
    """Bytes of one step counted by hand on a tiny shape: every K and V row of
    the prefix and the verify block once, Q and O, the capture written by
    verify and read by select, the selected rows plus the growing tail for
    every draft step, and the index list per draft step."""
    import bench
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec(batch=1, prefix_lens=(100,), num_q_heads=4, num_kv_heads=2, head_dim=64,
                      n_drafts=2, top_k=8, n_sink=2, n_recent=4)
    nb = bench.algorithmic_bytes(spec)
    R, row = 3, 2 * 64 * 2 * 2                      # verify rows; K+V bytes of one position
    assert nb["verify_kv"] == (100 + R) * row
    q_o = 2 * R * 4 * 64 * 2
    cap = 100 * 2 * 4
    assert nb["verify"] == (100 + R) * row + q_o + cap
    n_sel = 2 + 4 + 8
    assert nb["select"] == cap + n_sel * 4
    drafts = (n_sel + 1) * row + (n_sel + 2) * row + 2 * 2 * 4 * 64 * 2 + 2 * n_sel * 4
    assert nb["drafts"] == drafts
    assert nb["step"] == nb["verify"] + nb["select"] + nb["drafts"]


def test_summary_fractions():
    """The line's step and roofline fractions are bytes / time / peak."""
    import bench
    from self_speculative_sparse_vg_gb300.workloads import small_spec
    spec = small_spec()
    nb = bench.algorithmic_bytes(spec)
    m = {"value": 50.0, "graph_full_us": 80.0, "graph_flush_us": 30.0,
         "stages_graph_us": {"verify": 30.0, "select": 5.0, "drafts_total": 15.0},
         "stages_us": {"verify": 32.0, "select": 6.0, "drafts_total": 18.0},
         "events_us_per_step": 56.0}
    r = bench.summarize(spec, m, 1000.0, "measured", 7)
    assert math.isclose(r["hbm_frac_step"], nb["step"] / 50e-6 / 1e9 / 1000.0)
    assert math.isclose(r["hbm_frac_step_events"], nb["step"] / 56e-6 / 1e9 / 1000.0)
    assert math.isclose(r["roofline"]["frac"], nb["verify"] / 32e-6 / 1e9 / 1000.0)
    assert math.isclose(r["gap_to_0.70_us"], 50.0 - nb["step"] / (0.7 * 1000.0 * 1e9) * 1e6)
    assert r["launches_per_step"] == 7
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r["roofline"]
