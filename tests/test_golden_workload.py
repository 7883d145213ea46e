"""The generated workloads carry the shapes and tolerance the pages print
(tests/golden/pages_workload.json)."""
import json
import os

import mla_inputs as mi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_workload.json")


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_tiny_and_mid_prefill_shapes_match_pages():
    g = load_golden()["isolated_forward"]
    for n, s in zip((1, 2), g["shapes_sq_eq_skv"]):
        idx = mi.prefill_indices(1000 + n, s, s)
        assert idx.shape == (s, g["topk"])
    c = mi.config(1)
    assert c.q.shape == (64, g["h_q"], g["d_qk"]) and c.kv.shape == (64, g["d_qk"])
    assert c.d_v == g["d_v"] == load_golden()["kv_constraints"]["value_dim"]


def test_tolerance_admits_reported_differences():
    g = load_golden()["isolated_forward"]
    assert all(d <= g["atol"] for d in g["max_abs_diff_reported"])
