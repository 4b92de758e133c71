"""Pins of the scheduler oracle on hand-worked instances (tests/golden/).

W1 follows the vLLM blog's Figure 1 caption ("Adaptive Verification in
vLLM", *Scheduling the budget*): 3 requests x 7 slots, best B = 11.
W2 is built with exact binary values so that a wrong cost index, a wrong
N_sampling or an eligible prefill request each changes B.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_w1_fig1_best_b_is_11():
    g = _load("w1_fig1_b11.json")
    d = workloads.w1_instance()
    np.testing.assert_array_equal(d["conf"], np.array(g["conf"], np.float32))
    r = oracle.select_step(d["conf"], d["mask"], d["cost"], d["T"])
    e = g["expected"]
    assert r["B"] == e["B"]
    assert r["draft_len"].tolist() == e["draft_len"]
    assert r["cu_len"].tolist() == e["cu_len"]
    assert r["verify_idx"].tolist() == e["verify_idx"]
    assert r["order"][:12].tolist() == e["first_sorted"]
    tol = g["rel_tol_values"]
    assert r["prefix"][11] == pytest.approx(e["P_11"], rel=tol)
    for b in (10, 11, 12):
        assert r["f"][b] == pytest.approx(e[f"f_{b}"], rel=tol)
    # B is the unique maximiser
    f = r["f"]
    assert np.sum(f == f.max()) == 1


def test_w2_cost_index_and_sampling_count():
    g = _load("w2_cost_index.json")
    conf = np.array(g["conf"], np.float32)
    mask = np.array(g["mask"], np.uint8)
    cost = np.array(g["cost"], np.float32)
    r = oracle.select_step(conf, mask, cost, g["T"])
    e = g["expected"]
    assert r["n_sampling"] == e["n_sampling"]
    assert r["order"].tolist() == e["order"]
    assert r["B"] == e["B"]
    # every f value is exact in binary except 3/4.3125 and 3.25/6, which are
    # single correctly-rounded divisions
    np.testing.assert_array_equal(r["f"], np.array(e["f"]))
    assert r["draft_len"].tolist() == e["draft_len"]
    assert r["cu_len"].tolist() == e["cu_len"]
    assert r["verify_idx"].tolist() == e["verify_idx"]


def test_w2_mistakes_would_change_b():
    """The instance discriminates the readings it is meant to pin."""
    g = _load("w2_cost_index.json")
    cost = np.array(g["cost"], np.float64)
    s_sorted = np.array([0.5, 0.25, 0.25, 0.25])
    P = np.concatenate([[0.0], np.cumsum(s_sorted)])

    def best(ns, shift):
        T = g["T"]
        bmax = min(4, g["L"] - 1 - T - max(shift, 0))
        f = [(ns + P[b]) / cost[T + b + shift] for b in range(bmax + 1)]
        return int(np.argmax(f))

    assert best(2, 0) == 3
    assert best(2, -1) != 3
    assert best(2, +1) != 3
    assert best(3, 0) != 3


def test_table_edges():
    d = workloads.w1_instance()
    L = len(d["cost"])
    r = oracle.select_step(d["conf"], d["mask"], d["cost"], L - 1)
    assert r["B"] == 0 and r["b_max"] == 0 and r["status"] == 0
    r = oracle.select_step(d["conf"], d["mask"], d["cost"], L)
    assert r["B"] == 0 and r["status"] & oracle.TABLE_SHORT
    r = oracle.select_step(d["conf"], d["mask"], d["cost"], -1)
    assert r["B"] == 0 and r["status"] & oracle.TABLE_SHORT
    # b_max clipped by the table, not by the slots
    r = oracle.select_step(d["conf"], d["mask"], d["cost"], L - 5)
    assert r["b_max"] == 4 and r["B"] <= 4


def test_w3_stale_sizing():
    """B from the old buffer, allocation by the current order (W3)."""
    g = _load("w3_stale_sizing.json")
    conf_size = np.array(g["conf_size"], np.float32)
    conf = np.array(g["conf"], np.float32)
    mask = np.array(g["mask"], np.uint8)
    cost = np.array(g["cost"], np.float32)
    r = oracle.select_step_stale(conf_size, conf, mask, cost, g["T"])
    e = g["expected"]
    assert r["B"] == e["B"]
    np.testing.assert_array_equal(r["f"], np.array(e["f"]))
    assert r["order"].tolist() == e["order"]
    assert r["draft_len"].tolist() == e["draft_len"]
    assert r["cu_len"].tolist() == e["cu_len"]
    assert r["verify_idx"].tolist() == e["verify_idx"]
    # the two wrong readings the instance separates
    cur = oracle.select_step(conf, mask, cost, g["T"])
    assert cur["B"] == g["if_sized_from_current"]["B"]
    assert cur["draft_len"].tolist() == g["if_sized_from_current"]["draft_len"]
    old = oracle.select_step(conf_size, mask, cost, g["T"])
    assert old["draft_len"].tolist() == g["if_allocated_by_old_order"]["draft_len"]


def test_w4_draft_cost():
    """The drafter's cost is one fp32 constant added to every candidate
    budget's step cost ("Adaptive Verification in vLLM", *The cost model*:
    the verification and drafter tables are summed).  W4 is built so that
    this reading gives B = 2 through an exact tie of f(2) and f(3)."""
    g = _load("w4_draft_cost.json")
    conf = np.array(g["conf"], np.float32)
    mask = np.array(g["mask"], np.uint8)
    cost = np.array(g["cost"], np.float32)
    np.testing.assert_array_equal(cost.astype(np.float64), np.array(g["cost"]))
    r = oracle.select_step(conf, mask, cost, g["T"], draft_cost=g["draft_cost"])
    e = g["expected"]
    assert r["B"] == e["B"]
    np.testing.assert_array_equal(r["f"], np.array(e["f"]))
    assert r["objective"] == e["objective"]
    assert r["draft_len"].tolist() == e["draft_len"]
    assert r["cu_len"].tolist() == e["cu_len"]
    assert r["verify_idx"].tolist() == e["verify_idx"]
    # the drafter cost matters: without it the budget differs
    r0 = oracle.select_step(conf, mask, cost, g["T"], draft_cost=0.0)
    assert r0["B"] == g["wrong_readings_B"]["no_draft_cost"]


def test_w4_mistakes_would_change_b():
    """Each wrong reading of the drafter cost gives another B on W4, computed
    here in exact rationals (independent of the oracle's float path)."""
    from fractions import Fraction as Fr
    g = _load("w4_draft_cost.json")
    T = g["T"]
    cost = [Fr(c) for c in g["cost"]]
    s = [Fr(1), Fr(1), Fr(3, 4)]
    P = [Fr(0), s[0], s[0] + s[1], s[0] + s[1] + s[2]]
    c32 = Fr(11744051, 1 << 24)
    assert float(c32) == float(np.float32(g["draft_cost"]))

    def first_argmax(f):
        return f.index(max(f))

    def B(num, den):
        return first_argmax([num(b) / den(b) for b in range(4)])

    n = lambda b: 1 + P[b]  # noqa: E731
    assert B(n, lambda b: cost[T + b] + c32) == g["expected"]["B"]
    w = g["wrong_readings_B"]
    assert B(n, lambda b: cost[T + b]) == w["no_draft_cost"]
    assert B(lambda b: n(b) + c32, lambda b: cost[T + b]) == w["in_numerator"]
    assert B(n, lambda b: cost[T + b] + (c32 if b == 0 else 0)) == w["added_once_to_b0"]
    assert B(n, lambda b: cost[T + b] + b * c32) == w["per_drafted_token"]
    assert B(n, lambda b: cost[T + b] + Fr(g["draft_cost"])) == w["kept_in_fp64"]
    for v in w.values():
        assert v != g["expected"]["B"]
