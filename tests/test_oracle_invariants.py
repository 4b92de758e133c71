"""Invariants of the scheduler oracle on every workload's scheduler inputs.

"Adaptive Verification in vLLM", *Scheduling the budget* and *The cost
model*: survival only decreases with position; the global top-B is a
contiguous prefix of every request; B maximises the objective; the cost table
in use is monotone.  Checked on the seven synthetic workloads plus random
edge shapes.
"""
import numpy as np
import pytest

import oracle
import workloads


def check_select_invariants(r, conf, mask, cost, T, flags):
    N, K = conf.shape
    s = r["survival"]
    assert np.all(np.diff(s, axis=1) <= 0)
    assert np.all(s[mask == 0] == 0)
    assert np.all((s >= 0) & (s <= 1))
    order = r["order"]
    assert len(order) == int(mask.sum()) * K
    # order sorted by survival desc, ties by slot id
    sv = s.reshape(-1)[order]
    assert np.all(np.diff(sv) <= 0)
    eq = np.diff(sv) == 0
    assert np.all(np.diff(order)[eq] > 0)
    B = r["B"]
    assert 0 <= B <= r["b_max"] <= len(order)
    assert r["b_max"] == max(0, min(len(order), len(cost) - 1 - T)) or T >= len(cost)
    # prefix-closed selection
    sel = np.zeros(N * K, bool)
    sel[order[:B]] = True
    sel = sel.reshape(N, K)
    for n in range(N):
        ln = r["draft_len"][n]
        assert sel[n, :ln].all() and not sel[n, ln:].any()
    assert r["draft_len"].sum() == B
    cu = r["cu_len"]
    assert cu[0] == 0 and cu[-1] == B and np.all(np.diff(cu) == r["draft_len"])
    vi = r["verify_idx"]
    assert len(vi) == B and np.all(np.diff(vi) > 0)
    f = r["f"]
    assert np.all(f[B] >= f[~np.isnan(f)]) if B or len(f) else True
    assert np.all(f[:B] < f[B])               # first maximiser
    if flags & oracle.FORCE_RUNNING_MAX:
        cu_ = r["cost_used"]
        assert np.all(np.diff(cu_) >= 0) and np.all(cu_ >= cost)


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_workload_invariants(name):
    cfg = workloads.get_config(name)
    d = workloads.make_select_inputs(cfg)
    flags = oracle.FORCE_RUNNING_MAX if cfg.cost_kind == "noisy" else 0
    r = oracle.select_step(d["conf"], d["mask"], d["cost"], d["T"], flags=flags)
    check_select_invariants(r, d["conf"], d["mask"], d["cost"], d["T"], flags)
    assert r["status"] == 0
    # the workloads' survival profile: first position >70%, last <10%
    # ("Adaptive Verification in vLLM", *The problem*) for the logit-normal
    # recipes
    if cfg.conf_kind == "logitnormal" and cfg.conf_request_offset_sd == 0:
        m = d["conf"].astype(np.float64)
        assert np.median(m[:, 0]) > 0.6
        assert np.median(r["survival"][d["mask"] == 1, -1]) < 0.1


def test_stress_table_needs_forcing():
    cfg = workloads.get_config("stress")
    d = workloads.make_select_inputs(cfg)
    assert np.any(np.diff(d["cost"]) < 0)
    f = oracle.force_monotone(d["cost"])
    assert np.all(np.diff(f) >= 0)


def test_random_edge_shapes():
    rng = np.random.default_rng(21)
    for trial in range(40):
        N = int(rng.integers(1, 40))
        K = int(rng.integers(1, 17))
        conf = rng.uniform(0, 1, size=(N, K)).astype(np.float32)
        conf[rng.uniform(size=(N, K)) < 0.1] = 1.0
        conf[rng.uniform(size=(N, K)) < 0.05] = 0.0
        mask = (rng.uniform(size=N) < 0.8).astype(np.uint8)
        L = int(rng.integers(2, 3 * N * K + 4))
        cost = np.sort(rng.uniform(1, 100, L)).astype(np.float32)
        T = int(rng.integers(0, L))
        r = oracle.select_step(conf, mask, cost, T)
        check_select_invariants(r, conf, mask, cost, T, 0)
