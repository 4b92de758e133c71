"""GPU parity of stale sizing (dspark_select_step_stale, and the same thing
composed from the separate scheduler calls) against the oracle, bit for bit.

"Adaptive Verification in vLLM", *Scheduling the budget*, last paragraph: B
is sized from a confidence buffer one step old while the B slots are handed
to requests by current confidences; "How DSpark Speeds Up LLM Inference",
appendix Part B: capacity from confidences two steps earlier.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _both(conf_size, conf, mask, cost, T, draft_cost=0.0, flags=0, draft=None):
    from gpu_harness import run_select, check_select
    for fused in (True, False):
        got = run_select(conf, mask, cost, T, draft_cost, flags, draft,
                         fused=fused, conf_size=conf_size)
        r = check_select(got, conf, mask, cost, T, draft_cost, flags, draft,
                         conf_size=conf_size)
    return r


def test_w3_stale_sizing():
    with open(os.path.join(GOLD, "w3_stale_sizing.json")) as f:
        g = json.load(f)
    r = _both(np.array(g["conf_size"], np.float32), np.array(g["conf"], np.float32),
              np.array(g["mask"], np.uint8), np.array(g["cost"], np.float32), g["T"])
    assert r["B"] == g["expected"]["B"]
    assert r["draft_len"].tolist() == g["expected"]["draft_len"]


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
@pytest.mark.parametrize("steps_back", [1, 2])
def test_workload(name, steps_back):
    cfg = workloads.get_config(name)
    d = workloads.make_select_inputs(cfg)
    old = workloads.make_stale_confidences(cfg, steps_back)
    flags = oracle.FORCE_RUNNING_MAX if cfg.cost_kind == "noisy" else 0
    rng = np.random.default_rng(cfg.seed)
    draft = rng.integers(0, cfg.vocab, size=(cfg.N, cfg.K)).astype(np.int32)
    _both(old, d["conf"], d["mask"], d["cost"], d["T"], 0.0, flags, draft)


def test_same_buffer_equals_plain_select():
    from gpu_harness import run_select
    cfg = workloads.get_config("headline")
    d = workloads.make_select_inputs(cfg)
    a = run_select(d["conf"], d["mask"], d["cost"], d["T"], flags=1)
    b = run_select(d["conf"], d["mask"], d["cost"], d["T"], flags=1,
                   conf_size=d["conf"])
    for k in a:
        np.testing.assert_array_equal(np.asarray(a[k]), np.asarray(b[k]), err_msg=k)


@pytest.mark.parametrize("N,K", [(1, 32), (512, 32), (16384, 1), (1000, 15)])
def test_sizes_and_flags(N, K):
    rng = np.random.default_rng(N * 7 + K)
    conf = rng.uniform(0, 1, (N, K)).astype(np.float32) ** 0.3
    old = rng.uniform(0, 1, (N, K)).astype(np.float32) ** 0.5
    mask = (rng.uniform(size=N) < 0.9).astype(np.uint8)
    L = N * K + 50
    cost = (100 + 0.01 * np.arange(L) * rng.uniform(0.99, 1.01, L)).astype(np.float32)
    T = int(rng.integers(0, 40))
    for flags in (0, oracle.FORCE_RUNNING_MAX, oracle.BUDGET_GREEDY_STOP | 1):
        _both(old, conf, mask, cost, T, 0.5, flags)


def test_out_of_range_old_buffer_sets_status():
    rng = np.random.default_rng(3)
    conf = rng.uniform(0, 1, (16, 4)).astype(np.float32)
    old = rng.uniform(0, 1, (16, 4)).astype(np.float32)
    old[2, 1] = np.nan
    old[5, 0] = 1.5
    cost = (10 + np.arange(80)).astype(np.float32)
    r = _both(old, conf, None, cost, 2)
    assert r["status"] & oracle.CONF_OOR


def test_random_shapes_and_ties():
    """Random batch shapes, masks, T and flags, with an older confidence
    buffer that is either an independent draw or the current one with a
    few entries changed (tie-heavy values in half the cases): every output
    equals the oracle's bit for bit."""
    rng = np.random.default_rng(31337)
    vals = np.array([1.0, 0.5, 0.25, 0.75, 0.0, 0.125], np.float32)
    for case in range(16):
        K = int(rng.integers(1, 33))
        N = int(rng.integers(1, 16384 // K + 1))
        if rng.uniform() < 0.5:
            conf = vals[rng.integers(0, len(vals), (N, K))]
            old = vals[rng.integers(0, len(vals), (N, K))]
        else:
            conf = rng.uniform(0, 1, (N, K)).astype(np.float32) ** rng.uniform(0.2, 3.0)
            old = conf.copy()
            pick = rng.uniform(size=(N, K)) < 0.1
            old[pick] = rng.uniform(0, 1, int(pick.sum())).astype(np.float32)
        mask = (rng.uniform(size=N) < rng.uniform(0.3, 1.0)).astype(np.uint8)
        L = int(rng.integers(8, N * K + 64))
        cost = (100 + rng.uniform(0, 2, L).cumsum()).astype(np.float32)
        T = int(rng.integers(0, L))
        flags = int(rng.choice([0, oracle.FORCE_RUNNING_MAX]))
        _both(old, conf, mask, cost, T, 0.0, flags)
