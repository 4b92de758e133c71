"""Brute force over every slot subset and every budget on 3 x 7 instances.

"Adaptive Verification in vLLM", *Scheduling the budget*: for a budget B the
most probable draft sequences are the global top-B of survival, which is a
contiguous prefix of every request; B maximises (N_sampling + expected
accepted drafts) / cost[T + B].  Here the best subset of each size is found by
enumerating all 2^21 subsets, and the best budget by scanning all sizes,
without any sorting; the oracle must agree.
"""
import numpy as np
import pytest

import oracle
import workloads


def _all_subset_sums(x):
    sums = np.zeros(1)
    cnt = np.zeros(1, dtype=np.int8)
    for v in x:
        sums = np.concatenate([sums, sums + v])
        cnt = np.concatenate([cnt, cnt + 1])
    return sums, cnt


def _prefix_closed(bits, N, K):
    for n in range(N):
        row = [(bits >> (n * K + k)) & 1 for k in range(K)]
        seen_zero = False
        for b in row:
            if b and seen_zero:
                return False
            seen_zero |= not b
    return True


def _instances():
    w1 = workloads.w1_instance()
    yield "w1", w1["conf"], w1["cost"], w1["T"]
    tiny = workloads.make_select_inputs(workloads.get_config("tiny"))
    yield "tiny", tiny["conf"], tiny["cost"], tiny["T"]
    rng = np.random.default_rng(123)
    for i in range(3):
        conf = rng.uniform(0.05, 1.0, size=(3, 7)).astype(np.float32)
        # a staircase with a jump so the objective is not unimodal
        n = np.arange(64)
        cost = np.where(n <= 16, 10 + 0.8 * (1 << np.ceil(np.log2(np.maximum(n, 1))).astype(int)),
                        1.6 * (10 + 0.8 * n)).astype(np.float32)
        yield f"rand{i}", conf, cost, 3 + i


@pytest.mark.parametrize("name,conf,cost,T", list(_instances()))
def test_bruteforce_topb_and_budget(name, conf, cost, T):
    N, K = conf.shape
    mask = np.ones(N, np.uint8)
    r = oracle.select_step(conf, mask, cost, T)
    s = r["survival"].reshape(-1)
    sums, cnt = _all_subset_sums(s)
    S = N * K
    best_sum = np.array([sums[cnt == b].max() for b in range(S + 1)])
    # 1) the oracle's prefix sums are the best achievable sum of every size
    np.testing.assert_allclose(r["prefix"], best_sum, rtol=1e-13, atol=0)
    # 2) for every size, some maximal subset is prefix-closed, and the
    #    oracle's own top-b set is one of the maximisers
    for b in range(S + 1):
        idx = np.nonzero((cnt == b) & (sums >= best_sum[b] * (1 - 1e-13)))[0]
        assert any(_prefix_closed(int(i), N, K) for i in idx), (name, b)
        top = 0
        for slot in r["order"][:b]:
            top |= 1 << int(slot)
        assert _prefix_closed(top, N, K)
        assert sums[top] >= best_sum[b] * (1 - 1e-13)
    # 3) the budget found by scanning every size equals the oracle's B
    L = len(cost)
    bmax = min(S, L - 1 - T)
    f = [(N + best_sum[b]) / float(cost[T + b]) for b in range(bmax + 1)]
    assert int(np.argmax(f)) == r["B"], name
    # 4) and allocation follows from the chosen top-B set
    assert r["draft_len"].sum() == r["B"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bruteforce_stale_sizing(seed):
    """Stale sizing ("Adaptive Verification in vLLM", *Scheduling the budget*,
    last paragraph): B is the best budget for the old survivals (every subset
    enumerated), and the allocated set is a best subset of that size for the
    current survivals."""
    rng = np.random.default_rng(500 + seed)
    N, K, T = 3, 6, 2
    old = rng.uniform(0.05, 1.0, size=(N, K)).astype(np.float32)
    cur = rng.uniform(0.05, 1.0, size=(N, K)).astype(np.float32)
    n = np.arange(48)
    cost = (10 + 0.8 * n + np.where(n > 9, 6.0, 0.0)).astype(np.float32)
    mask = np.ones(N, np.uint8)
    r = oracle.select_step_stale(old, cur, mask, cost, T)
    s_old = np.cumprod(old.astype(np.float64), axis=1).reshape(-1)
    s_cur = np.cumprod(cur.astype(np.float64), axis=1).reshape(-1)
    sums_o, cnt = _all_subset_sums(s_old)
    sums_c, _ = _all_subset_sums(s_cur)
    S = N * K
    best_o = np.array([sums_o[cnt == b].max() for b in range(S + 1)])
    bmax = min(S, len(cost) - 1 - T)
    f = [(N + best_o[b]) / float(cost[T + b]) for b in range(bmax + 1)]
    assert int(np.argmax(f)) == r["B"]
    sel = 0
    for nn in range(N):
        for k in range(int(r["draft_len"][nn])):
            sel |= 1 << (nn * K + k)
    assert bin(sel).count("1") == r["B"]
    best_c = sums_c[cnt == r["B"]].max()
    assert sums_c[sel] >= best_c * (1 - 1e-13)
    assert _prefix_closed(sel, N, K)
