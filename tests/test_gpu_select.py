"""GPU parity of the scheduler calls against the oracle, bit for bit.

"Adaptive Verification in vLLM", *Scheduling the budget* and *The cost
model*.  Every output (survival, order, exact prefix sums, B, objective,
lengths, offsets, verify list, status bits) must equal the oracle's.
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


def _both(conf, mask, cost, T, draft_cost=0.0, flags=0, draft=None):
    from gpu_harness import run_select, check_select
    for fused in (True, False):
        got = run_select(conf, mask, cost, T, draft_cost, flags, draft, fused=fused)
        r = check_select(got, conf, mask, cost, T, draft_cost, flags, draft)
    return r


def test_w1_fig1():
    d = workloads.w1_instance()
    r = _both(d["conf"], d["mask"], d["cost"], d["T"])
    assert r["B"] == 11


def test_w2_cost_index():
    with open(os.path.join(GOLD, "w2_cost_index.json")) as f:
        g = json.load(f)
    r = _both(np.array(g["conf"], np.float32), np.array(g["mask"], np.uint8),
              np.array(g["cost"], np.float32), g["T"])
    assert r["B"] == g["expected"]["B"]


def test_w4_draft_cost():
    """The drafter cost on the device: fp32 constant in every denominator,
    B = 2 through an exact tie of f(2) and f(3) (first index wins)."""
    with open(os.path.join(GOLD, "w4_draft_cost.json")) as f:
        g = json.load(f)
    r = _both(np.array(g["conf"], np.float32), np.array(g["mask"], np.uint8),
              np.array(g["cost"], np.float32), g["T"], g["draft_cost"])
    assert r["B"] == g["expected"]["B"]
    assert r["objective"] == g["expected"]["objective"]


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_workload(name):
    cfg = workloads.get_config(name)
    d = workloads.make_select_inputs(cfg)
    flags = oracle.FORCE_RUNNING_MAX if cfg.cost_kind == "noisy" else 0
    rng = np.random.default_rng(cfg.seed)
    draft = rng.integers(0, cfg.vocab, size=(cfg.N, cfg.K)).astype(np.int32)
    _both(d["conf"], d["mask"], d["cost"], d["T"], 0.0, flags, draft)


def test_stress_table_forced_by_prep_call():
    import torch
    from gpu_harness import up
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    cfg = workloads.get_config("stress")
    d = workloads.make_select_inputs(cfg)
    for mode in (D.COST_FORCE_MONOTONE, D.COST_FORCE_SUFFIX_MIN):
        c = up(d["cost"])
        out = torch.empty_like(c)
        D.dspark_force_monotone(c, out, mode)
        D.dspark_force_monotone(c, c, mode)            # in place
        torch.cuda.synchronize()
        want = oracle.force_monotone(d["cost"], mode)
        np.testing.assert_array_equal(out.cpu().numpy(), want)
        np.testing.assert_array_equal(c.cpu().numpy(), want)
    forced = oracle.force_monotone(d["cost"])
    _both(d["conf"], d["mask"], forced, d["T"])


@pytest.mark.parametrize("flags", [0, 1, 2, 4, 5, 6])
def test_flags_on_staircase(flags):
    cfg = workloads.get_config("dsv4")
    d = workloads.make_select_inputs(cfg)
    cost = d["cost"].copy()
    rng = np.random.default_rng(77)
    cost *= rng.uniform(0.97, 1.03, size=cost.shape).astype(np.float32)
    for T in (0, 100, 2288, 4000, 8000):
        _both(d["conf"], d["mask"], cost, T, 1.5, flags)


def test_edges():
    rng = np.random.default_rng(5)
    cost = (10 + 0.5 * np.arange(64)).astype(np.float32)
    conf = rng.uniform(0, 1, (3, 7)).astype(np.float32)
    for T in (-5, 0, 62, 63, 64, 1000):             # table edges
        _both(conf, None, cost, T)
    _both(conf, np.zeros(3, np.uint8), cost, 3)       # nobody samples
    _both(conf[:1], None, cost, 3)                   # one request
    _both(conf[:, :1], None, cost, 3)                # K = 1
    bad = conf.copy()
    bad[0, 1] = np.nan
    bad[1, 2] = 1.5
    bad[2, 0] = -0.25
    bad[2, 3] = -0.0
    _both(bad, None, cost, 3)                         # clamped + flagged
    ones = conf.copy()
    ones[:, 2:5] = 1.0                                # survival ties
    _both(ones, None, cost, 3)
    zcost = cost.copy()
    zcost[10] = 0.0
    zcost[12] = -1.0
    _both(conf, None, zcost, 3)                       # non-positive cost
    ncost = cost.copy()
    ncost[9] = np.nan
    for fl in (0, 1, 2, 4):
        _both(conf, None, ncost, 3, 0.0, fl)          # NaN cost


@pytest.mark.parametrize("N,K", [(1, 32), (512, 32), (16384, 1), (2048, 8),
                                 (1000, 15), (37, 3)])
def test_sizes(N, K):
    rng = np.random.default_rng(N * 100 + K)
    conf = rng.uniform(0, 1, (N, K)).astype(np.float32) ** 0.3
    conf[rng.uniform(size=(N, K)) < 0.02] = 1.0
    mask = (rng.uniform(size=N) < 0.9).astype(np.uint8)
    L = N * K + 50
    base = 100 + 0.01 * np.arange(L)
    cost = (base * rng.uniform(0.99, 1.01, L)).astype(np.float32)
    T = int(rng.integers(0, 40))
    _both(conf, mask, cost, T, 0.0, oracle.FORCE_RUNNING_MAX)


@pytest.mark.parametrize("N,K", [(2048, 8), (1024, 15), (16384, 1), (5, 32)])
def test_cross_request_ties(N, K):
    """Survivals from a handful of exactly repeated values across thousands
    of requests, all-equal and all-zero confidences: the global order must
    break every tie by slot id, as the oracle's stable sort does."""
    rng = np.random.default_rng(N + 7 * K)
    vals = np.array([1.0, 0.5, 0.25, 0.75, 0.0], np.float32)
    conf = vals[rng.integers(0, 5, (N, K))]
    conf[rng.uniform(size=(N, K)) < 0.5] = 1.0
    mask = (rng.uniform(size=N) < 0.8).astype(np.uint8)
    L = N * K + 50
    cost = (100 + 0.01 * np.arange(L)).astype(np.float32)
    _both(conf, mask, cost, 7, 0.0, oracle.FORCE_RUNNING_MAX)
    _both(np.ones((N, K), np.float32), None, cost, 7)
    _both(np.zeros((N, K), np.float32), mask, cost, 7)


def test_random_shapes_and_ties():
    """Random batch shapes (N*K up to 16384, K up to 32) with tie-heavy and
    continuous confidences, random masks, T and flags: every output equals
    the oracle's bit for bit."""
    rng = np.random.default_rng(2027)
    for case in range(24):
        K = int(rng.integers(1, 33))
        N = int(rng.integers(1, 16384 // K + 1))
        if rng.uniform() < 0.5:
            vals = np.array([1.0, 0.5, 0.25, 0.75, 0.0, 0.125], np.float32)
            conf = vals[rng.integers(0, len(vals), (N, K))]
        else:
            conf = rng.uniform(0, 1, (N, K)).astype(np.float32) ** rng.uniform(0.2, 3.0)
        mask = (rng.uniform(size=N) < rng.uniform(0.3, 1.0)).astype(np.uint8)
        L = int(rng.integers(8, N * K + 64))
        cost = (100 + rng.uniform(0, 2, L).cumsum()).astype(np.float32)
        T = int(rng.integers(0, L))
        flags = int(rng.choice([0, oracle.FORCE_RUNNING_MAX]))
        _both(conf, mask, cost, T, 0.0, flags)


def test_survivals_equal_in_fp32_but_not_in_fp64():
    """Survivals that differ in fp64 but round to the same fp32 value must
    still be ordered by their fp64 values (then slot).  Request 1's second
    survival, (1 - 2^-24)^2 = 1 - 2^-23 + 2^-48, rounds to the fp32 value of
    request 0's survivals, 1 - 2^-23, yet is larger and has a larger slot id;
    a larger random batch repeats the pattern with confidences a few ulps
    below 1."""
    a = np.float32(1.0 - 2.0 ** -23)
    b = np.float32(1.0 - 2.0 ** -24)
    conf = np.array([[a, 1.0], [b, b]], np.float32)
    cost = (10.0 + 0.5 * np.arange(16)).astype(np.float32)
    r = _both(conf, None, cost, 2)
    assert r["order"].tolist() == [2, 3, 0, 1]
    rng = np.random.default_rng(99)
    for N, K in ((300, 6), (256, 7), (600, 6), (1200, 6), (1500, 6)):
        ulps = rng.integers(0, 6, (N, K))
        conf = (1.0 - ulps * 2.0 ** -24).astype(np.float32)
        conf[rng.uniform(size=(N, K)) < 0.3] = np.float32(0.5)
        cost = (10.0 + 0.5 * np.arange(N * K + 8)).astype(np.float32)
        _both(conf, None, cost, N)


def test_survival_products_through_the_subnormal_range():
    """Products that round inside the fp64 subnormal range and underflow to
    zero, fp32 subnormal confidences, and survivals whose fp32 copies are
    fp32 subnormals: survivals, order, sums and selection equal the
    oracle's bit for bit (the products are IEEE multiplies rounded to
    nearest even, the copies IEEE conversions), in a batch of 3072 slots
    and one of 6144 (the kernel converts between fp32 and fp64 on the fp64
    pipe below 4096 slots and in integer arithmetic from there)."""
    rng = np.random.default_rng(31)
    K = 32
    for N in (96, 192):
        m = N // 3
        conf = rng.uniform(0.5, 1.0, (N, K)).astype(np.float32)
        # 2^-1008 after eight factors, then down through the subnormals
        # (2^-1022 .. 2^-1074) with rounding at every step
        conf[:m, :8] = np.float32(2.0 ** -126)
        conf[:m, 8:] = (2.0 ** rng.uniform(-12, 0, (m, K - 8))).astype(np.float32)
        # an fp32 subnormal first factor
        sub = rng.integers(1, 1 << 23, m).astype(np.uint32).view(np.float32)
        conf[m:2 * m, 0] = sub
        conf[m:2 * m, 1:] = rng.uniform(0.01, 1.0, (m, K - 1)).astype(np.float32)
        # survivals near 2^-140, whose fp32 copies are subnormal
        conf[2 * m:, 0] = (2.0 ** -60 * rng.uniform(1, 2, N - 2 * m)).astype(np.float32)
        conf[2 * m:, 1] = (2.0 ** -80 * rng.uniform(1, 2, N - 2 * m)).astype(np.float32)
        conf[2 * m:, 2:] = rng.uniform(0.3, 1.0, (N - 2 * m, K - 2)).astype(np.float32)
        # the cases are reached: fp64 subnormal products, products that
        # underflow to zero, and fp32 subnormal copies
        p = np.asarray(oracle.survival(conf, None)[0], np.float64)
        assert np.any((p > 0) & (p < 2.0 ** -1022)) and np.any(p == 0)
        f = p.astype(np.float32)
        assert np.any((f > 0) & (f < np.float32(2.0 ** -126)))
        cost = (5 + 0.001 * np.arange(N * K + 8)).astype(np.float32)
        _both(conf, None, cost, 1)


def test_tiny_survivals_exact_sums():
    """Survivals spanning hundreds of binary orders of magnitude (the wide
    fixed-point sums), in a small batch and in one of 15360 slots; and a
    batch of that size within 2^61 of its largest survival (the narrow
    sums)."""
    rng = np.random.default_rng(8)
    conf = rng.uniform(0, 1, (64, 32)).astype(np.float32) ** 8
    conf[:4, :] = 1e-30
    cost = (5 + 0.001 * np.arange(4096)).astype(np.float32)
    _both(conf, None, cost, 1)
    cost = (5 + 0.001 * np.arange(16384)).astype(np.float32)
    for power, wide in ((6.0, True), (0.25, False)):
        conf = rng.uniform(0, 1, (1024, 15)).astype(np.float32) ** power
        p = np.asarray(oracle.survival(conf, None)[0], np.float64)
        nz = p[p > 0]
        assert (nz.min() < nz.max() * 2.0 ** -61) == wide
        _both(conf, None, cost, 1)


def test_scheduler_alongside_chain_then_gather():
    """The scheduler runs on a second stream while the chain runs, without
    the draft; after the join dspark_gather_verify_tokens fills the verify
    tokens.  Results equal the oracle's serial step."""
    import torch
    from gpu_harness import up, up_bf16, i32
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    cfg = workloads.get_config("dsv4")
    sel = workloads.make_select_inputs(cfg)
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    N, K = cfg.N, cfg.K
    d_logits = up(logits.view(np.int16)).view(torch.bfloat16)
    draft = torch.zeros(N, K, dtype=torch.int32, device="cuda")
    cws = D.new_workspace(D.dspark_chain_workspace_size(N, K))
    conf, mask, cost = up(sel["conf"]), up(sel["mask"]), up(sel["cost"])
    T = up(np.array([sel["T"]], np.int32))
    surv = torch.zeros(N, K, dtype=torch.float32, device="cuda")
    srt, pre = i32(N * K), torch.zeros(N * K + 1, dtype=torch.float64, device="cuda")
    ne, ns, B = i32(1), i32(1), i32(1)
    obj = torch.zeros(1, dtype=torch.float64, device="cuda")
    ln, cu, vi, vt = i32(N), i32(N + 1), i32(N * K), i32(N * K)
    sws = D.new_workspace(D.dspark_select_workspace_size(N, K, cost.numel()))
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    fork = torch.cuda.Event()
    fork.record(main)
    side.wait_event(fork)
    D.dspark_chain_draft(d_logits, up_bf16(fac["U"]), up_bf16(fac["V"]),
                         up(last), draft, None, cws)
    with torch.cuda.stream(side):
        D.dspark_select_step(conf, mask, cost, T, 0.0, 0, None, surv, srt, pre,
                             ne, ns, B, obj, ln, cu, vi, None, sws)
    join = torch.cuda.Event()
    join.record(side)
    main.wait_event(join)
    D.dspark_gather_verify_tokens(vi, B, draft, vt)
    torch.cuda.synchronize()
    ch = oracle.chain(logits, "bf16", fac["U"], fac["V"], last)
    dg = draft.cpu().numpy()
    r = oracle.select_step(sel["conf"], sel["mask"], sel["cost"], sel["T"],
                           draft=ch["draft"])
    Bg = int(B.item())
    assert Bg == r["B"]
    got_idx = vi.cpu().numpy()[:Bg]
    np.testing.assert_array_equal(got_idx, r["verify_idx"])
    # tokens: equal to the oracle's wherever the drafts agree (everywhere
    # outside fp32 near-ties), and always the device's own draft tokens
    same = dg.reshape(-1)[got_idx] == ch["draft"].reshape(-1)[got_idx]
    assert same.mean() > 0.999
    got_tok = vt.cpu().numpy()[:Bg]
    np.testing.assert_array_equal(got_tok[same], r["verify_tok"][same])
    np.testing.assert_array_equal(got_tok, dg.reshape(-1)[got_idx])
