"""Closed forms and special cases that pin the oracle.

Each case reduces the method to something known independently: a plain
argmax of the logits when the Markov factors vanish ("DSpark on MAX", *What
DSpark is*, item 3), powers for constant confidences and the count of positive
survivals for a flat cost table ("Adaptive Verification in vLLM",
*Scheduling the budget*), the marginal admission rule for a linear cost,
a running maximum for the forced table (same page, *The cost model*), and the
NaN rule of the argmax kernel fix ("DSpark on MAX", *Scaling to 31B*).
"""
import math

import numpy as np
import pytest

import oracle
import workloads


def _tiny_chain_inputs(seed=7, N=4, K=5, vocab=512, rank=16):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 2, size=(N, K, vocab)).astype(np.float32)
    U = workloads.f32_to_bf16_bits(rng.normal(0, 0.1, (vocab, rank)).astype(np.float32))
    V = workloads.f32_to_bf16_bits(rng.normal(0, 0.1, (vocab, rank)).astype(np.float32))
    last = rng.integers(0, vocab, N).astype(np.int32)
    return logits, U, V, last


@pytest.mark.parametrize("zero", ["U", "V"])
def test_zero_factor_reduces_to_plain_argmax(zero):
    logits, U, V, last = _tiny_chain_inputs()
    if zero == "U":
        U = np.zeros_like(U)
    else:
        V = np.zeros_like(V)
    r = oracle.chain(logits, "f32", U, V, last)
    np.testing.assert_array_equal(r["draft"], np.argmax(logits, axis=2))


def test_bias_uses_previous_token_row_of_U_and_all_rows_of_V():
    """A one-hot construction: U[p] selects column j of V, so the bias of
    token v is V[v, j]; a transposed operand or the wrong previous token
    picks a different winner."""
    vocab, rank, K = 64, 16, 3
    U = np.zeros((vocab, rank), np.float32)
    V = np.zeros((vocab, rank), np.float32)
    for p in range(vocab):
        U[p, p % rank] = 1.0
    # token t gets a large bias exactly when prev % rank == (t + 1) % rank
    for t in range(vocab):
        V[t, (t + 1) % rank] = 8.0
    logits = np.zeros((1, K, vocab), np.float32)
    logits[0, :, :] = np.linspace(0, 1, vocab, dtype=np.float32)[None, :] * 0.01
    Ub, Vb = workloads.f32_to_bf16_bits(U), workloads.f32_to_bf16_bits(V)
    last = np.array([5], np.int32)
    r = oracle.chain(logits, "f32", Ub, Vb, last)
    # prev=5 -> columns v with (v+1)%16 == 5 -> v%16 == 4; the largest logit
    # among them is v = 52.  Then prev=52 -> v%16 == 3 -> 51; then 50.
    assert r["draft"].tolist() == [[52, 51, 50]]


def test_constant_confidence_gives_powers():
    N, K = 5, 9
    conf = np.full((N, K), 0.5, np.float32)
    s, st = oracle.survival(conf, np.ones(N, np.uint8))
    assert st == 0
    expect = np.array([math.ldexp(1.0, -(k + 1)) for k in range(K)])
    np.testing.assert_array_equal(s, np.broadcast_to(expect, (N, K)))


def test_flat_cost_admits_every_positive_survival():
    rng = np.random.default_rng(3)
    conf = rng.uniform(0, 1, size=(6, 7)).astype(np.float32)
    conf[2, 3] = 0.0            # request 2 has zero survival from position 3
    mask = np.array([1, 1, 1, 0, 1, 1], np.uint8)
    cost = np.full(128, 50.0, np.float32)
    r = oracle.select_step(conf, mask, cost, 6)
    s = r["survival"]
    assert r["B"] == int(np.sum((s > 0) & (mask[:, None] == 1)))


def test_linear_cost_marginal_rule():
    """For cost a + b*n, admitting the next slot raises the objective iff its
    survival exceeds b times the current objective; the objective is then
    unimodal and B is where the rule first fails."""
    rng = np.random.default_rng(11)
    for trial in range(20):
        N, K = rng.integers(1, 9), rng.integers(1, 9)
        conf = rng.uniform(0.2, 1.0, size=(N, K)).astype(np.float32)
        a, b = float(rng.uniform(5, 50)), float(rng.uniform(0.05, 2.0))
        L = N * K + 40
        cost = (a + b * np.arange(L)).astype(np.float32)
        T = int(rng.integers(0, 30))
        r = oracle.select_step(conf, np.ones(N, np.uint8), cost, T)
        srt = np.sort(r["survival"].reshape(-1))[::-1]
        num, B = float(N), 0
        while B < len(srt):
            den_now = float(cost[T + B])
            step = float(cost[T + B + 1]) - den_now
            if srt[B] * den_now > step * num:
                num += srt[B]
                B += 1
            else:
                break
        assert r["B"] == B, (trial, r["B"], B)


def test_no_sampling_request_gives_empty_budget():
    conf = np.full((4, 7), 0.9, np.float32)
    r = oracle.select_step(conf, np.zeros(4, np.uint8), np.arange(1, 65, dtype=np.float32), 100 % 64)
    assert r["B"] == 0 and r["n_sampling"] == 0 and r["n_eligible"] == 0
    assert r["draft_len"].tolist() == [0, 0, 0, 0]
    assert r["cu_len"].tolist() == [0, 0, 0, 0, 0]
    assert r["verify_idx"].size == 0


def test_single_request_length_is_budget():
    conf = np.array([[0.9, 0.8, 0.7, 0.5, 0.3, 0.2, 0.1]], np.float32)
    cost = (10 + 2.0 * np.arange(32)).astype(np.float32)
    r = oracle.select_step(conf, np.ones(1, np.uint8), cost, 1)
    assert r["draft_len"].tolist() == [r["B"]]
    assert r["verify_idx"].tolist() == list(range(r["B"]))


def test_k_equals_one():
    conf = np.array([[0.3], [0.9], [0.6]], np.float32)
    s, _ = oracle.survival(conf, np.ones(3, np.uint8))
    np.testing.assert_array_equal(s, conf.astype(np.float64))
    order = oracle.order_slots(s, np.ones(3, np.uint8))
    assert order.tolist() == [1, 2, 0]


def test_slot_ties_keep_request_prefixes():
    """Confidence 1.0 makes equal survivals inside a request; slot-id order
    keeps the selection prefix-closed."""
    conf = np.array([[0.5, 1.0, 1.0, 0.5], [0.5, 1.0, 0.5, 0.5]], np.float32)
    s, _ = oracle.survival(conf, np.ones(2, np.uint8))
    order = oracle.order_slots(s, np.ones(2, np.uint8))
    assert order[:5].tolist() == [0, 1, 2, 4, 5]


def test_force_monotone_running_max_and_suffix_min():
    cfg = workloads.get_config("stress")
    cost = workloads.make_select_inputs(cfg)["cost"]
    f = oracle.force_monotone(cost, oracle.FORCE_RUNNING_MAX)
    run, out = -np.inf, []
    for c in cost.tolist():
        run = max(run, c)
        out.append(run)
    np.testing.assert_array_equal(f, np.array(out, np.float32))
    assert np.all(np.diff(f) >= 0) and np.all(f >= cost)
    np.testing.assert_array_equal(oracle.force_monotone(f), f)   # idempotent
    g = oracle.force_monotone(cost, oracle.FORCE_SUFFIX_MIN)
    run, out = np.inf, []
    for c in cost.tolist()[::-1]:
        run = min(run, c)
        out.append(run)
    np.testing.assert_array_equal(g, np.array(out[::-1], np.float32))
    assert np.all(np.diff(g) >= 0) and np.all(g <= cost)


def test_nan_logit_first_nan_wins_and_sets_status():
    logits, U, V, last = _tiny_chain_inputs(N=2, K=3, vocab=64)
    logits[0, 1, 40] = np.nan
    logits[0, 1, 17] = np.nan
    r = oracle.chain(logits, "f32", U, V, last)
    assert r["draft"][0, 1] == 17
    assert r["status"] & oracle.NAN_LOGIT
    assert 0 <= r["draft"].min() and r["draft"].max() < 64


def test_all_minus_inf_row_gives_token_zero():
    logits, U, V, last = _tiny_chain_inputs(N=2, K=2, vocab=64)
    logits[1, 0, :] = -np.inf
    r = oracle.chain(logits, "f32", U, V, last)
    assert r["draft"][1, 0] == 0


def test_exact_tie_picks_lowest_index():
    logits, U, V, last = _tiny_chain_inputs(N=1, K=1, vocab=64)
    V = np.zeros_like(V)
    logits[0, 0, 9] = logits[0, 0, 33] = 100.0
    r = oracle.chain(logits, "f32", U, V, last)
    assert r["draft"][0, 0] == 9


def test_out_of_range_last_token_is_clamped_and_flagged():
    logits, U, V, last = _tiny_chain_inputs(N=2, K=1, vocab=64)
    last = np.array([-3, 70], np.int32)
    r = oracle.chain(logits, "f32", U, V, last)
    ref = oracle.chain(logits, "f32", U, V, np.array([0, 0], np.int32))
    np.testing.assert_array_equal(r["draft"], ref["draft"])
    assert r["status"] & oracle.TOKEN_OOR


def test_confidence_out_of_range_is_clamped_and_flagged():
    conf = np.array([[1.5, np.nan, 0.5], [-0.2, 0.5, 0.5]], np.float32)
    s, st = oracle.survival(conf, np.ones(2, np.uint8))
    assert st & oracle.CONF_OOR
    np.testing.assert_array_equal(s, [[1.0, 0.0, 0.0], [0.0, 0.0, 0.0]])


def test_greedy_stop_differs_from_global_argmax_on_a_staircase():
    """A stepped table makes the objective non-unimodal: admitting slots one at
    a time stops at the first drop ("How DSpark Speeds Up LLM Inference",
    *Verify smarter*), the global argmax looks past it."""
    conf = np.full((1, 8), 0.97, np.float32)
    cost = np.array([10, 10, 10, 30, 30, 30, 30, 30, 30, 30, 30, 30], np.float32)
    g = oracle.select_step(conf, np.ones(1, np.uint8), cost, 1,
                           flags=oracle.BUDGET_GREEDY_STOP)
    a = oracle.select_step(conf, np.ones(1, np.uint8), cost, 1)
    assert g["B"] == 1      # f(2) on the 30 us step is below f(1)
    assert a["B"] == 8      # the whole step pays for itself further on
    assert a["objective"] > g["objective"]


def test_greedy_verify_hand_instance():
    """Two sampling requests and one in prefill; target rows built so the
    matches are known: request 0 accepts 2 of 3 and gets the target's third
    token as bonus, request 2 accepts its single draft and gets the bonus
    from its second row ("DSpark on MAX", *The kernel pass*, item 2)."""
    vocab = 16
    draft = np.array([[3, 5, 7], [1, 1, 1], [9, 0, 0]])
    draft_len = np.array([3, 0, 1])
    mask = np.array([1, 0, 1], np.uint8)
    rows = oracle.verify_rows(draft_len, mask)
    assert rows.tolist() == [0, 4, 4, 6]
    tl = np.zeros((6, vocab), np.float32)
    best = [3, 5, 8, 2, 9, 4]        # row r's argmax
    for r, b in enumerate(best):
        tl[r, b] = 1.0
    tl[5, 4] = tl[5, 11] = 1.0       # tie: the lower index wins
    r = oracle.greedy_verify(tl, "f32", draft, draft_len, mask)
    assert r["target_argmax"].tolist() == best
    assert r["accepted"].tolist() == [2, -1, 1]
    assert r["bonus"].tolist() == [8, -1, 4]


def test_greedy_verify_accepts_everything_when_target_agrees():
    rng = np.random.default_rng(4)
    N, K, vocab = 5, 4, 64
    draft = rng.integers(0, vocab, (N, K))
    ln = rng.integers(0, K + 1, N)
    mask = np.ones(N, np.uint8)
    rows = oracle.verify_rows(ln, mask)
    tl = rng.normal(size=(rows[-1], vocab)).astype(np.float32)
    for n in range(N):
        for j in range(ln[n]):
            tl[rows[n] + j, draft[n, j]] = 100.0
    r = oracle.greedy_verify(tl, "f32", draft, ln, mask)
    assert r["accepted"].tolist() == ln.tolist()
    for n in range(N):
        assert r["bonus"][n] == np.argmax(tl[rows[n] + ln[n]])
