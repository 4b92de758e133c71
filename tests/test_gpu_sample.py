"""GPU parity of probabilistic drafting (dspark_chain_sample) against the
oracle.

"Adaptive Verification in vLLM", *Appendix: reproducing*: the drafter runs
with draft_sample_method "probabilistic".  Each draft token is a draw from
softmax(adj / tau), taken in two steps over blocks of 16 vocabulary
entries: the block by Gumbel-max on its log partition function, then the
entry by inverting the block's cumulative weights; Philox4x32-10 keyed on
the seed with counter (block / 2, n, k, offset) gives every block its two
words, and the oracle draws from the same words in fp64.  Tokens must agree
except at a near-tie of the block keys or a boundary tie inside the block,
and scores (the winning block's key) to 1e-5 relative.  Also: the same
(seed, offset) reproduces the same drafts, the offset changes them, a
vanishing temperature gives the greedy chain, a forcing bias makes the
chain deterministic, and the draw frequencies over many rows and offsets
follow the softmax over several blocks.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(N, K, vocab, rank, dtype, seed, uv_sd=0.05, sd=2.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, K, vocab), dtype=np.float32) * np.float32(sd)
    logits = workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(uv_sd))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(uv_sd))
    last = rng.integers(0, vocab, N).astype(np.int32)
    return logits, U, V, last


SM = dict(seed=0x0123_4567_89AB_CDEF, offset=11, tau=1.0)


def test_tiny_workload():
    from gpu_harness import run_chain, check_chain
    cfg = workloads.get_config("tiny")
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    got, score, st = run_chain(logits, "f32", fac["U"], fac["V"], last, sample=SM)
    assert st == 0
    near = check_chain(got, score, logits, "f32", fac["U"], fac["V"], last, sample=SM)
    assert near == 0


@pytest.mark.parametrize("N,K,vocab,rank,dtype,tau", [
    (1, 1, 256, 16, "bf16", 1.0),
    (3, 7, 1024, 16, "f32", 0.7),
    (5, 3, 3000, 64, "bf16", 1.0),      # ragged vocabulary tail
    (130, 2, 2048, 80, "bf16", 1.3),    # two request tiles
    (257, 3, 4104, 256, "bf16", 1.0),   # three request tiles, ragged both ways
    (64, 9, 5000, 128, "f32", 2.0),
    (200, 4, 65536, 256, "bf16", 1.0),  # many vocabulary tiles per CTA
    (32, 5, 4104, 128, "bf16", 1.0),    # 32 requests: each held four times
    (33, 2, 2048, 64, "f32", 1.0),      # 33 requests: each held twice
    (40, 3, 5000, 64, "bf16", 0.8),     # twice, ragged vocabulary tail
])
def test_shapes(N, K, vocab, rank, dtype, tau):
    from gpu_harness import run_chain, check_chain
    logits, U, V, last = _inputs(N, K, vocab, rank, dtype, seed=N + K + vocab)
    sm = dict(SM, tau=tau, offset=N)
    got, score, st = run_chain(logits, dtype, U, V, last, sample=sm)
    assert st == 0
    assert got.min() >= 0 and got.max() < vocab
    near = check_chain(got, score, logits, dtype, U, V, last, sample=sm)
    assert near <= max(2, N * K // 50)


@pytest.mark.parametrize("layout,pad", [("knv", 0), ("nkv", 64)])
def test_strided_layouts(layout, pad):
    from gpu_harness import run_chain, check_chain
    logits, U, V, last = _inputs(37, 5, 2560, 64, "bf16", seed=3)
    got, score, st = run_chain(logits, "bf16", U, V, last, layout=layout, pad=pad,
                               sample=SM)
    assert st == 0
    check_chain(got, score, logits, "bf16", U, V, last, sample=SM)


def test_reproducible_and_offset_dependent():
    from gpu_harness import run_chain
    logits, U, V, last = _inputs(96, 6, 4096, 64, "bf16", seed=21)
    a, sa, _ = run_chain(logits, "bf16", U, V, last, sample=SM)
    b, sb, _ = run_chain(logits, "bf16", U, V, last, sample=SM)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(sa, sb)
    c, _, _ = run_chain(logits, "bf16", U, V, last, sample=dict(SM, offset=12))
    d, _, _ = run_chain(logits, "bf16", U, V, last, sample=dict(SM, seed=SM["seed"] ^ (1 << 40)))
    assert np.mean(a == c) < 0.2 and np.mean(a == d) < 0.2


def test_vanishing_temperature_is_greedy():
    from gpu_harness import run_chain
    logits, U, V, last = _inputs(64, 4, 3072, 64, "f32", seed=5)
    g, _, _ = run_chain(logits, "f32", U, V, last)
    s, _, _ = run_chain(logits, "f32", U, V, last, sample=dict(SM, tau=1e-20))
    np.testing.assert_array_equal(s, g)


def test_forcing_bias_makes_the_chain_deterministic():
    """U[t] . V[v] = 40 iff v = t + 1: every draw is prev + 1 whatever the
    noise (softmax mass elsewhere < vocab e^-40)."""
    from gpu_harness import run_chain
    vocab, rank, K, n = 64, 64, 6, 5
    U = np.zeros((vocab, rank), np.float32)
    Vf = np.zeros((vocab, rank), np.float32)
    for t in range(vocab):
        U[t, t] = 40.0
        Vf[(t + 1) % vocab, t] = 1.0
    Ub, Vb = workloads.f32_to_bf16_bits(U), workloads.f32_to_bf16_bits(Vf)
    logits = np.zeros((n, K, vocab), np.float32)
    last = np.array([0, 5, 62, 63, 30], np.int32)
    got, _, st = run_chain(logits, "f32", Ub, Vb, last, sample=SM)
    assert st == 0
    np.testing.assert_array_equal(got, (last[:, None] + 1 + np.arange(K)) % vocab)


def test_frequencies_follow_softmax():
    """One position, N identical rows whose 24 finite logits sit in three
    16-entry blocks (8 each; the other 40 entries of the 64-entry vocabulary
    are -inf): the rows are independent draws (the request index is a
    counter field); over 4 offsets x 4096 rows the counts follow
    softmax(adj / tau) (chi-square, 23 degrees of freedom), and the first 64
    rows of every offset match the oracle's draws."""
    from gpu_harness import run_chain, check_chain
    vocab, rank, N = 64, 16, 4096
    vals = np.array([1.0, 0.0, 2.5, -1.0, 2.0, 0.5, -0.5, 1.5,
                     0.2, 1.8, -0.8, 0.9, 2.2, -0.3, 0.6, 1.1,
                     -1.5, 0.4, 1.3, 2.8, -0.6, 0.1, 1.6, 0.7], np.float32)
    pos = np.concatenate([np.arange(0, 8), np.arange(16, 24), np.arange(32, 40)])
    full = np.full(vocab, -np.inf, np.float32)
    full[pos] = vals
    logits = np.broadcast_to(full, (N, 1, vocab)).copy()
    U = workloads.f32_to_bf16_bits(np.zeros((vocab, rank), np.float32))
    last = np.zeros(N, np.int32)
    tau = 0.8
    counts = np.zeros(vocab)
    for off in range(4):
        sm = dict(seed=77, offset=off, tau=tau)
        got, score, st = run_chain(logits, "f32", U, U, last, sample=sm)
        assert st == 0
        counts += np.bincount(got[:, 0], minlength=vocab)
        check_chain(got, score, logits, "f32", U, U, last, rows=np.arange(64), sample=sm)
    assert counts[np.isinf(full)].sum() == 0
    p = np.exp(vals / tau - np.max(vals / tau))
    p /= p.sum()
    S = counts.sum()
    chi2 = float(np.sum((counts[pos] - S * p) ** 2 / (S * p)))
    assert chi2 < 60.0, (chi2, counts[pos], S * p)   # df = 23: p-value ~ 4e-5


def test_nan_row_and_bad_last_token():
    from gpu_harness import run_chain, check_chain
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    logits, U, V, last = _inputs(8, 3, 1024, 32, "f32", seed=9)
    logits[1, 0, 500] = np.nan
    logits[1, 0, 100] = np.nan          # first NaN wins over any noise
    logits[5, 1, 700] = np.inf
    logits[5, 1, 333] = np.inf          # the first +inf holds all the weight
    last[3] = 5000                      # out of range -> 0
    got, score, st = run_chain(logits, "f32", U, V, last, sample=SM)
    assert got[1, 0] == 100 and got[5, 1] == 333
    assert st & D.DEV_NAN_LOGIT and st & D.DEV_TOKEN_OOR
    last_ref = last.copy()
    last_ref[3] = 0
    check_chain(got, score, logits, "f32", U, V, last_ref, sample=SM)


@pytest.mark.parametrize("name", ["gemma4_12b", "conc64", "headline"])
def test_full_size_workloads(name):
    from gpu_harness import run_chain, check_chain
    cfg = workloads.get_config(name)
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    got, score, st = run_chain(logits, cfg.logits_dtype, fac["U"], fac["V"], last,
                               sample=SM)
    assert st == 0
    assert got.min() >= 0 and got.max() < cfg.vocab
    from gpu_harness import report_near
    near = check_chain(got, score, logits, cfg.logits_dtype, fac["U"], fac["V"],
                       last, sample=SM)
    report_near(f"sample {name}", near, cfg.N * cfg.K)
    assert near <= max(1, cfg.N * cfg.K // 100)
