"""GPU parity of the chaining kernel against the oracle.

"DSpark on MAX", *What DSpark is*, item 3: per position, logits + U[prev] .
V^T, then a vocabulary argmax, prev being the token chosen at the previous
position.  Small cases span several 128 x 256 tiles with ragged tails in the
batch, the vocabulary and the rank; full-size workloads are checked on every
row against one oracle pass per workload.  Also covered: the
NaN rule of "DSpark on MAX", *Scaling to 31B* (a NaN must never turn into a
sentinel index), exact ties, all -inf rows, out-of-range previous tokens and
strided logits layouts.
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


def test_tiny_workload():
    from gpu_harness import run_chain, check_chain
    cfg = workloads.get_config("tiny")
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    got, score, st = run_chain(logits, "f32", fac["U"], fac["V"], last)
    assert st == 0
    ref = oracle.chain(logits, "f32", fac["U"], fac["V"], last)
    np.testing.assert_array_equal(got, ref["draft"])
    check_chain(got, score, logits, "f32", fac["U"], fac["V"], last)


@pytest.mark.parametrize("N,K,vocab,rank,dtype", [
    (1, 1, 256, 16, "bf16"),
    (3, 7, 1024, 16, "f32"),
    (5, 3, 3000, 64, "bf16"),       # ragged vocabulary tail
    (130, 2, 2048, 80, "bf16"),     # two request tiles, rank not /64
    (257, 3, 4104, 256, "bf16"),    # three request tiles, ragged both ways
    (64, 9, 5000, 128, "f32"),
    (200, 4, 65536, 256, "bf16"),   # many vocabulary tiles per CTA
])
def test_shapes(N, K, vocab, rank, dtype):
    from gpu_harness import run_chain, check_chain
    logits, U, V, last = _inputs(N, K, vocab, rank, dtype, seed=N + K + vocab)
    got, score, st = run_chain(logits, dtype, U, V, last)
    assert st == 0
    assert got.min() >= 0 and got.max() < vocab
    near = check_chain(got, score, logits, dtype, U, V, last)
    assert near <= max(1, N * K // 100)


@pytest.mark.parametrize("layout,pad", [("knv", 0), ("nkv", 64), ("knv", 8)])
def test_strided_layouts(layout, pad):
    from gpu_harness import run_chain, check_chain
    logits, U, V, last = _inputs(37, 5, 2560, 64, "bf16", seed=3)
    got, score, st = run_chain(logits, "bf16", U, V, last, layout=layout, pad=pad)
    assert st == 0
    check_chain(got, score, logits, "bf16", U, V, last)


def test_nan_inf_ties_and_bad_last_token():
    from gpu_harness import run_chain
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    N, K, vocab, rank = 6, 3, 1536, 32
    logits, U, V, last = _inputs(N, K, vocab, rank, "f32", seed=11)
    logits[0, 1, 700] = np.nan                 # NaN in a later tile...
    logits[0, 1, 90] = np.nan                  # ...and an earlier one: 90 wins
    logits[1, 0, :] = -np.inf                  # all -inf: index 0
    V[1000] = V[200]                           # identical bias for 200/1000
    logits[2, 2, 200] = logits[2, 2, 1000] = 50.0
    last[3] = -7                               # out of range -> 0, flagged
    last[4] = vocab + 3
    got, score, st = run_chain(logits, "f32", U, V, last)
    ref = oracle.chain(logits, "f32", U, V, last)
    np.testing.assert_array_equal(got, ref["draft"])
    assert got[0, 1] == 90 and np.isnan(score[0, 1])
    assert got[1, 0] == 0 and score[1, 0] == -np.inf
    assert got[2, 2] == 200
    assert st == (D.DEV_NAN_LOGIT | D.DEV_TOKEN_OOR)
    assert got.min() >= 0 and got.max() < vocab


def test_zero_factor_equals_plain_argmax():
    from gpu_harness import run_chain
    logits, U, V, last = _inputs(140, 4, 3072, 64, "bf16", seed=12)
    got, _, _ = run_chain(logits, "bf16", np.zeros_like(U), V, last)
    vals = workloads.bf16_bits_to_f32(logits)
    np.testing.assert_array_equal(got, np.argmax(vals, axis=2))


def _full(name, rows):
    from gpu_harness import run_chain, check_chain
    cfg = workloads.get_config(name)
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    got, score, st = run_chain(logits, cfg.logits_dtype, fac["U"], fac["V"], last)
    assert st == 0
    assert got.min() >= 0 and got.max() < cfg.vocab
    near = check_chain(got, score, logits, cfg.logits_dtype, fac["U"], fac["V"],
                       last, rows=rows)
    return cfg, logits, got, near


@pytest.mark.parametrize("name", ["gemma4_12b", "conc64", "dsv4", "headline"])
def test_full_size_workloads(name):
    """Every row of the workload against the oracle, under teacher forcing."""
    from gpu_harness import report_near
    cfg = workloads.get_config(name)
    _, _, _, near = _full(name, np.arange(cfg.N))
    report_near(f"chain {name}", near, cfg.N * cfg.K)
    assert near <= max(1, cfg.N * cfg.K // 100)


def test_stress_all_rows_and_planted_ties():
    from gpu_harness import report_near
    cfg = workloads.get_config("stress")
    cfg, logits, got, near = _full("stress", np.arange(cfg.N))
    report_near("chain stress", near, cfg.N * cfg.K)
    assert near <= max(1, cfg.N * cfg.K // 100)
    ties = workloads.planted_ties(cfg, logits[:64], rows=np.arange(64))
    assert len(ties) > 0
    # a planted tie survives the bias exactly; the lower index must win
    # whenever the tie is the row's maximum given the device's prefix
    fac = workloads.make_chain_factors(cfg)
    U64, V64 = oracle.bf16_to_f64(fac["U"]), oracle.bf16_to_f64(fac["V"])
    last = workloads.make_last_token(cfg)
    for n, k, c0, c1 in ties:
        prev = last[n] if k == 0 else got[n, k - 1]
        r = oracle.chain_position(oracle.to_f64(logits[n:n + 1, k], "bf16"),
                                  U64, V64, np.array([prev]))
        if r["tok"][0] in (c0, c1):
            assert r["tok"][0] == c0
            assert got[n, k] == c0


def test_random_shapes():
    """Random shapes with ragged batch, vocabulary and rank tails (vocabulary
    a multiple of 8, rank a multiple of 16, as the boundary requires), both
    logits dtypes and layouts, argmax and probabilistic drafting: tokens
    follow the near-tie rule against the oracle."""
    from gpu_harness import run_chain, check_chain
    rng = np.random.default_rng(4242)
    for case in range(12):
        N = int(rng.integers(1, 400))
        K = int(rng.integers(1, 9))
        vocab = 8 * int(rng.integers(1, 1200))
        rank = 16 * int(rng.integers(1, 17))
        dtype = "bf16" if rng.uniform() < 0.7 else "f32"
        layout = "nkv" if rng.uniform() < 0.7 else "knv"
        x = rng.standard_normal((N, K, vocab), dtype=np.float32) * np.float32(rng.uniform(0.5, 4))
        logits = workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x
        sd = np.float32(rng.uniform(0.01, 0.2))
        U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * sd)
        V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * sd)
        last = rng.integers(0, vocab, N).astype(np.int32)
        sample = None
        if rng.uniform() < 0.3:
            sample = dict(seed=int(rng.integers(0, 2**63)), offset=int(rng.integers(0, 2**31)),
                          tau=float(rng.uniform(0.5, 2.0)))
        got, score, st = run_chain(logits, dtype, U, V, last, layout=layout, sample=sample)
        assert st == 0, case
        assert got.min() >= 0 and got.max() < vocab, case
        assert check_chain(got, score, logits, dtype, U, V, last, sample=sample) \
            <= max(1, N * K // 50), case
