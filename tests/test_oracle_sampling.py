"""Pins of the oracle's probabilistic drafting: a two-level Gumbel-max draw
over blocks of 16 vocabulary entries with Philox4x32-10 words.

"Adaptive Verification in vLLM", *Appendix: reproducing*: the drafter runs
with draft_sample_method "probabilistic", i.e. each draft token is drawn
from the adjusted distribution instead of taken as its argmax.  The random
words come from Philox4x32-10 (Salmon et al., SC 2011), pinned here by its
published known-answer vectors.  The sampling rule is pinned by its
distribution (chi-square against the softmax over several blocks, a
ragged last block included), with planted mistakes in each of its steps
failing that pin; by closed forms (one block of equal entries, blocks with
one finite entry, NaN and infinite rows); by its zero-temperature limit (the
greedy oracle) and by a chain whose bias forces the next token.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import dspark_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
G = O.SAMPLE_BLOCK


def test_philox_known_answers():
    with open(os.path.join(GOLD, "philox4x32_10_kat.json")) as f:
        g = json.load(f)
    for v in g["vectors"]:
        c = [int(x, 16) for x in v["ctr"]]
        k = [int(x, 16) for x in v["key"]]
        out = oracle.philox4x32_10(*c, *k)
        assert [int(o) for o in out] == [int(x, 16) for x in v["out"]]


def test_uniforms_exact_and_in_range():
    xg, xc = oracle.block_words(seed=0x1234_5678_9ABC, offset=3, n=5, k=2, n_blocks=4096)
    for x in (xg, xc):
        u = oracle.word_uniform(x)
        assert np.all((u > 0) & (u < 1))
        assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
        m = u * 2.0 ** 24
        assert np.array_equal(m, np.round(m)) and np.all(np.round(m) % 2 == 1)
    # blocks 2 and 3 take the words of counter 1: 0, 1 and 2, 3
    seed = 0x1234_5678_9ABC
    w = oracle.philox4x32_10(1, 5, 2, 3, seed & 0xFFFFFFFF, seed >> 32)
    assert (int(xg[2]), int(xc[2]), int(xg[3]), int(xc[3])) == tuple(int(x) for x in w)


def test_streams_differ_by_every_counter_field():
    base = oracle.block_words(7, 0, 0, 0, 64)[0]
    for kw in (dict(seed=8, offset=0, n=0, k=0), dict(seed=7, offset=1, n=0, k=0),
               dict(seed=7, offset=0, n=1, k=0), dict(seed=7, offset=0, n=0, k=1),
               dict(seed=7 + (1 << 32), offset=0, n=0, k=0)):
        other = oracle.block_words(n_blocks=64, **kw)[0]
        assert np.mean(other == base) < 0.05


def test_gumbel_moments():
    """Standard Gumbel from the block words: mean = Euler-Mascheroni
    constant, variance = pi^2/6."""
    x = np.concatenate([oracle.block_words(11, off, 0, 0, 1 << 15)[0] for off in range(8)])
    g = -np.log(-np.log(oracle.word_uniform(x)))
    n = g.size
    assert abs(g.mean() - 0.5772156649015329) < 5 * math.sqrt(math.pi ** 2 / 6 / n)
    # the variance of the sample variance of a Gumbel: (mu4 - sigma^4) / n,
    # mu4 = 27/5 sigma^4 (excess kurtosis 12/5)
    s2 = math.pi ** 2 / 6
    assert abs(g.var() - s2) < 5 * math.sqrt((27 / 5 - 1) * s2 ** 2 / n)


# three blocks (16, 16 and a ragged 5) of very different masses and shapes
ADJ = np.concatenate([np.linspace(-1.0, 2.0, 16), np.full(16, 0.5),
                      np.array([3.0, -2.0, 1.0, 0.0, 2.5])])
S_DRAWS = 30000


def _chi2(tau):
    s = oracle.sample_position(np.tile(ADJ, (S_DRAWS, 1)), tau, seed=99, offset=4,
                               ns=np.arange(S_DRAWS), k=1)
    counts = np.bincount(s["tok"], minlength=ADJ.size)
    p = np.exp(ADJ / tau - np.max(ADJ / tau))
    p /= p.sum()
    return float(np.sum((counts - S_DRAWS * p) ** 2 / (S_DRAWS * p)))


# df = 36; P(chi2 > 80) is about 3e-5
CHI2_LIMIT = 80.0


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_sampling_matches_softmax(tau):
    """Tokens drawn by the two-level rule follow softmax(adj / tau)."""
    chi2 = _chi2(tau)
    assert chi2 < CHI2_LIMIT, chi2


def test_planted_mistakes_fail_the_distribution(monkeypatch):
    """Each step of the rule, done wrong, moves the draws off the softmax."""
    # block weight: its largest entry instead of its log partition function
    with monkeypatch.context() as m:
        m.setattr(O, "_block_log_partition", lambda b: np.max(b, axis=-1))
        assert _chi2(1.0) > CHI2_LIMIT
    # entry inside the block: uniform instead of by weight
    with monkeypatch.context() as m:
        m.setattr(O, "_within_block",
                  lambda b, u: int(min(int(u * np.sum(np.isfinite(b))), G - 1)))
        assert _chi2(1.0) > CHI2_LIMIT
    # the entry drawn with the block's Gumbel word instead of its own word
    real = O.block_words
    with monkeypatch.context() as m:
        m.setattr(O, "block_words", lambda *a: (real(*a)[0], real(*a)[0]))
        assert _chi2(1.0) > CHI2_LIMIT


def test_one_block_of_equal_entries_is_the_floor():
    """Equal weights: the inverse CDF picks floor(16 u) (16 u is never an
    integer for u an odd multiple of 2^-24)."""
    xg, xc = oracle.block_words(3, 8, 2, 5, 1)
    u = float(oracle.word_uniform(xc)[0])
    r = oracle.sample_position(np.full((1, G), 0.25), 1.0, 3, 8, [2], 5)
    assert r["tok"][0] == math.floor(G * u)
    # and the score is log(16 * e^0.25) + g
    g = -math.log(-math.log(float(oracle.word_uniform(xg)[0])))
    assert abs(r["score"][0] - (0.25 + math.log(16.0) + g)) < 1e-12


def test_blocks_with_one_finite_entry_reduce_to_gumbel_max():
    """With one finite entry per block the block key is that entry plus its
    block's Gumbel, and the draw is that entry: plain Gumbel-max over them."""
    nb = 6
    adj = np.full((1, nb * G), -np.inf)
    vals = np.array([0.5, 1.25, -3.0, 2.0, 0.0, 1.0])
    pos = np.array([3, 0, 15, 7, 9, 1])
    adj[0, np.arange(nb) * G + pos] = vals
    xg, _ = oracle.block_words(21, 2, 4, 3, nb)
    key = vals - np.log(-np.log(oracle.word_uniform(xg)))
    r = oracle.sample_position(adj, 1.0, 21, 2, [4], 3)
    j = int(np.argmax(key))
    assert r["tok"][0] == j * G + pos[j]
    assert r["score"][0] == key[j]
    top2 = np.sort(key)[-2:]
    assert r["margin"][0] == top2[1] - top2[0]


def test_nan_and_infinite_rows():
    adj = np.random.default_rng(1).standard_normal((4, 50))
    adj[0, 20] = np.nan
    adj[0, 3] = np.nan           # the first NaN wins, whatever the noise
    adj[1, :] = -np.inf          # nothing finite: the first entry
    adj[2, 40:] = -np.inf        # a ragged, partly -inf last block
    adj[3, 37] = np.inf
    adj[3, 21] = np.inf          # the first +inf holds all the weight
    r = oracle.sample_position(adj, 1.0, 5, 0, [0, 1, 2, 3], 0)
    assert r["tok"][0] == 3 and np.isnan(r["score"][0])
    assert r["tok"][1] == 0 and r["score"][1] == -np.inf
    assert r["tok"][2] < 40
    assert r["tok"][3] == 21 and r["score"][3] == np.inf


def _factors(vocab, rank):
    """U[t] . V[v] = 40 if v == (t + 1) % vocab else 0 (rank >= vocab)."""
    U = np.zeros((vocab, rank), np.float32)
    Vf = np.zeros((vocab, rank), np.float32)
    for t in range(vocab):
        U[t, t] = 40.0
        Vf[(t + 1) % vocab, t] = 1.0
    import workloads
    return workloads.f32_to_bf16_bits(U), workloads.f32_to_bf16_bits(Vf)


def test_chain_wiring_under_sampling():
    """The bias keyed on the sampled previous token forces prev + 1 (softmax
    mass of any other token < vocab * e^-40), so the sampled chain is
    last + 1, last + 2, ... whatever the noise."""
    vocab, rank, K, n = 32, 32, 5, 4
    U, V = _factors(vocab, rank)
    logits = np.zeros((n, K, vocab), np.float32)
    last = np.array([0, 7, 30, 31])
    r = oracle.chain(logits, "f32", U, V, last, sample=dict(seed=5, offset=9, tau=1.0))
    want = (last[:, None] + 1 + np.arange(K)[None, :]) % vocab
    np.testing.assert_array_equal(r["draft"], want)


def test_zero_temperature_limit_is_greedy():
    rng = np.random.default_rng(4)
    vocab, rank, K, n = 256, 16, 4, 6
    import workloads
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank)).astype(np.float32))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank)).astype(np.float32))
    logits = (2 * rng.standard_normal((n, K, vocab))).astype(np.float32)
    last = rng.integers(0, vocab, n)
    g = oracle.chain(logits, "f32", U, V, last)
    s = oracle.chain(logits, "f32", U, V, last, sample=dict(seed=1, offset=0, tau=1e-9))
    np.testing.assert_array_equal(s["draft"], g["draft"])
    # at temperature 1 the draws differ from the argmax somewhere
    s1 = oracle.chain(logits, "f32", U, V, last, sample=dict(seed=1, offset=0, tau=1.0))
    assert np.any(s1["draft"] != g["draft"])


def test_rows_pick_the_request_counter():
    """A subset of rows reproduces the same draws as the full batch."""
    rng = np.random.default_rng(6)
    vocab, rank, K, n = 128, 16, 3, 5
    import workloads
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank)).astype(np.float32))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank)).astype(np.float32))
    logits = rng.standard_normal((n, K, vocab)).astype(np.float32)
    last = rng.integers(0, vocab, n)
    sm = dict(seed=3, offset=2, tau=1.0)
    full = oracle.chain(logits, "f32", U, V, last, sample=sm)
    sub = oracle.chain(logits[[1, 3]], "f32", U, V, last[[1, 3]], sample=sm,
                       rows=np.array([1, 3]))
    np.testing.assert_array_equal(sub["draft"], full["draft"][[1, 3]])
