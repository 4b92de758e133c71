"""Pins of the oracle's probabilistic drafting (Gumbel-max over the adjusted
logits with Philox4x32-10 noise).

"Adaptive Verification in vLLM", *Appendix: reproducing*: the drafter runs
with draft_sample_method "probabilistic", i.e. each draft token is drawn
from the adjusted distribution instead of taken as its argmax.  The random
numbers come from Philox4x32-10 (Salmon et al., SC 2011), pinned here by its
published known-answer vectors; the sampling rule is pinned by its
distribution (chi-square against the softmax), its zero-temperature limit
(the greedy oracle) and a chain whose bias forces the next token.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    with open(os.path.join(GOLD, "philox4x32_10_kat.json")) as f:
        g = json.load(f)
    for v in g["vectors"]:
        c = [int(x, 16) for x in v["ctr"]]
        k = [int(x, 16) for x in v["key"]]
        out = oracle.philox4x32_10(*c, *k)
        assert [int(o) for o in out] == [int(x, 16) for x in v["out"]]


def test_uniforms_exact_and_in_range():
    u = oracle.draft_uniforms(seed=0x1234_5678_9ABC, offset=3, n=5, k=2, vocab=4096)
    assert np.all((u > 0) & (u < 1))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    m = u * 2.0 ** 24
    assert np.array_equal(m, np.round(m)) and np.all(np.round(m) % 2 == 1)
    # word v % 4 of counter v // 4: recompute four entries by hand
    seed = 0x1234_5678_9ABC
    w = oracle.philox4x32_10(1, 5, 2, 3, seed & 0xFFFFFFFF, seed >> 32)
    for j in range(4):
        assert u[4 + j] == (2 * (int(w[j]) >> 9) + 1) * 2.0 ** -24


def test_streams_differ_by_every_counter_field():
    base = oracle.draft_uniforms(7, 0, 0, 0, 64)
    for kw in (dict(seed=8, offset=0, n=0, k=0), dict(seed=7, offset=1, n=0, k=0),
               dict(seed=7, offset=0, n=1, k=0), dict(seed=7, offset=0, n=0, k=1),
               dict(seed=7 + (1 << 32), offset=0, n=0, k=0)):
        other = oracle.draft_uniforms(vocab=64, **kw)
        assert np.mean(other == base) < 0.05


def test_gumbel_moments():
    """Standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2/6."""
    g = np.concatenate([oracle.gumbel_noise(11, off, 0, 0, 1 << 16) for off in range(8)])
    n = g.size
    mean, var = g.mean(), g.var()
    assert abs(mean - 0.5772156649015329) < 5 * math.sqrt(math.pi ** 2 / 6 / n)
    # the variance of the sample variance of a Gumbel: (mu4 - sigma^4) / n,
    # mu4 = 27/5 sigma^4 (excess kurtosis 12/5)
    s2 = math.pi ** 2 / 6
    assert abs(var - s2) < 5 * math.sqrt((27 / 5 - 1) * s2 ** 2 / n)


@pytest.mark.parametrize("tau", [1.0, 0.5, 2.0])
def test_sampling_matches_softmax(tau):
    """Tokens drawn with the chain's rule follow softmax(adj / tau)."""
    adj = np.array([[1.0, 0.0, 2.5, -1.0, 2.0, 0.5]])
    V = adj.shape[1]
    S = 20000
    counts = np.zeros(V)
    U64 = np.zeros((V, 1))
    for off in range(S):
        noise = oracle.gumbel_noise(99, off, 0, 0, V)[None, :]
        r = oracle.chain_position(adj, U64, U64, np.zeros(1, np.int64), noise, tau)
        counts[r["tok"][0]] += 1
    p = np.exp(adj[0] / tau - np.max(adj[0] / tau))
    p /= p.sum()
    chi2 = float(np.sum((counts - S * p) ** 2 / (S * p)))
    assert chi2 < 30.0, (chi2, counts, S * p)      # df = 5: p-value ~ 1.5e-5


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
