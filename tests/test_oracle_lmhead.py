"""Pins of the oracle's fused LM head (adj = h . W^T + U[prev] . V^T).

"DSpark on MAX", *What DSpark is*, items 2-3: the block drafter scores all K
positions in one forward pass and the chain adds a low-rank bias keyed on the
previous token before the argmax.  Pinned by exact integer arithmetic (small
integers are exact in bf16, and every sum stays far below 2^53), by the
special cases W = 0 and h = 0 (the plain chain on zero logits) and by a
one-hot construction whose drafts are known in advance.
"""
import numpy as np

import oracle
import workloads


def _bits(a):
    return workloads.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_exact_integers_against_python_ints():
    rng = np.random.default_rng(0)
    n, K, d, vocab, r = 3, 4, 24, 40, 16
    h = rng.integers(-3, 4, (n, K, d))
    W = rng.integers(-3, 4, (vocab, d))
    U = rng.integers(-2, 3, (vocab, r))
    V = rng.integers(-2, 3, (vocab, r))
    last = rng.integers(0, vocab, n)
    res = oracle.chain_lmhead(_bits(h), _bits(W), _bits(U), _bits(V), last)
    for i in range(n):
        prev = int(last[i])
        for k in range(K):
            adj = [sum(int(h[i, k, j]) * int(W[v, j]) for j in range(d)) +
                   sum(int(U[prev, j]) * int(V[v, j]) for j in range(r))
                   for v in range(vocab)]
            best = max(adj)
            tok = adj.index(best)              # first maximal index
            assert res["draft"][i, k] == tok, (i, k)
            assert res["score"][i, k] == best
            prev = tok


def test_zero_projection_or_hidden_is_the_bias_chain():
    rng = np.random.default_rng(1)
    n, K, d, vocab, r = 4, 3, 32, 64, 16
    h = _bits(rng.standard_normal((n, K, d)))
    W = _bits(rng.standard_normal((vocab, d)))
    U = _bits(rng.standard_normal((vocab, r)))
    V = _bits(rng.standard_normal((vocab, r)))
    last = rng.integers(0, vocab, n)
    zero_logits = np.zeros((n, K, vocab))
    ref = oracle.chain(zero_logits, "f64", U, V, last)
    for hh, WW in ((h, np.zeros_like(W)), (np.zeros_like(h), W)):
        res = oracle.chain_lmhead(hh, WW, U, V, last)
        np.testing.assert_array_equal(res["draft"], ref["draft"])


def test_one_hot_construction():
    """h[n, k] = e_{c(n,k)} and W[v, j] = 10 * [v == j] make the logits
    10 * [v == c(n,k)]; with a bias that adds 20 to v = prev + 1, the token
    is prev + 1 unless c(n,k) = prev + 1 too (30 then, same answer) — and a
    zero bias would give c(n,k).  Both cases are checked."""
    n, K, vocab = 3, 5, 32
    d = vocab
    rng = np.random.default_rng(2)
    c = rng.integers(0, vocab, (n, K))
    h = np.zeros((n, K, d))
    for i in range(n):
        for k in range(K):
            h[i, k, c[i, k]] = 1.0
    W = 10.0 * np.eye(vocab)
    last = np.array([0, 9, 31])
    # zero bias: the drafts are the one-hot positions
    Z = np.zeros((vocab, 16))
    res = oracle.chain_lmhead(_bits(h), _bits(W), _bits(Z), _bits(Z), last)
    np.testing.assert_array_equal(res["draft"], c)
    # bias 20 on prev + 1 dominates the logits' 10
    U = np.zeros((vocab, vocab))
    Vb = np.zeros((vocab, vocab))
    for t in range(vocab):
        U[t, t] = 20.0
        Vb[(t + 1) % vocab, t] = 1.0
    res = oracle.chain_lmhead(_bits(h), _bits(W), _bits(U), _bits(Vb), last)
    np.testing.assert_array_equal(res["draft"], (last[:, None] + 1 + np.arange(K)) % vocab)
