"""Pins of the chain oracle's top-2 margin and |max| per row.

The parity tests accept a device token that differs from the oracle's only
where the oracle's own top-2 margin (largest adjusted value minus the second
largest, over the whole vocabulary) is below 1e-3 * |largest|.  These
values therefore decide which device tokens are tolerated, and are pinned
here on rows whose top two values are known by construction: a distinct
second best with a close third, an exact tie (margin 0), a NaN row (margin
NaN: never tolerated), negative rows, the maximum at either end, an all
-inf row, +inf, a one-entry vocabulary and a bias that reorders the top
two.  The probabilistic path's margin (over block keys) is pinned with the
sampler in test_oracle_sampling.py.
"""
import numpy as np
import pytest

import oracle
import workloads

NAN, INF = np.nan, np.inf


def _zero_bias(vocab, rank=16):
    z = np.zeros((vocab, rank), np.float64)
    return z, z.copy()


# (row, token, score, margin, |max|); the margin is exact for dyadic values
ROWS = [
    ([0.5, 4.0, -1.0, 3.25, 2.0, 3.0], 1, 4.0, 0.75, 4.0),    # third is 3.0
    ([2.0, 7.0, 1.0, 7.0, 6.5, 0.0], 1, 7.0, 0.0, 7.0),       # exact tie
    ([1.0, NAN, 3.0, 2.0, NAN, 0.0], 1, NAN, NAN, NAN),       # first NaN
    ([-3.0, -1.0, -2.0, -1.5, -8.0, -4.0], 1, -1.0, 0.5, 1.0),
    ([5.5, 1.0, 2.0, 3.0, 4.0, 6.0], 5, 6.0, 0.5, 6.0),       # max last, 2nd first
    ([6.0, 1.0, 2.0, 3.0, 4.0, 5.75], 0, 6.0, 0.25, 6.0),     # max first, 2nd last
    ([-INF] * 6, 0, -INF, NAN, INF),                          # undefined margin
    ([1.0, INF, 2.0, 0.0, 0.0, 0.0], 1, INF, INF, INF),
    ([1.0, INF, 2.0, INF, 0.0, 0.0], 1, INF, NAN, INF),       # inf - inf
]


def _check(r, i, tok, score, margin, absmax):
    assert r["tok"][i] == tok
    for got, want in ((r["score"][i], score), (r["margin"][i], margin),
                      (r["absmax"][i], absmax)):
        if np.isnan(want):
            assert np.isnan(got)
        else:
            assert got == want


def test_margin_rows_by_construction():
    logits = np.array([row for row, *_ in ROWS], np.float64)
    U, V = _zero_bias(logits.shape[1])
    r = oracle.chain_position(logits, U, V, np.zeros(len(ROWS), np.int64))
    for i, (_, tok, score, margin, absmax) in enumerate(ROWS):
        _check(r, i, tok, score, margin, absmax)


def test_margin_is_top_minus_second_on_random_rows():
    """Brute force: sort each row and take the two largest values."""
    rng = np.random.default_rng(7)
    # rows long enough that a partial selection does not sort them whole
    logits = rng.integers(-3000, 3000, (40, 4096)).astype(np.float64) / 8.0
    logits[:4, 100] = logits[:4].max(axis=1)    # planted exact top ties
    U, V = _zero_bias(4096)
    r = oracle.chain_position(logits, U, V, np.zeros(40, np.int64))
    srt = np.sort(logits, axis=1)
    np.testing.assert_array_equal(r["margin"], srt[:, -1] - srt[:, -2])
    np.testing.assert_array_equal(r["absmax"], np.abs(srt[:, -1]))
    assert np.all(r["margin"][:4] == 0.0) and np.all(r["margin"][4:] >= 0.0)


def test_margin_uses_adjusted_values():
    """A bias that reorders the top two: the margin is taken after the bias.
    Rank-2 factors with U[prev] = (1, 0) and V[v] = (x_v, 0) give bias x_v
    exactly, so adj = logits + x."""
    logits = np.array([[3.0, 2.5, 1.0, 2.75]])
    x = np.array([0.0, 1.0, 0.5, 0.0])
    U = np.zeros((4, 2)); U[2] = (1.0, 0.0)
    V = np.stack([x, np.zeros(4)], axis=1)
    r = oracle.chain_position(logits, U, V, np.array([2]))
    # adj = [3.0, 3.5, 1.5, 2.75]
    assert r["tok"][0] == 1 and r["score"][0] == 3.5
    assert r["margin"][0] == 0.5 and r["absmax"][0] == 3.5
    # prev = 0 (bias zero): logits alone decide
    r0 = oracle.chain_position(logits, U, V, np.array([0]))
    assert r0["tok"][0] == 0 and r0["margin"][0] == 0.25


def test_single_entry_vocabulary():
    r = oracle.chain_position(np.array([[1.5], [-2.0]]), np.zeros((1, 16)),
                              np.zeros((1, 16)), np.zeros(2, np.int64))
    assert r["tok"].tolist() == [0, 0]
    assert np.all(np.isinf(r["margin"])) and np.all(r["margin"] > 0)


def test_chain_reports_each_positions_margin():
    """chain() returns, per position, the margin of the row it chained
    (position 1 sees the bias of the token chosen at position 0)."""
    vocab, rank = 4, 16
    U = np.zeros((vocab, rank), np.float32)
    V = np.zeros((vocab, rank), np.float32)
    U[1, 0] = 1.0           # prev = 1 adds V[:, 0] at the next position
    V[:, 0] = [0.0, 0.0, 1.0, 0.0]
    logits = np.array([[[0.0, 2.0, 1.0, 1.5],      # -> 1 (margin 0.5)
                        [3.0, 0.0, 2.5, 0.0]]],    # adj [3, 0, 3.5, 0] -> 2
                      np.float32)
    r = oracle.chain(logits, "f32", workloads.f32_to_bf16_bits(U),
                     workloads.f32_to_bf16_bits(V), np.array([0]))
    assert r["draft"].tolist() == [[1, 2]]
    assert r["margin"].tolist() == [[0.5, 0.5]]
    assert r["absmax"].tolist() == [[2.0, 3.5]]
