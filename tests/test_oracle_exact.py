"""Exact-arithmetic pins of the oracle's floating-point steps.

* Chaining ("DSpark on MAX", *What DSpark is*, item 3): at vocabulary 1024 and
  rank 16 the bias U[prev] . V[v] of bf16 factors is computed here with Python
  integers (every bf16 and fp32 value is an integer multiple of 2^-149, every
  product of two bf16 values one of 2^-266), so the argmax below is exact and
  independent of numpy's fp64 GEMM.
* Cumulative sums ("Adaptive Verification in vLLM", *Scheduling the budget*,
  "an np.argmax over a cumulative sum"): the oracle reads the cumulative sum
  as the exact sum rounded once; it is checked against ``math.fsum`` (a
  correctly rounded summation) and against a constructed case where adding
  left to right in doubles would round the other way.
"""
import math
from fractions import Fraction

import numpy as np

import oracle
import workloads

SCALE = 266  # exponent of the common unit 2^-266


def _exact_int(x: float) -> int:
    fr = Fraction(x)
    v = fr * (1 << SCALE)
    assert v.denominator == 1
    return int(v)


def test_chain_matches_exact_integer_argmax():
    cfg = workloads.get_config("tiny")
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    r = oracle.chain(logits, "f32", fac["U"], fac["V"], last)
    U = workloads.bf16_bits_to_f32(fac["U"]).astype(np.float64)
    V = workloads.bf16_bits_to_f32(fac["V"]).astype(np.float64)
    Ui = [[_exact_int(float(x)) >> 133 for x in row] for row in U.tolist()]
    Vi = [[_exact_int(float(x)) >> 133 for x in row] for row in V.tolist()]
    # Ui, Vi are in units of 2^-133; their products are in units of 2^-266
    N, K, vocab = logits.shape
    for n in range(N):
        prev = int(last[n])
        for k in range(K):
            lk = [_exact_int(float(x)) for x in logits[n, k].tolist()]
            up = Ui[prev]
            best, arg = None, -1
            for v in range(vocab):
                val = lk[v] + sum(a * b for a, b in zip(up, Vi[v]))
                if best is None or val > best:
                    best, arg = val, v
            assert r["draft"][n, k] == arg, (n, k)
            assert r["score"][n, k] == float(Fraction(best, 1 << SCALE))
            prev = arg


def test_exact_prefix_sums_match_fsum():
    rng = np.random.default_rng(5)
    for trial in range(6):
        x = np.sort(rng.uniform(0, 1, 300) ** rng.integers(1, 40))[::-1]
        if trial == 5:
            x[150:] = x[150:] * 1e-300           # deep subnormal tail
        P = oracle.exact_prefix_sums(x)
        for b in range(len(x) + 1):
            assert P[b] == math.fsum(x[:b].tolist())


def test_exact_prefix_sum_differs_from_left_to_right_doubles():
    # 1 + 2^-53 is a tie that rounds to even (1.0) when added alone; the exact
    # sum with 2^-105 lies above the midpoint and rounds up
    x = np.array([1.0, 2.0 ** -53, 2.0 ** -105])
    P = oracle.exact_prefix_sums(x)
    assert P[3] == 1.0 + 2.0 ** -52
    assert np.cumsum(x)[2] == 1.0


def test_survival_is_left_to_right_double_product():
    """np.cumprod multiplies left to right; each step is one correctly
    rounded double product, which is what the device reproduces."""
    rng = np.random.default_rng(9)
    conf = rng.uniform(0, 1, size=(50, 15)).astype(np.float32)
    s, _ = oracle.survival(conf, np.ones(50, np.uint8))
    for n in range(50):
        acc = 1.0
        for k in range(15):
            acc = acc * float(conf[n, k])
            assert s[n, k] == acc
