"""GPU parity of the fused output projection (dspark_chain_lmhead) against
the oracle.

"DSpark on MAX", *What DSpark is*, items 2-3: adj = h . W^T + U[prev] . V^T
with the backbone logits never stored.  The oracle computes h . W^T in fp64
and runs the same chain; the device accumulates bf16 products in fp32 over
d + rank terms, so tokens follow the chain's near-tie rule and scores agree
to 1e-5 relative.  Shapes span several tiles with ragged batch, vocabulary
and rank tails, both hidden-state layouts, and the full headline size
(every row).
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


def _inputs(N, K, vocab, d, rank, seed, sd=2.0):
    rng = np.random.default_rng(seed)
    h = workloads.f32_to_bf16_bits(rng.standard_normal((N, K, d), dtype=np.float32))
    W = workloads.f32_to_bf16_bits(
        rng.standard_normal((vocab, d), dtype=np.float32) * np.float32(sd / np.sqrt(d)))
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    last = rng.integers(0, vocab, N).astype(np.int32)
    return h, W, U, V, last


def _run(h, W, U, V, last, layout="nkv", pad=0):
    import torch
    from gpu_harness import up, up_bf16, DEV
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    N, K, d = h.shape
    base = h if layout == "nkv" else np.ascontiguousarray(h.transpose(1, 0, 2))
    if pad:
        padded = np.zeros(base.shape[:-1] + (d + pad,), np.uint16)
        padded[..., :d] = base
        base = padded
    th = up_bf16(base)
    row = d + pad
    sn, sk = (K * row, row) if layout == "nkv" else (row, N * row)
    tW, tU, tV, tl = up_bf16(W), up_bf16(U), up_bf16(V), up(last)
    draft = torch.full((N, K), -1, dtype=torch.int32, device=DEV)
    score = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    ws = D.new_workspace(D.dspark_chain_workspace_size(N, K), DEV)
    D.dspark_chain_lmhead(th, tW, tU, tV, tl, draft, score, ws, N=N, K=K, d=d,
                          stride_n=sn, stride_k=sk)
    torch.cuda.synchronize()
    return (draft.cpu().numpy().astype(np.int64), score.cpu().numpy(),
            D.dspark_read_status(ws))


def _check(got, score, h, W, U, V, last, rows=None):
    from gpu_harness import check_chain
    rows = np.arange(h.shape[0]) if rows is None else np.asarray(rows)
    logits = oracle.lmhead_logits(h[rows], W)
    return check_chain(got[rows], score[rows], logits, "f64", U, V, last[rows])


@pytest.mark.parametrize("N,K,vocab,d,rank", [
    (1, 1, 256, 64, 16),
    (3, 7, 1024, 128, 16),
    (5, 3, 3000, 64, 64),        # ragged vocabulary tail
    (130, 2, 2048, 256, 80),     # two request tiles, rank not /64
    (257, 3, 4104, 192, 256),    # three request tiles, ragged both ways
    (64, 5, 5000, 512, 128),
])
def test_shapes(N, K, vocab, d, rank):
    h, W, U, V, last = _inputs(N, K, vocab, d, rank, seed=N + K + vocab + d)
    got, score, st = _run(h, W, U, V, last)
    assert st == 0
    assert got.min() >= 0 and got.max() < vocab
    near = _check(got, score, h, W, U, V, last)
    assert near <= max(1, N * K // 100)


@pytest.mark.parametrize("layout,pad", [("knv", 0), ("nkv", 64), ("knv", 8)])
def test_hidden_state_layouts(layout, pad):
    h, W, U, V, last = _inputs(37, 5, 2560, 128, 64, seed=3)
    got, score, st = _run(h, W, U, V, last, layout=layout, pad=pad)
    assert st == 0
    _check(got, score, h, W, U, V, last)


def test_zero_projection_is_the_bias_chain():
    from gpu_harness import run_chain
    h, W, U, V, last = _inputs(70, 4, 3072, 128, 64, seed=12)
    got, _, st = _run(h, np.zeros_like(W), U, V, last)
    assert st == 0
    zero = np.zeros((70, 4, 3072), np.float32)
    ref, _, _ = run_chain(zero, "f32", U, V, last)
    np.testing.assert_array_equal(got, ref)


def test_bad_last_token_and_many_vocabulary_tiles():
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    h, W, U, V, last = _inputs(200, 3, 65536, 256, 256, seed=8)
    last[7] = -5
    got, score, st = _run(h, W, U, V, last)
    assert st == D.DEV_TOKEN_OOR
    fixed = last.copy()
    fixed[7] = 0
    rows = np.random.default_rng(0).choice(200, 24, replace=False)
    rows[0] = 7
    assert _check(got, score, h, W, U, V, fixed, rows=rows) <= 2


def test_headline_full_size():
    cfg = workloads.get_config("headline")
    x = workloads.make_lmhead_inputs(cfg)
    fac = workloads.make_chain_factors(cfg)
    last = workloads.make_last_token(cfg)
    got, score, st = _run(x["h"], x["W"], fac["U"], fac["V"], last)
    assert st == 0
    assert got.min() >= 0 and got.max() < cfg.vocab
    from gpu_harness import report_near
    near = _check(got, score, x["h"], x["W"], fac["U"], fac["V"], last)
    report_near("lmhead headline (d 2048)", near, cfg.N * cfg.K)
    assert near <= max(1, cfg.N * cfg.K // 100)


def test_random_shapes():
    """Random shapes (batch, positions, vocabulary a multiple of 8, d a
    multiple of 64, rank a multiple of 16) and hidden-state layouts."""
    rng = np.random.default_rng(515)
    for case in range(6):
        N = int(rng.integers(1, 300))
        K = int(rng.integers(1, 7))
        vocab = 8 * int(rng.integers(1, 700))
        d = 64 * int(rng.integers(1, 9))
        rank = 16 * int(rng.integers(1, 17))
        layout = "nkv" if rng.uniform() < 0.6 else "knv"
        pad = int(rng.choice([0, 8, 64]))
        h, W, U, V, last = _inputs(N, K, vocab, d, rank, seed=1000 + case,
                                   sd=float(rng.uniform(1.0, 3.0)))
        got, score, st = _run(h, W, U, V, last, layout=layout, pad=pad)
        assert st == 0, case
        assert got.min() >= 0 and got.max() < vocab, case
        assert _check(got, score, h, W, U, V, last) <= max(1, N * K // 100), case
