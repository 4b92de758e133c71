"""GPU parity at the limits the C ABI documents.

The chain (argmax and probabilistic), the fused output projection and the
greedy verification at K = 32 positions, the smallest vocabularies (one
16-byte vector of logits), ranks 16 and 256, and the largest batch one
cooperative launch holds (128 requests per SM), plus the first batch past it
(rejected before launch).  Same tolerance rules as the other parity tests.
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


def _chain_inputs(N, K, vocab, rank, dtype, seed, uv_sd=0.05):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, K, vocab), dtype=np.float32) * np.float32(2.0)
    logits = workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(uv_sd))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(uv_sd))
    last = rng.integers(0, vocab, N).astype(np.int32)
    return logits, U, V, last


@pytest.mark.parametrize("N,K,vocab,rank,dtype", [
    (3, 32, 8, 16, "bf16"),       # smallest bf16 vocabulary, most positions
    (2, 32, 4, 16, "f32"),        # smallest fp32 vocabulary
    (64, 32, 2048, 256, "bf16"),  # K = 32 at full rank
    (1100, 2, 1024, 32, "bf16"),  # nine request tiles
])
def test_chain_limits(N, K, vocab, rank, dtype):
    from gpu_harness import run_chain, check_chain
    logits, U, V, last = _chain_inputs(N, K, vocab, rank, dtype, seed=N * K + vocab)
    got, score, st = run_chain(logits, dtype, U, V, last)
    assert st == 0
    assert got.min() >= 0 and got.max() < vocab
    assert check_chain(got, score, logits, dtype, U, V, last) <= max(1, N * K // 100)


def test_chain_largest_batch_and_one_past_it():
    import torch
    from gpu_harness import run_chain, check_chain
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = 128 * sms
    logits, U, V, last = _chain_inputs(N, 1, 64, 16, "bf16", seed=9)
    got, score, st = run_chain(logits, "bf16", U, V, last)
    assert st == 0
    rows = np.random.default_rng(1).choice(N, 256, replace=False)
    assert check_chain(got, score, logits, "bf16", U, V, last, rows=rows) <= 2
    with pytest.raises(D.DsparkError) as e:
        run_chain(np.concatenate([logits, logits[:1]]), "bf16", U, V,
                  np.concatenate([last, last[:1]]))
    assert e.value.code == D.ERR_UNSUPPORTED


@pytest.mark.parametrize("N,K,vocab,rank", [(5, 32, 64, 16), (3, 4, 8, 16)])
def test_sampling_limits(N, K, vocab, rank):
    from gpu_harness import run_chain, check_chain
    logits, U, V, last = _chain_inputs(N, K, vocab, rank, "bf16", seed=K + vocab)
    sm = dict(seed=123456789, offset=7, tau=1.0)
    got, score, st = run_chain(logits, "bf16", U, V, last, sample=sm)
    assert st == 0
    assert got.min() >= 0 and got.max() < vocab
    assert check_chain(got, score, logits, "bf16", U, V, last, sample=sm) <= max(1, N * K // 50)


@pytest.mark.parametrize("N,K,vocab,d,rank", [(1, 32, 8, 64, 16), (300, 2, 1000, 128, 256)])
def test_lmhead_limits(N, K, vocab, d, rank):
    import torch
    from gpu_harness import up, up_bf16, DEV, check_chain
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    rng = np.random.default_rng(N + d)
    h = workloads.f32_to_bf16_bits(rng.standard_normal((N, K, d), dtype=np.float32))
    W = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, d), dtype=np.float32) * np.float32(2 / np.sqrt(d)))
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    last = rng.integers(0, vocab, N).astype(np.int32)
    th, tW, tU, tV, tl = up_bf16(h), up_bf16(W), up_bf16(U), up_bf16(V), up(last)
    draft = torch.full((N, K), -1, dtype=torch.int32, device=DEV)
    score = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    ws = D.new_workspace(D.dspark_chain_workspace_size(N, K), DEV)
    D.dspark_chain_lmhead(th, tW, tU, tV, tl, draft, score, ws)
    torch.cuda.synchronize()
    assert D.dspark_read_status(ws) == 0
    got = draft.cpu().numpy().astype(np.int64)
    assert got.min() >= 0 and got.max() < vocab
    logits = oracle.lmhead_logits(h, W)
    assert check_chain(got, score.cpu().numpy(), logits, "f64", U, V, last) <= max(1, N * K // 100)


def test_verify_k32_smallest_vocabulary():
    import torch
    from gpu_harness import up, i32
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    rng = np.random.default_rng(3)
    N, K, vocab = 40, 32, 8
    mask = (rng.uniform(size=N) < 0.8).astype(np.uint8)
    ln = np.where(mask == 1, rng.integers(0, K + 1, N), 0).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(ln)]).astype(np.int32)
    draft = rng.integers(0, vocab, (N, K)).astype(np.int32)
    rows = oracle.verify_rows(ln, mask)
    R = int(rows[-1])
    x = rng.standard_normal((R, vocab), dtype=np.float32)
    for n in range(N):
        for j in range(int(ln[n])):
            if mask[n] and rng.uniform() < 0.7:
                x[rows[n] + j, draft[n, j]] = x[rows[n] + j].max() + 1.0
    tl = workloads.f32_to_bf16_bits(x)
    tgt = torch.full((N * (K + 1),), -7, dtype=torch.int32, device="cuda")
    acc, bon = i32(N), i32(N)
    ws = D.new_workspace(256)
    D.dspark_greedy_verify(up(tl.view(np.int16)).view(torch.bfloat16), up(draft), up(ln),
                           up(cu), up(mask), tgt, acc, bon, ws)
    torch.cuda.synchronize()
    ref = oracle.greedy_verify(tl, "bf16", draft, ln, mask)
    np.testing.assert_array_equal(tgt.cpu().numpy()[:R], ref["target_argmax"])
    np.testing.assert_array_equal(acc.cpu().numpy(), ref["accepted"])
    np.testing.assert_array_equal(bon.cpu().numpy(), ref["bonus"])
    assert D.dspark_read_status(ws) == 0


def test_special_values_and_odd_position_ties():
    """Ties at odd positions (the vocabulary is swept downwards there, so the
    lower index is met last), +inf pairs, NaN beating +inf, and NaN reaching
    a column through the bias (a NaN in a V row)."""
    from gpu_harness import run_chain
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    N, K, vocab, rank = 5, 4, 40960, 32     # many tiles per CTA at every position
    logits, U, V, last = _chain_inputs(N, K, vocab, rank, "f32", seed=21)
    V[33000] = V[1000]                      # identical bias for columns 1000 / 33000
    for k in (1, 3):                        # odd positions: downward sweep
        logits[0, k, 1000] = logits[0, k, 33000] = 60.0
    logits[1, 1, 5000] = logits[1, 1, 39000] = np.inf
    logits[2, 3, 7000] = np.inf
    logits[2, 3, 20000] = np.nan            # NaN outranks +inf
    Vf = workloads.bf16_bits_to_f32(V).copy()
    Vf[12345, 3] = np.nan                   # column 12345 is NaN for every row
    Vn = workloads.f32_to_bf16_bits(Vf)
    got, score, st = run_chain(logits, "f32", U, V, last)
    ref = oracle.chain(logits, "f32", U, V, last)
    np.testing.assert_array_equal(got, ref["draft"])
    assert got[0, 1] == 1000 and got[0, 3] == 1000
    assert got[1, 1] == 5000 and score[1, 1] == np.inf
    assert got[2, 3] == 20000
    got2, _, st2 = run_chain(logits, "f32", U, Vn, last)
    ref2 = oracle.chain(logits, "f32", U, Vn, last)
    np.testing.assert_array_equal(got2, ref2["draft"])
    assert np.all(got2 == 12345) and st2 & D.DEV_NAN_LOGIT
