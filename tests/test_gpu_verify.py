"""GPU parity of dspark_greedy_verify against the oracle (bit-exact).

"DSpark on MAX", *The kernel pass*, item 2 (compare-only acceptance under
greedy sampling) and "How DSpark Speeds Up LLM Inference", *Context* (keep
the longest matching run plus the target's next token).  Target rows are
synthetic: N(0, 2) logits where, with probability equal to the slot's
confidence, the draft token is planted as the row's maximum, so accepted
lengths follow the confidences.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _setup(cfg_name, vocab=None, dtype="bf16", seed=0, **over):
    cfg = workloads.get_config(cfg_name, **over)
    vocab = vocab or cfg.vocab
    sel = workloads.make_select_inputs(cfg)
    rng = np.random.default_rng(1000 + seed)
    draft = rng.integers(0, vocab, size=(cfg.N, cfg.K)).astype(np.int32)
    r = oracle.select_step(sel["conf"], sel["mask"], sel["cost"], sel["T"],
                           draft=draft)
    ln, cu, mask = r["draft_len"], r["cu_len"], sel["mask"]
    rows = oracle.verify_rows(ln, mask)
    R = int(rows[-1])
    x = rng.standard_normal((max(R, 1), vocab), dtype=np.float32) * np.float32(2.0)
    for n in range(cfg.N):
        if mask[n] == 0:
            continue
        for j in range(int(ln[n])):
            if rng.uniform() < sel["conf"][n, j]:
                x[rows[n] + j, draft[n, j]] = x[rows[n] + j].max() + 1.0
    tl = workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x
    return cfg, draft, ln, cu, mask, tl


def _run(tl, dtype, draft, ln, cu, mask, vocab):
    import torch
    from gpu_harness import up, i32
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    N, K = draft.shape
    t = up(tl.view(np.int16)).view(torch.bfloat16) if dtype == "bf16" else up(tl)
    tgt = torch.full((N * (K + 1),), -7, dtype=torch.int32, device="cuda")
    acc, bon = i32(N), i32(N)
    ws = D.new_workspace(256)
    D.dspark_greedy_verify(t, up(draft), up(ln.astype(np.int32)),
                           up(cu.astype(np.int32)), up(mask), tgt, acc, bon, ws,
                           vocab=vocab, row_stride=tl.shape[1],
                           logits_dtype=D.BF16 if dtype == "bf16" else D.F32)
    torch.cuda.synchronize()
    return (tgt.cpu().numpy(), acc.cpu().numpy(), bon.cpu().numpy(),
            D.dspark_read_status(ws))


def _check(tl, dtype, draft, ln, cu, mask, vocab):
    tgt, acc, bon, st = _run(tl, dtype, draft, ln, cu, mask, vocab)
    ref = oracle.greedy_verify(tl, dtype, draft, ln, mask)
    R = int(ref["rows"][-1])
    np.testing.assert_array_equal(tgt[:R], ref["target_argmax"])
    assert np.all(tgt[R:] == -7)
    np.testing.assert_array_equal(acc, ref["accepted"])
    np.testing.assert_array_equal(bon, ref["bonus"])
    return ref, st


@pytest.mark.parametrize("name,vocab,dtype", [
    ("dsv4", 65536, "bf16"),
    ("conc64", 4096, "f32"),
    ("tiny", 1000, "bf16"),       # one partial chunk per row, many rows per CTA
    ("gemma4_12b", None, "bf16"),
])
def test_workloads(name, vocab, dtype):
    cfg, draft, ln, cu, mask, tl = _setup(name, vocab, dtype)
    ref, st = _check(tl, dtype, draft, ln, cu, mask, vocab or cfg.vocab)
    assert st == 0
    assert 0 <= ref["accepted"].max()


def test_headline_full_size():
    cfg, draft, ln, cu, mask, tl = _setup("headline")
    ref, st = _check(tl, "bf16", draft, ln, cu, mask, cfg.vocab)
    assert st == 0
    acc = ref["accepted"][mask == 1]
    assert acc.mean() > 0.5            # planted matches are accepted


def test_nan_ties_and_minus_inf_rows():
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    cfg, draft, ln, cu, mask, tl = _setup("tiny", 4096, "f32", seed=3)
    R = tl.shape[0]
    tl[0, 2000] = np.nan
    tl[0, 17] = np.nan                 # first NaN wins
    tl[1, :] = -np.inf                 # index 0
    tl[2, 100] = tl[2, 3000] = 1e6     # tie: lower index
    tl[R - 1, 4095] = 1e7              # last element of the last row
    ref, st = _check(tl, "f32", draft, ln, cu, mask, 4096)
    assert ref["target_argmax"][0] == 17 and ref["target_argmax"][1] == 0
    assert ref["target_argmax"][2] == 100
    assert st & D.DEV_NAN_LOGIT


def test_nobody_sampling():
    cfg, draft, ln, cu, mask, tl = _setup("tiny", 1024, "bf16", seed=5)
    mask = np.zeros_like(mask)
    ln = np.zeros_like(ln)
    cu = np.zeros_like(cu)
    tgt, acc, bon, st = _run(tl, "bf16", draft, ln, cu, mask, 1024)
    assert np.all(acc == -1) and np.all(bon == -1) and np.all(tgt == -7)


def test_random_batches():
    """Random batches: request count, draft length, vocabulary (a multiple of
    8 for bf16, of 4 for fp32), sampling mask, per-request verify lengths
    and planted matches; every output equals the oracle's bit for bit."""
    rng = np.random.default_rng(77)
    for case in range(10):
        N = int(rng.integers(1, 200))
        K = int(rng.integers(1, 33))
        dtype = "bf16" if rng.uniform() < 0.7 else "f32"
        vocab = (8 if dtype == "bf16" else 4) * int(rng.integers(1, 2000))
        mask = (rng.uniform(size=N) < rng.uniform(0.2, 1.0)).astype(np.uint8)
        ln = np.where(mask == 1, rng.integers(0, K + 1, N), 0).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(ln)]).astype(np.int32)
        draft = rng.integers(0, vocab, (N, K)).astype(np.int32)
        rows = oracle.verify_rows(ln, mask)
        R = int(rows[-1])
        x = rng.standard_normal((max(R, 1), vocab), dtype=np.float32) * np.float32(2.0)
        for n in range(N):
            for j in range(int(ln[n])):
                if rng.uniform() < 0.6:
                    x[rows[n] + j, draft[n, j]] = x[rows[n] + j].max() + 1.0
        tl = workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x
        _, st = _check(tl, dtype, draft, ln, cu, mask, vocab)
        assert st == 0, case
