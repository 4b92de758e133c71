"""A bounded wait inside the chain kernel runs out: the kernel must report
DSPARK_DEV_TIMEOUT, return, write no out-of-range token, and leave the CUDA
context usable for the next call.

The workspace's test hook makes every barrier between positions wait for one
arrival more than can come (a count nobody completes), so the wait ends by
its time limit; nothing faults, traps or hangs.
"""
import time

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


def test_barrier_wait_runs_out_and_context_survives():
    import torch
    import __graft_entry__
    from gpu_harness import up, up_bf16
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    __graft_entry__.build()
    N, K, vocab, rank = 130, 3, 4096, 64
    rng = np.random.default_rng(41)
    x = rng.standard_normal((N, K, vocab), dtype=np.float32) * np.float32(2.0)
    logits = workloads.f32_to_bf16_bits(x)
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    last = rng.integers(0, vocab, N).astype(np.int32)
    d_logits = up(logits.view(np.int16)).view(torch.bfloat16)
    d_U, d_V, d_last = up_bf16(U), up_bf16(V), up(last)

    ws = D.new_workspace(D.dspark_chain_workspace_size(N, K))
    ws.view(torch.int32)[1] = 1          # test hook: barriers cannot complete
    draft = torch.full((N, K), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    D.dspark_chain_draft(d_logits, d_U, d_V, d_last, draft, None, ws)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    st = D.dspark_read_status(ws)
    assert st & D.DEV_TIMEOUT, st
    assert 0.5 < dt < 30.0, dt
    d = draft.cpu().numpy()
    assert np.all((d == -1) | ((d >= 0) & (d < vocab)))

    # the same context and workspace work normally once the hook is cleared
    ws.view(torch.int32)[1] = 0
    D.dspark_clear_status(ws)
    draft.fill_(-1)
    D.dspark_chain_draft(d_logits, d_U, d_V, d_last, draft, None, ws)
    torch.cuda.synchronize()
    assert D.dspark_read_status(ws) == 0
    ref = oracle.chain(logits, "bf16", U, V, last)
    np.testing.assert_array_equal(draft.cpu().numpy(), ref["draft"])


def _hooked(ws, on):
    import torch
    ws.view(torch.int32)[1] = 1 if on else 0


def test_sampling_and_fused_projection_time_out_and_recover():
    """The same hook on the probabilistic chain (12 epilogue warps, of which
    only the first four wait at the barrier) and on the fused output
    projection: both report DSPARK_DEV_TIMEOUT, write no out-of-range token
    and leave the context usable."""
    import torch
    import __graft_entry__
    from gpu_harness import up, up_bf16, check_chain
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    __graft_entry__.build()
    N, K, vocab, rank, d = 130, 3, 4096, 64, 128
    rng = np.random.default_rng(43)
    x = rng.standard_normal((N, K, vocab), dtype=np.float32) * np.float32(2.0)
    logits = workloads.f32_to_bf16_bits(x)
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    h = workloads.f32_to_bf16_bits(rng.standard_normal((N, K, d), dtype=np.float32))
    W = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, d), dtype=np.float32) * np.float32(2 / np.sqrt(d)))
    last = rng.integers(0, vocab, N).astype(np.int32)
    d_logits = up(logits.view(np.int16)).view(torch.bfloat16)
    d_U, d_V, d_last, d_h, d_W = up_bf16(U), up_bf16(V), up(last), up_bf16(h), up_bf16(W)
    ws = D.new_workspace(D.dspark_chain_workspace_size(N, K))
    draft = torch.full((N, K), -1, dtype=torch.int32, device="cuda")
    score = torch.zeros(N, K, dtype=torch.float32, device="cuda")
    sm = dict(seed=5, offset=0, tau=1.0)
    calls = [
        lambda: D.dspark_chain_sample(d_logits, d_U, d_V, d_last, draft, score, ws,
                                      seed=sm["seed"], offset=sm["offset"],
                                      temperature=sm["tau"]),
        lambda: D.dspark_chain_lmhead(d_h, d_W, d_U, d_V, d_last, draft, score, ws),
    ]
    for call in calls:
        _hooked(ws, True)
        D.dspark_clear_status(ws)
        draft.fill_(-1)
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert D.dspark_read_status(ws) & D.DEV_TIMEOUT
        assert 0.5 < dt < 30.0, dt
        dd = draft.cpu().numpy()
        assert np.all((dd == -1) | ((dd >= 0) & (dd < vocab)))
        _hooked(ws, False)
        D.dspark_clear_status(ws)
        call()
        torch.cuda.synchronize()
        assert D.dspark_read_status(ws) == 0
    # after both, the last (fused projection) result matches the oracle
    got = draft.cpu().numpy().astype(np.int64)
    assert check_chain(got, score.cpu().numpy(), oracle.lmhead_logits(h, W), "f64",
                       U, V, last) <= 2
