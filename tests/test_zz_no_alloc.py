"""dspark_chain_draft_noalloc against dspark_chain_draft and the oracle.

The no-allocation entry point serves callers that cannot allocate device
memory: engines that reserve all device memory at start-up, plugins under a
host runtime that owns every allocation, and latency-critical code where
cudaMalloc is not permitted.  It must give the same drafts as the workspace
entry point, call after call, even though every call reuses one fixed
scratch array inside the library; the drafts are also checked against the
oracle under the chain's near-tie rule.  This file is collected last so a
stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu


def _inputs(N, K, vocab, rank, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, K, vocab), dtype=np.float32) * np.float32(2.0)
    U = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    V = workloads.f32_to_bf16_bits(rng.standard_normal((vocab, rank), dtype=np.float32) * np.float32(0.05))
    last = rng.integers(0, vocab, N).astype(np.int32)
    return workloads.f32_to_bf16_bits(x), U, V, last


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    import torch
    import __graft_entry__
    from gpu_harness import up, up_bf16, check_chain, SCORE_RTOL
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    __graft_entry__.build()

    cases = [
        # (N, K, vocab, rank, seed, bad_last_token)
        (257, 5, 4104, 256, 1, True),    # three request tiles, ragged tails
        (64, 7, 8192, 128, 2, False),    # different shape right after
    ]
    for N, K, vocab, rank, seed, bad in cases:
        logits, U, V, last = _inputs(N, K, vocab, rank, seed)
        if bad:
            last[3] = vocab + 11          # flagged and replaced by token 0
        d_logits = up(logits.view(np.int16)).view(torch.bfloat16)
        d_U, d_V, d_last = up_bf16(U), up_bf16(V), up(last)

        ref_draft = torch.full((N, K), -1, dtype=torch.int32, device="cuda")
        ref_score = torch.zeros(N, K, dtype=torch.float32, device="cuda")
        ws = D.new_workspace(D.dspark_chain_workspace_size(N, K))
        D.dspark_chain_draft(d_logits, d_U, d_V, d_last, ref_draft, ref_score, ws)

        draft = torch.full((N, K), -1, dtype=torch.int32, device="cuda")
        score = torch.zeros(N, K, dtype=torch.float32, device="cuda")
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
        D.dspark_chain_draft_noalloc(d_logits, d_U, d_V, d_last, draft, score,
                                     status)
        torch.cuda.synchronize()
        got = draft.cpu().numpy()
        np.testing.assert_array_equal(got, ref_draft.cpu().numpy())
        np.testing.assert_allclose(score.cpu().numpy(), ref_score.cpu().numpy(),
                                   rtol=SCORE_RTOL, atol=0)
        want = D.DEV_TOKEN_OOR if bad else 0
        assert int(status.item()) == want
        assert D.dspark_read_status(ws) == want
        # and against the oracle itself
        assert check_chain(got.astype(np.int64), score.cpu().numpy(), logits,
                           "bf16", U, V, last) <= max(1, N * K // 100)


def test_noalloc_rejected_call_leaves_next_call_intact():
    """A call rejected by the host checks returns before touching the GPU;
    the next valid call gives the workspace entry point's drafts and a clear
    status."""
    import torch
    import __graft_entry__
    from gpu_harness import up, up_bf16
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    __graft_entry__.build()
    lib = D.load()
    N, K, vocab, rank = 130, 6, 2048, 64
    logits, U, V, last = _inputs(N, K, vocab, rank, 3)
    d_logits = up(logits.view(np.int16)).view(torch.bfloat16)
    d_U, d_V, d_last = up_bf16(U), up_bf16(V), up(last)
    ref = torch.full((N, K), -1, dtype=torch.int32, device="cuda")
    ws = D.new_workspace(D.dspark_chain_workspace_size(N, K))
    D.dspark_chain_draft(d_logits, d_U, d_V, d_last, ref, None, ws)

    status = torch.full((1,), 0x5A5A, dtype=torch.int32, device="cuda")
    draft = torch.full((N, K), -1, dtype=torch.int32, device="cuda")
    code = lib.dspark_chain_draft_noalloc(
        None, D.BF16, K * vocab, vocab, d_U.data_ptr(), d_V.data_ptr(),
        d_last.data_ptr(), N, K, vocab, rank, draft.data_ptr(), None,
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == D.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == 0x5A5A          # nothing was written
    assert np.all(draft.cpu().numpy() == -1)

    D.dspark_chain_draft_noalloc(d_logits, d_U, d_V, d_last, draft, None, status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(draft.cpu().numpy(), ref.cpu().numpy())
    assert int(status.item()) == 0
