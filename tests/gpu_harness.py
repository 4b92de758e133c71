"""Helpers of the GPU parity tests: upload numpy inputs, call the C ABI
through the Python binding, and compare with the oracle under the tolerance
rules of the test plan.

Chain tolerance: integer tokens must equal the oracle's, except where the
oracle's top-2 margin is below 1e-3 * |max| (the adjusted values are fp32 on
the device, fp64 in the oracle); there the device token must be within
1e-3 * |max| of the maximum, and the rest of that row is checked for
validity given the device's own earlier tokens.  Scores agree to 1e-5
relative.  Sampled draws (the two-level block draw) must equal the
oracle's except at a near-tie of the block keys, or, inside the block,
where the uniform lands within 1e-5 of the block's weight of a boundary;
after a tolerated divergence the row continues from the device's token.
Scheduler outputs are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_draft_dspark_gb300 import dspark as D

DEV = "cuda:0"
NEAR_TIE = 1e-3
SCORE_RTOL = 1e-5

# (case, near-tie divergences, rows x positions checked), printed at the end
# of the run by the terminal-summary hook in conftest.py
NEAR_TIE_LOG: list = []


def report_near(case: str, near: int, checked: int) -> None:
    NEAR_TIE_LOG.append((case, int(near), int(checked)))


def up(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def up_bf16(bits: np.ndarray) -> torch.Tensor:
    return up(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def i32(n) -> torch.Tensor:
    return torch.zeros(n, dtype=torch.int32, device=DEV)


# --------------------------------------------------------------- chain
def run_chain(logits: np.ndarray, dtype: str, U: np.ndarray, V: np.ndarray,
              last: np.ndarray, layout: str = "nkv", pad: int = 0,
              with_score: bool = True, sample: dict | None = None):
    """Runs dspark_chain_draft (or dspark_chain_sample with ``sample`` =
    dict(seed, offset, tau)); logits [N, K, vocab] stored in `layout`
    ("nkv" row-major, "knv" position-major) with `pad` extra elements per
    innermost row.  Returns (draft, score, status)."""
    N, K, vocab = logits.shape
    if dtype == "bf16":
        base = np.ascontiguousarray(logits).view(np.int16)
    else:
        base = np.ascontiguousarray(logits, dtype=np.float32)
    if layout == "knv":
        base = np.ascontiguousarray(base.transpose(1, 0, 2))
    if pad:
        shp = base.shape[:-1] + (base.shape[-1] + pad,)
        padded = np.zeros(shp, dtype=base.dtype)
        padded[..., :vocab] = base
        base = padded
    t = up(base)
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    row = vocab + pad
    if layout == "knv":
        stride_n, stride_k = row, N * row
    else:
        stride_n, stride_k = K * row, row
    draft = torch.full((N, K), -1, dtype=torch.int32, device=DEV)
    score = torch.zeros(N, K, dtype=torch.float32, device=DEV) if with_score else None
    ws = D.new_workspace(D.dspark_chain_workspace_size(N, K), DEV)
    kw = dict(N=N, K=K, vocab=vocab, rank=U.shape[1], stride_n=stride_n,
              stride_k=stride_k, logits_dtype=D.BF16 if dtype == "bf16" else D.F32)
    if sample is None:
        D.dspark_chain_draft(t, up_bf16(U), up_bf16(V), up(last.astype(np.int32)),
                             draft, score, ws, **kw)
    else:
        D.dspark_chain_sample(t, up_bf16(U), up_bf16(V), up(last.astype(np.int32)),
                              draft, score, ws, seed=sample["seed"],
                              offset=sample["offset"], temperature=sample["tau"],
                              **kw)
    torch.cuda.synchronize()
    st = D.dspark_read_status(ws)
    return (draft.cpu().numpy().astype(np.int64),
            None if score is None else score.cpu().numpy(), st)


def check_chain(got, got_score, logits, dtype, U, V, last, rows=None,
                sample=None):
    """Compares device tokens of `rows` (indices into logits' first axis)
    with the oracle; returns the number of accepted near-tie divergences.
    With ``sample`` the draws are compared with the oracle's two-level draw
    (block keys, then the entry inside the block)."""
    rows = np.arange(logits.shape[0]) if rows is None else np.asarray(rows)
    if sample is not None:
        return _check_sampled(got, got_score, logits, dtype, U, V, last, rows, sample)
    sub = logits[rows]
    ref = oracle.chain(sub, dtype, U, V, np.asarray(last)[rows])

    def position(i, k, prev):
        return oracle.chain_position(oracle.to_f64(sub[i:i + 1, k, :], dtype),
                                     U64, V64, np.array([prev]))

    g = got[rows]
    near = 0
    U64, V64 = oracle.bf16_to_f64(U), oracle.bf16_to_f64(V)
    for i in range(len(rows)):
        diverged = False
        prev_tok = None
        for k in range(sub.shape[1]):
            if not diverged:
                if g[i, k] == ref["draft"][i, k]:
                    if got_score is not None:
                        _score_ok(got_score[rows[i], k], ref["score"][i, k])
                    continue
                # tolerated only at a near-tie of the oracle's own values
                mx, mg = ref["score"][i, k], ref["margin"][i, k]
                tol = NEAR_TIE * abs(mx)
                r = position(i, k, _prev(ref["draft"], last, rows, i, k))
                assert mg < tol and r["adj"][0, g[i, k]] >= mx - tol, \
                    (rows[i], k, g[i, k], ref["draft"][i, k], mx, mg)
                near += 1
                diverged = True
                prev_tok = g[i, k]
                continue
            # validity of the rest of a diverged row, given the device's
            # own previous token
            r = position(i, k, prev_tok)
            mx = r["score"][0]
            tol = NEAR_TIE * abs(mx)
            assert r["adj"][0, g[i, k]] >= mx - tol, (rows[i], k)
            if g[i, k] != r["tok"][0]:
                assert r["margin"][0] < tol
            prev_tok = g[i, k]
    return near


# the device's block weights come from fp32 ex2 / lg2 approximations, so its
# choice inside a block may differ from the fp64 one where the uniform lands
# this close (relative to the block's total weight) to a boundary
BOUNDARY_TIE = 1e-5


def _draw_tolerated(r, tok):
    """A device draw `tok` that differs from the oracle's (r, one row of
    sample_position) is accepted at a near-tie of the block keys (another
    block whose key is within NEAR_TIE * |max| of the largest) or, inside
    the oracle's block, where the uniform's target lies within BOUNDARY_TIE
    of the total weight of a boundary between the two entries."""
    G = oracle.SAMPLE_BLOCK
    keys, jr = r["keys"][0], int(r["block"][0])
    mx = keys[jr]
    if np.isnan(mx):
        return False
    jd = int(tok) // G
    if jd != jr:
        tol = NEAR_TIE * abs(mx)
        return r["margin"][0] < tol and keys[jd] >= mx - tol
    cum, target = r["cum"][0], r["target"][0]
    ed, er = int(tok) % G, int(r["tok"][0]) % G
    lo, hi = min(ed, er), max(ed, er)
    gap = np.min(np.abs(cum[lo:hi] - target))
    return gap <= BOUNDARY_TIE * cum[-1]


def _check_sampled(got, got_score, logits, dtype, U, V, last, rows, sample):
    seed, offset, tau = int(sample["seed"]), int(sample["offset"]), float(sample["tau"])
    sub = logits[rows]
    ref = oracle.chain(sub, dtype, U, V, np.asarray(last)[rows], sample=sample, rows=rows)
    U64, V64 = oracle.bf16_to_f64(U), oracle.bf16_to_f64(V)
    g = got[rows]
    near = 0
    for i in range(len(rows)):
        prev = None  # the device's previous token once the row has diverged
        for k in range(sub.shape[1]):
            if prev is None and g[i, k] == ref["draft"][i, k]:
                if got_score is not None:
                    _score_ok(got_score[rows[i], k], ref["score"][i, k], floor=1.0)
                continue
            p = _prev(ref["draft"], last, rows, i, k) if prev is None else prev
            adj = oracle.chain_position(oracle.to_f64(sub[i:i + 1, k, :], dtype),
                                        U64, V64, np.array([p]))["adj"]
            r = oracle.sample_position(adj, tau, seed, offset, [rows[i]], k)
            if g[i, k] != r["tok"][0]:
                assert _draw_tolerated(r, g[i, k]), \
                    (rows[i], k, g[i, k], int(r["tok"][0]), r["score"][0], r["margin"][0])
                near += 1
            prev = int(g[i, k])
    return near


def _prev(draft, last, rows, i, k):
    if k == 0:
        p = int(np.asarray(last)[rows[i]])
        return p
    return int(draft[i, k - 1])


def _score_ok(got, want, floor=1e-3):
    if np.isnan(want):
        assert np.isnan(got)
        return
    if np.isinf(want):
        assert got == want, (got, want)
        return
    assert abs(float(got) - want) <= SCORE_RTOL * max(abs(want), floor), (got, want)


# ----------------------------------------------------------- scheduler
def run_select(conf, mask, cost, T, draft_cost=0.0, flags=0, draft=None,
               fused=True, conf_size=None):
    """Runs the scheduler through the fused call or the four separate calls
    (with ``conf_size``: stale sizing, fused or composed from the separate
    calls); returns numpy outputs and the status word."""
    N, K = conf.shape
    d_conf = up(np.asarray(conf, np.float32))
    d_mask = None if mask is None else up(np.asarray(mask, np.uint8))
    d_cost = up(np.asarray(cost, np.float32))
    d_T = up(np.array([T], np.int32))
    d_draft = None if draft is None else up(np.asarray(draft, np.int32))
    surv = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    srt = torch.full((N * K,), -1, dtype=torch.int32, device=DEV)
    pre = torch.full((N * K + 1,), -1.0, dtype=torch.float64, device=DEV)
    ne, ns, B = i32(1), i32(1), i32(1)
    obj = torch.zeros(1, dtype=torch.float64, device=DEV)
    ln, cu = i32(N), i32(N + 1)
    vi = torch.full((N * K,), -1, dtype=torch.int32, device=DEV)
    vt = torch.full((N * K,), -1, dtype=torch.int32, device=DEV)
    ws = D.new_workspace(D.dspark_select_workspace_size(N, K, len(cost)), DEV)
    if conf_size is not None and fused:
        D.dspark_select_step_stale(up(np.asarray(conf_size, np.float32)), d_conf,
                                   d_mask, d_cost, d_T, draft_cost, flags,
                                   d_draft, surv, srt, pre, ne, ns, B, obj, ln,
                                   cu, vi, vt if d_draft is not None else None,
                                   ws)
    elif conf_size is not None:
        # size from the old buffer, then order the current one and allocate
        s_old = torch.zeros(N, K, dtype=torch.float32, device=DEV)
        srt_old = torch.full((N * K,), -1, dtype=torch.int32, device=DEV)
        pre_cur = torch.full((N * K + 1,), -1.0, dtype=torch.float64, device=DEV)
        D.dspark_survival_topb(up(np.asarray(conf_size, np.float32)), d_mask,
                               s_old, srt_old, pre, ne, ns, ws)
        D.dspark_choose_budget(pre, ne, ns, d_cost, d_T, draft_cost, flags, B,
                               obj, ws)
        D.dspark_survival_topb(d_conf, d_mask, surv, srt, pre_cur, ne, ns, ws)
        D.dspark_allocate_prefix(srt, B, N, K, ln, ws)
        D.dspark_compact_verify(ln, d_draft, N, K, cu, vi,
                                vt if d_draft is not None else None, ws)
    elif fused:
        D.dspark_select_step(d_conf, d_mask, d_cost, d_T, draft_cost, flags,
                             d_draft, surv, srt, pre, ne, ns, B, obj, ln, cu,
                             vi, vt if d_draft is not None else None, ws)
    else:
        D.dspark_survival_topb(d_conf, d_mask, surv, srt, pre, ne, ns, ws)
        D.dspark_choose_budget(pre, ne, ns, d_cost, d_T, draft_cost, flags, B,
                               obj, ws)
        D.dspark_allocate_prefix(srt, B, N, K, ln, ws)
        D.dspark_compact_verify(ln, d_draft, N, K, cu, vi,
                                vt if d_draft is not None else None, ws)
    torch.cuda.synchronize()
    st = D.dspark_read_status(ws)
    out = dict(survival=surv.cpu().numpy(), sorted=srt.cpu().numpy(),
               prefix=pre.cpu().numpy(), n_eligible=int(ne.item()),
               n_sampling=int(ns.item()), B=int(B.item()),
               objective=float(obj.item()), draft_len=ln.cpu().numpy(),
               cu_len=cu.cpu().numpy(), verify_idx=vi.cpu().numpy(),
               verify_tok=vt.cpu().numpy(), status=st)
    return out


def check_select(got, conf, mask, cost, T, draft_cost=0.0, flags=0, draft=None,
                 conf_size=None):
    N, K = np.asarray(conf).shape
    if conf_size is None:
        r = oracle.select_step(conf, mask, cost, T, draft_cost, flags, draft)
    else:
        r = oracle.select_step_stale(conf_size, conf, mask, cost, T, draft_cost,
                                     flags, draft)
    S = r["n_eligible"]
    # survival: fp64 product rounded once to fp32 on both sides
    np.testing.assert_array_equal(got["survival"], r["survival"].astype(np.float32))
    assert got["n_eligible"] == S and got["n_sampling"] == r["n_sampling"]
    np.testing.assert_array_equal(got["sorted"][:S], r["order"])
    # exact prefix sums: identical bits
    np.testing.assert_array_equal(got["prefix"][:S + 1], r["prefix"])
    assert got["B"] == r["B"], (got["B"], r["B"])
    if np.isnan(r["objective"]):
        assert np.isnan(got["objective"])
    else:
        assert got["objective"] == r["objective"], (got["objective"], r["objective"])
    np.testing.assert_array_equal(got["draft_len"], r["draft_len"])
    np.testing.assert_array_equal(got["cu_len"], r["cu_len"])
    B = r["B"]
    np.testing.assert_array_equal(got["verify_idx"][:B], r["verify_idx"])
    assert np.all(got["verify_idx"][B:] == -1)
    if draft is not None:
        np.testing.assert_array_equal(got["verify_tok"][:B], r["verify_tok"])
    want_status = r["status"]
    assert got["status"] == want_status, (got["status"], want_status)
    return r
