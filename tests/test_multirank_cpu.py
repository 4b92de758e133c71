"""World-size-2 tests on CPU (gloo) of the multi-rank paths.

* bench.py's timing aggregation: the maximum over ranks and job-wide µs per
  step for replicas.
* The sharding the design relies on ("Adaptive Verification in vLLM",
  *Results*: every tensor-parallel rank sees the whole batch): the chain is
  independent per request, so requests split across ranks need no exchange;
  the scheduler couples requests only through the global order, so one
  all-gather of survivals lets every rank reach the same budget and the same
  verify list.  Checked with the oracle on two gloo ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, fn, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    finally:
        dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def _aggregation(rank, world):
    import bench
    t = bench.max_over_ranks(10.0 + rank * 5.0, "cpu")
    return t, bench.job_us_per_step(t, 100, world)


def test_bench_aggregation_two_ranks():
    out = _run(_aggregation)
    for r in (0, 1):
        t, us = out[r]
        assert t == 15.0                       # max over ranks
        assert us == pytest.approx(15.0 * 1e3 / 100 / 2)


def _sharded_step(rank, world):
    import torch
    import torch.distributed as dist
    import oracle
    import workloads
    cfg = workloads.get_config("tiny", N=6, n_nonsampling=1,
                               prefill_tokens_each=4)
    sel = workloads.make_select_inputs(cfg)
    fac = workloads.make_chain_factors(cfg)
    logits = workloads.make_logits_rows(cfg)
    last = workloads.make_last_token(cfg)
    rows = np.arange(cfg.N)[rank::world]                 # request sharding
    mine = oracle.chain(logits[rows], cfg.logits_dtype, fac["U"], fac["V"],
                        last[rows])["draft"]
    # no exchange for the chain; gather only to compare here
    full = torch.zeros(cfg.N, cfg.K, dtype=torch.int64)
    part = torch.zeros(cfg.N, cfg.K, dtype=torch.int64)
    part[torch.from_numpy(rows)] = torch.from_numpy(mine)
    dist.all_reduce(part)
    full = part.numpy()
    # scheduler: local survivals, one all-gather, then the same decision
    s_local, _ = oracle.survival(sel["conf"][rows], sel["mask"][rows])
    s_all = torch.zeros(cfg.N, cfg.K, dtype=torch.float64)
    s_all[torch.from_numpy(rows)] = torch.from_numpy(s_local)
    dist.all_reduce(s_all)
    s_all = s_all.numpy()
    order = oracle.order_slots(s_all, sel["mask"])
    n_s = int(sel["mask"].sum())
    bud = oracle.budget(s_all.reshape(-1)[order], n_s, sel["cost"], sel["T"])
    ln = oracle.allocate(order, bud["B"], cfg.N, cfg.K)
    return full, bud["B"], ln


def test_request_sharding_two_ranks():
    import oracle
    import workloads
    out = _run(_sharded_step)
    cfg = workloads.get_config("tiny", N=6, n_nonsampling=1,
                               prefill_tokens_each=4)
    sel = workloads.make_select_inputs(cfg)
    fac = workloads.make_chain_factors(cfg)
    ref_chain = oracle.chain(workloads.make_logits_rows(cfg), cfg.logits_dtype,
                             fac["U"], fac["V"], workloads.make_last_token(cfg))
    ref = oracle.select_step(sel["conf"], sel["mask"], sel["cost"], sel["T"])
    for r in (0, 1):
        draft, B, ln = out[r]
        np.testing.assert_array_equal(draft, ref_chain["draft"])
        assert B == ref["B"]
        np.testing.assert_array_equal(ln, ref["draft_len"])
