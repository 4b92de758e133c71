#!/usr/bin/env python3
"""Benchmark of the DSpark draft-and-schedule step on one GB300 per rank.

One step = dspark_chain_draft (K = 7 positions of bias GEMM + fused
bias-add/argmax) followed by dspark_select_step (survival, global order,
exact prefix sums, budget, allocation, compaction) over the headline
workload: batch 256, K 7, vocabulary 262144, rank 256, with the DeepSeek-V4
confidence, sampling-mask and stepped cost-table recipe (seeded synthetic
inputs; the pages' datasets are not reproduced).  The two calls are captured
in CUDA graphs and replayed; the timed region replays exactly --steps steps
with CUDA events on the launching stream.  The inputs (939.5 MB of logits,
134 MB of V) are larger than L2, so no flush is needed between steps.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.
Multi-GPU (torchrun): every rank runs an independent replica on its own
batch (the step has no cross-request exchange in the chain; see the design
notes), the timed region is bracketed by barriers and the maximum time over
ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("µs per draft-chain+schedule step at batch 256, K=7, vocab "
          "262144; % of roofline")
WORKLOAD = "headline"
CHAIN_SRC = os.path.join(ROOT, "speculative_decoding_draft_dspark_gb300",
                         "csrc", "chain.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "chain_kernel_headline_ncu.md")
SAMPLE_PROFILE = os.path.join(ROOT, "profiles", "chain_kernel_sample_headline_ncu.md")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-graph", action="store_true",
                    help="launch eagerly instead of replaying CUDA graphs")
    ap.add_argument("--no-extras", "--no-verify", dest="no_extras", action="store_true",
                    help="skip the measurements of the NEXT rows (greedy verify, stale sizing, sampling, fused output projection)")
    ap.add_argument("--serial", action="store_true",
                    help="run the scheduler after the chain on one stream "
                         "instead of alongside it")
    ap.add_argument("--l2", action="store_true",
                    help="measure how much of a V-sized buffer L2 keeps between "
                         "re-reads while a logits-sized stream passes through (the "
                         "chain's access pattern without its compute); run under "
                         "ncu with dram__bytes_read.sum for the DRAM bytes")
    ap.add_argument("--link", action="store_true",
                    help="measure the host-to-device link alone (pinned copies "
                         "on 1/2/4/8 streams, and a kernel reading mapped pinned "
                         "memory), the bound of the e2e number")
    return ap.parse_args()


# --------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device) -> float:
    """Largest value over all ranks of the process group (1 rank: itself)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_step(total_ms: float, steps: int, world: int) -> float:
    """Job-wide microseconds per step: every rank runs its own step in each
    iteration, so one iteration completes `world` steps."""
    return total_ms * 1e3 / steps / world


def algorithmic_bytes_per_launch(cfg) -> float:
    """Minimum HBM bytes of one chain launch (all K draft positions): every
    logits element once, V once, the gathered U rows and the tokens."""
    esz = 2 if cfg.logits_dtype == "bf16" else 4
    logits = cfg.N * cfg.K * cfg.vocab * esz
    v_once = cfg.vocab * cfg.rank * 2
    u_rows = cfg.N * cfg.K * cfg.rank * 2
    tokens = cfg.N * cfg.K * 4 * 2
    return logits + v_once + u_rows + tokens


def flops_per_launch(cfg) -> float:
    return 2.0 * cfg.N * cfg.K * cfg.vocab * cfg.rank


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), \
            d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _recorded(path, field):
    """A per-launch figure from a committed ncu summary, if the summary was
    taken on the current chain kernel source (else None)."""
    if not os.path.exists(path):
        return None
    src_hash = hashlib.sha256(open(CHAIN_SRC, "rb").read()).hexdigest()[:16]
    value = None
    hash_ok = False
    for line in open(path):
        if line.startswith("kernel_source_sha256_16:"):
            hash_ok = line.split(":", 1)[1].strip() == src_hash
        if line.startswith(field + ":"):
            value = float(line.split(":", 1)[1].strip())
    return value if hash_ok else None


def recorded_traffic():
    """Per-launch DRAM bytes of the argmax chain (ncu summary)."""
    return _recorded(TRAFFIC_FILE, "dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = os.path.join("/tmp", f"dspark_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.out):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 active=parts[4], hw=parts[5], hwt=parts[6],
                                 swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.out)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ----------------------------------------------------------- GPU arm
class Step:
    """Device-resident inputs and outputs of one headline step, and the two
    calls that make the step."""

    def __init__(self, cfg, device, seed_offset=0):
        import numpy as np
        import torch
        import workloads
        from speculative_decoding_draft_dspark_gb300 import dspark as D
        self.D = D
        self.cfg = cfg
        dev = device
        self.sel = workloads.make_select_inputs(cfg)
        self.fac = workloads.make_chain_factors(cfg)
        self.last_np = workloads.make_last_token(cfg)
        self.logits_np = workloads.make_logits_rows(cfg)
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        bf = lambda a: up(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
        self.logits = bf(self.logits_np) if cfg.logits_dtype == "bf16" else up(self.logits_np)
        self.U, self.V = bf(self.fac["U"]), bf(self.fac["V"])
        self.last = up(self.last_np)
        self.conf, self.mask = up(self.sel["conf"]), up(self.sel["mask"])
        self.cost = up(self.sel["cost"])
        self.T = torch.tensor([self.sel["T"]], dtype=torch.int32, device=dev)
        N, K = cfg.N, cfg.K
        i32 = lambda n: torch.zeros(n, dtype=torch.int32, device=dev)  # noqa: E731
        self.draft = torch.zeros(N, K, dtype=torch.int32, device=dev)
        self.score = torch.zeros(N, K, dtype=torch.float32, device=dev)
        self.surv = torch.zeros(N, K, dtype=torch.float32, device=dev)
        self.srt = i32(N * K)
        self.pre = torch.zeros(N * K + 1, dtype=torch.float64, device=dev)
        self.ne, self.ns, self.B = i32(1), i32(1), i32(1)
        self.obj = torch.zeros(1, dtype=torch.float64, device=dev)
        self.ln, self.cu, self.vi, self.vt = i32(N), i32(N + 1), i32(N * K), i32(N * K)
        self.cws = D.new_workspace(D.dspark_chain_workspace_size(N, K), dev)
        self.sws = D.new_workspace(D.dspark_select_workspace_size(N, K, len(self.sel["cost"])), dev)
        self.flags = D.COST_FORCE_MONOTONE if cfg.cost_kind == "noisy" else 0

    def chain(self):
        self.D.dspark_chain_draft(self.logits, self.U, self.V, self.last,
                                  self.draft, self.score, self.cws)

    def select(self):
        self.D.dspark_select_step(self.conf, self.mask, self.cost, self.T, 0.0,
                                  self.flags, self.draft, self.surv, self.srt,
                                  self.pre, self.ne, self.ns, self.B, self.obj,
                                  self.ln, self.cu, self.vi, self.vt, self.sws)

    def select_nodraft(self):
        """The scheduler without the draft (verify_tok filled by gather)."""
        self.D.dspark_select_step(self.conf, self.mask, self.cost, self.T, 0.0,
                                  self.flags, None, self.surv, self.srt,
                                  self.pre, self.ne, self.ns, self.B, self.obj,
                                  self.ln, self.cu, self.vi, None, self.sws)

    def gather(self):
        self.D.dspark_gather_verify_tokens(self.vi, self.B, self.draft, self.vt)


def logits_desc(cfg):
    """Element types of the chain's inputs, as the workload line names them."""
    return ("bf16 logits/U/V" if cfg.logits_dtype == "bf16"
            else f"{cfg.logits_dtype} logits, bf16 U/V")


def cost_desc(cfg):
    """The step-cost table's recipe, as the workload line names it."""
    if cfg.cost_kind == "stepped":
        return f"cost table L={cfg.L} stepped to {cfg.cost_cap}"
    if cfg.cost_kind == "noisy":
        return f"cost table L={cfg.L} noisy, forced monotone"
    return f"cost table L={cfg.L} {cfg.cost_kind}"


def workload_desc(cfg):
    """The config.workload string both arms print for the same workload."""
    return (f"{cfg.name}: batch {cfg.N}, K {cfg.K}, vocab {cfg.vocab}, rank "
            f"{cfg.rank}, {logits_desc(cfg)}, {cfg.n_nonsampling} "
            f"chunked-prefill requests, T={cfg.T}, {cost_desc(cfg)}")


def l2_desc(cfg):
    """How the timed loop relates to the 129 MB L2: the logits stream (and V)
    of one step against its size."""
    lb = cfg.N * cfg.K * cfg.vocab * (2 if cfg.logits_dtype == "bf16" else 4)
    vb = cfg.vocab * cfg.rank * 2
    big = lb + vb > 129e6
    return (f"{'inputs larger than' if big else 'inputs within'} L2 (logits "
            f"{lb / 1e6:.1f} MB, V {vb / 1e6:.1f} MB); no flush")


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import workloads
    import __graft_entry__

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    # one process compiles the in-tree library; the others wait and load it
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
        if rank != 0:
            __graft_entry__.build()  # up to date by now: only loads
    cfg = workloads.get_config(args.workload)
    st = Step(cfg, dev)
    D = st.D
    stream = torch.cuda.Stream(device=dev)

    side = torch.cuda.Stream(device=dev)
    serial = args.serial

    # eager warm-up (also sets the kernels' shared-memory attributes)
    with torch.cuda.stream(stream):
        for _ in range(3):
            st.chain()
            st.select()
    stream.synchronize()
    assert D.dspark_read_status(st.cws) == 0 and D.dspark_read_status(st.sws) == 0

    # the three parts of a step: chain (main stream), scheduler (side stream
    # alongside the chain, or main stream after it when --serial) and the
    # verify-token gather after the join.  The timed steps replay them as one
    # CUDA graph per step (no events inside the timed region); a separate
    # pass replays the parts as three graphs with events between them for
    # the per-part breakdown.
    if args.no_graph:
        run_chain = st.chain
        run_select = st.select if serial else st.select_nodraft
        run_gather = st.gather
    else:
        g_chain, g_sel, g_gat = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                 torch.cuda.CUDAGraph())
        with torch.cuda.graph(g_chain, stream=stream):
            st.chain()
        with torch.cuda.graph(g_sel, stream=side if not serial else stream):
            if serial:
                st.select()
            else:
                st.select_nodraft()
        with torch.cuda.graph(g_gat, stream=stream):
            st.gather()
        run_chain, run_select, run_gather = g_chain.replay, g_sel.replay, g_gat.replay
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=stream):
            if serial:
                st.chain()
                st.select()
            else:
                fork_c = torch.cuda.Event()
                fork_c.record(stream)
                side.wait_event(fork_c)
                st.chain()
                with torch.cuda.stream(side):
                    st.select_nodraft()
                join_c = torch.cuda.Event()
                join_c.record(side)
                stream.wait_event(join_c)
                st.gather()

    def step(e=None):
        if serial:
            if e is not None:
                e[0].record(stream)
            with torch.cuda.stream(stream):
                run_chain()
            if e is not None:
                e[1].record(stream)
            with torch.cuda.stream(stream):
                run_select()
            if e is not None:
                e[2].record(stream)
                e[3].record(stream)
            return
        fork = e[0] if e is not None else torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        with torch.cuda.stream(stream):
            run_chain()
        if e is not None:
            e[1].record(stream)
        with torch.cuda.stream(side):
            run_select()
        joined = e[2] if e is not None else torch.cuda.Event()
        joined.record(side)
        stream.wait_event(joined)
        with torch.cuda.stream(stream):
            run_gather()
        if e is not None:
            e[3].record(stream)

    if args.no_graph:
        timed_step = step
    else:
        def timed_step():
            with torch.cuda.stream(stream):
                g_step.replay()

    K_steps, W = args.steps, args.warmup
    for _ in range(W):
        timed_step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler come up
    t_host0 = time.perf_counter()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K_steps):
        timed_step()
    end.record(stream)
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)

    # per-part breakdown (separate pass, events between the parts)
    n_b = max(1, min(K_steps, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_b)]
    for _ in range(3):
        step()
    for i in range(n_b):
        step(ev[i])
    torch.cuda.synchronize()
    chain_us = [ev[i][0].elapsed_time(ev[i][1]) * 1e3 for i in range(n_b)]
    if serial:
        sel_us = [ev[i][1].elapsed_time(ev[i][2]) * 1e3 for i in range(n_b)]
    else:  # the scheduler starts with the chain
        sel_us = [ev[i][0].elapsed_time(ev[i][2]) * 1e3 for i in range(n_b)]
    step_us = [ev[i][0].elapsed_time(ev[i][3]) * 1e3 for i in range(n_b)]
    total_ms = max_over_ranks(total_ms, dev)

    # the timed steps raised no device status bit (cheap integrity check)
    assert D.dspark_read_status(st.cws) == 0 and D.dspark_read_status(st.sws) == 0

    ms_per_iter = total_ms / K_steps
    value_us = job_us_per_step(total_ms, K_steps, world)
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    chain_med = statistics.median(chain_us)
    per_launch_s = chain_med * 1e-6  # the chain is one launch per step
    achieved_gbs = algorithmic_bytes_per_launch(cfg) / per_launch_s / 1e9
    achieved_tf = flops_per_launch(cfg) / per_launch_s / 1e12
    traffic = recorded_traffic()
    q = lambda xs, p: float(np.percentile(np.array(xs), p))  # noqa: E731

    v_streamed_bytes = (algorithmic_bytes_per_launch(cfg)
                        + (cfg.K - 1) * cfg.vocab * cfg.rank * 2)
    result = {
        "metric": METRIC, "value": round(value_us, 3), "unit": "us/step",
        "n_gpus": world, "steps": K_steps, "warmup": W,
        "ms_per_step": round(ms_per_iter, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy; shapes and distributions of the "
                "pages' workloads)",
        "config": {
            "workload": workload_desc(cfg),
            "timing": (("eager launches" if args.no_graph else
                        "one CUDA graph replayed per step") + "; " +
                       ("scheduler after the chain on one stream" if serial
                        else "scheduler on a second stream alongside the "
                        "chain, verify-token gather after the join") +
                       "; CUDA events around the timed steps; breakdown_us "
                       "from a separate pass with events between the parts"),
            "l2": l2_desc(cfg),
            "parallelism": f"replicas x{world}",
        },
        "breakdown_us": {
            "chain_median": round(chain_med, 3), "chain_p10": round(q(chain_us, 10), 3),
            "chain_p90": round(q(chain_us, 90), 3),
            "select_median": round(statistics.median(sel_us), 3),
            "select_p10": round(q(sel_us, 10), 3), "select_p90": round(q(sel_us, 90), 3),
            "step_median": round(statistics.median(step_us), 3),
            "host_clock_us_per_step": round(t_host * 1e6 / K_steps, 3),
        },
        "roofline": {
            "bound": "hbm", "kernel": "chain_kernel (one launch = all K positions)",
            "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved_gbs / hbm, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": algorithmic_bytes_per_launch(cfg),
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
            # V re-read at every position (the bound when no V line survives
            # in L2 between positions): context for frac, not the roofline
            "v_streamed_bytes_per_launch": v_streamed_bytes,
            "frac_v_streamed": round(v_streamed_bytes / (chain_med * 1e-6) / 1e9 / hbm, 4),
        },
        "roofline_tensor": {
            "bound": "tensor", "achieved": round(achieved_tf, 2),
            "peak": tf_burst, "unit": "TFLOP/s",
            "frac": round(achieved_tf / tf_burst, 4),
            "frac_of_sustained": round(achieved_tf / tf_sus, 4),
            "flops_per_launch": flops_per_launch(cfg),
        },
        # chain_kernel + select_kernel (+ gather_verify_kernel) per step
        "gpu_launches": K_steps * (2 if serial else 3),
        "clocks": clocks,
    }
    if rank == 0:
        result["e2e"] = run_e2e(st, cfg, stream, args.e2e_steps)
        if not args.no_extras:
            result["next_greedy_verify"] = run_greedy_verify(st, cfg, stream)
            result["next_stale_select"] = run_stale_select(st, cfg, stream)
            result["next_sample_chain"] = run_sample_chain(st, cfg, stream)
            result["next_lmhead_chain"] = run_lmhead_chain(st, cfg, stream)
            if cfg.name == "headline":
                result["workloads"] = run_other_workloads(dev)
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(cfg)
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_other_workloads(dev, names=("tiny", "gemma4_12b", "conc64", "dsv4"),
                        steps=100):
    """The same overlapped step (chain on one stream, scheduler alongside on
    another, verify-token gather after the join) on the other workloads of
    the test plan: the step as one CUDA graph per step with CUDA events
    around the loop, the chain and scheduler medians from a pass with events
    between the parts, and the chain's fractions of the HBM (V-once bytes)
    and bf16 tensor rooflines.  Stress (8 GB of logits)
    and DSV4-alt (the DSV4 chain) are left to ``--workload``."""
    import torch
    import workloads
    hbm, tf_burst, _, _ = measured_peaks()
    out = {}
    for name in names:
        cfg = workloads.get_config(name)
        st = Step(cfg, dev)
        main, side = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        with torch.cuda.stream(main):
            for _ in range(3):
                st.chain()
                st.select()
        main.synchronize()
        graphs = []
        for fn, sm in ((st.chain, main), (st.select_nodraft, side), (st.gather, main)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=sm):
                fn()
            graphs.append(g)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(steps + 5):
            e = ev[i - 5] if i >= 5 else [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(main)
            side.wait_event(e[0])
            with torch.cuda.stream(main):
                graphs[0].replay()
            e[1].record(main)
            with torch.cuda.stream(side):
                graphs[1].replay()
            e[2].record(side)
            main.wait_event(e[2])
            with torch.cuda.stream(main):
                graphs[2].replay()
            e[3].record(main)
        torch.cuda.synchronize()
        # the step itself: one multi-stream graph per step, events around
        # all of them
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=main):
            f0 = torch.cuda.Event()
            f0.record(main)
            side.wait_event(f0)
            st.chain()
            with torch.cuda.stream(side):
                st.select_nodraft()
            j0 = torch.cuda.Event()
            j0.record(side)
            main.wait_event(j0)
            st.gather()
        with torch.cuda.stream(main):
            for _ in range(5):
                g_step.replay()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(main)
            for _ in range(steps):
                g_step.replay()
            t1.record(main)
        torch.cuda.synchronize()
        assert st.D.dspark_read_status(st.cws) == 0 and st.D.dspark_read_status(st.sws) == 0
        med = lambda a, b: statistics.median(ev[i][a].elapsed_time(ev[i][b]) * 1e3  # noqa: E731
                                             for i in range(steps))
        step_us, chain_us, sel_us = t0.elapsed_time(t1) * 1e3 / steps, med(0, 1), med(0, 2)
        out[name] = {
            "workload": workload_desc(cfg), "step_us": round(step_us, 2),
            "chain_us": round(chain_us, 2), "select_us": round(sel_us, 2),
            "chain_frac_hbm": round(algorithmic_bytes_per_launch(cfg) / (chain_us * 1e-6) / 1e9 / hbm, 4),
            "chain_frac_tensor": round(flops_per_launch(cfg) / (chain_us * 1e-6) / 1e12 / tf_burst, 4),
            "steps": steps}
        del st, graphs, g_step
        torch.cuda.empty_cache()
    return out


def run_greedy_verify(st, cfg, stream, iters=100):
    """Downstream of the step (not part of the metric): greedy verification
    of this step's verify list against synthetic target logits (one row per
    verified draft token plus one bonus row per sampling request), timed
    with CUDA events; reports the streaming argmax's HBM roofline."""
    import numpy as np
    import torch
    import workloads
    D = st.D
    ln = st.ln.cpu().numpy()
    mask = st.sel["mask"]
    R = int(ln.sum() + mask.sum())
    rng = np.random.default_rng(cfg.seed + 77)
    x = rng.standard_normal((R, cfg.vocab), dtype=np.float32) * np.float32(2.0)
    tl = torch.from_numpy(workloads.f32_to_bf16_bits(x).view(np.int16)).to(
        st.logits.device).view(torch.bfloat16)
    del x
    N, K = cfg.N, cfg.K
    tgt = torch.zeros(N * (K + 1), dtype=torch.int32, device=tl.device)
    acc = torch.zeros(N, dtype=torch.int32, device=tl.device)
    bon = torch.zeros(N, dtype=torch.int32, device=tl.device)
    ws = D.new_workspace(256, tl.device)

    def one():
        D.dspark_greedy_verify(tl, st.draft, st.ln, st.cu, st.mask, tgt, acc,
                               bon, ws)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
    stream.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s.record(stream)
        for _ in range(iters):
            one()
        e.record(stream)
    stream.synchronize()
    us = s.elapsed_time(e) * 1e3 / iters
    hbm = measured_peaks()[0]
    nbytes = R * cfg.vocab * 2
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "rows": R, "bytes": nbytes,
            "achieved_GBs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
            "note": "dspark_greedy_verify (row argmax + acceptance), not part "
                    "of the step metric"}


def run_stale_select(st, cfg, stream, iters=200):
    """Scheduler variant (not part of the metric): B sized from a confidence
    buffer one step old, allocation by the current confidences, against the
    plain fused scheduler on the same inputs; single-CTA, latency-bound."""
    import torch
    import workloads
    D = st.D
    old = torch.from_numpy(workloads.make_stale_confidences(cfg, 1)).to(st.conf.device)

    def stale():
        D.dspark_select_step_stale(old, st.conf, st.mask, st.cost, st.T, 0.0,
                                   st.flags, st.draft, st.surv, st.srt, st.pre,
                                   st.ne, st.ns, st.B, st.obj, st.ln, st.cu,
                                   st.vi, st.vt, st.sws)

    out = {}
    for name, fn in (("stale_us", stale), ("plain_us", st.select)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s.record(stream)
            for _ in range(iters):
                fn()
            e.record(stream)
        stream.synchronize()
        out[name] = round(s.elapsed_time(e) * 1e3 / iters, 2)
    out["note"] = ("dspark_select_step_stale (two sorts in one CTA) vs "
                   "dspark_select_step; back-to-back calls, not part of the "
                   "step metric")
    return out


def run_sample_chain(st, cfg, stream, iters=50):
    """Probabilistic drafting (not part of the metric): dspark_chain_sample
    (a Gumbel-max draw over 16-entry blocks with Philox4x32-10 words, then
    the entry inside the block) against dspark_chain_draft on the same
    inputs, back-to-back launches timed with CUDA events."""
    import torch
    D = st.D

    def sample():
        D.dspark_chain_sample(st.logits, st.U, st.V, st.last, st.draft,
                              st.score, st.cws, seed=0x5EED, offset=1,
                              temperature=1.0)

    out = {}
    for name, fn in (("sample_us", sample), ("greedy_us", st.chain)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s.record(stream)
            for _ in range(iters):
                fn()
            e.record(stream)
        stream.synchronize()
        out[name] = round(s.elapsed_time(e) * 1e3 / iters, 2)
    elems = cfg.N * cfg.K * cfg.vocab
    out["elements"] = elems
    out["gelem_per_s"] = round(elems / (out["sample_us"] * 1e-6) / 1e9, 2)
    # Issue roofline: the work is the warp instructions one launch issues,
    # measured by ncu (smsp__inst_executed.sum, recorded with the kernel
    # source's hash), and the peak is four warp instructions per SM per clock
    # at the 2070 MHz maximum SM clock.  The launch also moves the greedy
    # chain's bytes (logits once, V once), reported against HBM beside it.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    peak = sms * 4 * 2.070e9 / 1e12
    inst = (_recorded(SAMPLE_PROFILE, "warp_instructions_per_launch")
            if cfg.name == "headline" else None)
    achieved = None if inst is None else inst / (out["sample_us"] * 1e-6) / 1e12
    out["roofline"] = {"bound": "issue", "achieved": None if achieved is None else round(achieved, 4),
                       "peak": round(peak, 4), "unit": "T warp instructions/s",
                       "frac": None if achieved is None else round(achieved / peak, 4),
                       "warp_instructions_per_launch": inst,
                       "thread_instructions_per_element":
                           None if inst is None else round(inst * 32 / elems, 2),
                       "peak_source": "derived: SMs x 4 issue slots x 2070 MHz",
                       "frac_hbm": round(algorithmic_bytes_per_launch(cfg)
                                         / (out["sample_us"] * 1e-6) / 1e9
                                         / measured_peaks()[0], 4)}
    out["note"] = ("dspark_chain_sample vs dspark_chain_draft, back-to-back "
                   "launches; not part of the step metric")
    return out


def run_lmhead_chain(st, cfg, stream, iters=20):
    """Fused output projection (not part of the metric): dspark_chain_lmhead
    on hidden states h [N, K, d] and a projection W [vocab, d] (d = 2048)
    instead of stored logits; CUDA events over back-to-back launches."""
    import numpy as np
    import torch
    import workloads
    D = st.D
    x = workloads.make_lmhead_inputs(cfg)
    dev = st.logits.device
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa: E731
    h, W = bf(x["h"]), bf(x["W"])
    del x

    def one():
        D.dspark_chain_lmhead(h, W, st.U, st.V, st.last, st.draft, st.score, st.cws)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
    stream.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s.record(stream)
        for _ in range(iters):
            one()
        e.record(stream)
    stream.synchronize()
    us = s.elapsed_time(e) * 1e3 / iters
    d = W.shape[1]
    flops = 2.0 * cfg.N * cfg.K * cfg.vocab * (d + cfg.rank)
    # W and V streamed once per position (neither fits in L2), h once
    hbm = cfg.K * cfg.vocab * (d + cfg.rank) * 2 + cfg.N * cfg.K * d * 2
    hbm_peak, tf_peak, _, src = measured_peaks()
    tf = flops / (us * 1e-6) / 1e12
    gbs = hbm / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "d": d, "flops_per_launch": flops,
            "hbm_bytes_per_launch": hbm,
            "roofline_tensor": {"achieved": round(tf, 1), "peak": tf_peak,
                                "unit": "TFLOP/s", "frac": round(tf / tf_peak, 4)},
            "roofline_hbm": {"achieved": round(gbs, 1), "peak": hbm_peak,
                             "unit": "GB/s", "frac": round(gbs / hbm_peak, 4)},
            "peak_source": src,
            "note": "dspark_chain_lmhead (h . W^T + U[prev] . V^T, logits never "
                    "stored), not part of the step metric"}


def run_e2e(st, cfg, stream, steps):
    """The same step through the public API with host buffers: per step the
    inputs are copied from pinned host memory and the scheduler's results
    are read back, all inside the timed region.  Two device buffer sets let
    the copy engine fill step i+1's inputs while the GPU computes step i
    (host-to-device on one copy stream, device-to-host on another)."""
    import numpy as np
    import torch
    D = st.D
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_logits = pin(st.logits_np.view(np.int16) if cfg.logits_dtype == "bf16" else st.logits_np)
    h_conf, h_mask = pin(st.sel["conf"]), pin(st.sel["mask"])
    h_last = pin(st.last_np)
    h_T = torch.tensor([st.sel["T"]], dtype=torch.int32).pin_memory()
    h_in = (h_logits, h_conf, h_mask, h_last, h_T)

    base = dict(logits=st.logits, conf=st.conf, mask=st.mask, last=st.last,
                T=st.T, draft=st.draft, score=st.score, surv=st.surv, srt=st.srt,
                pre=st.pre, ne=st.ne, ns=st.ns, B=st.B, obj=st.obj, ln=st.ln,
                cu=st.cu, vi=st.vi, vt=st.vt)

    def buffers(first):
        d = dict(base) if first else {k: torch.empty_like(v) for k, v in base.items()}
        d["in"] = (d["logits"].view(torch.int16) if cfg.logits_dtype == "bf16"
                   else d["logits"], d["conf"], d["mask"], d["last"], d["T"])
        d["outs"] = [d["B"], d["ln"], d["cu"], d["vi"], d["vt"], d["draft"]]
        d["h_outs"] = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in d["outs"]]
        return d

    sets = [buffers(True), buffers(False)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["h_outs"])
    cs, ds = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("h2d", "comp", "d2h")}
    started = [False, False]

    def one(i):
        j = i % 2
        b = sets[j]
        if started[j]:
            cs.wait_event(ev["comp"][j])   # step i-2 has finished reading set j
        with torch.cuda.stream(cs):
            for d_t, h_t in zip(b["in"], h_in):
                d_t.copy_(h_t, non_blocking=True)
            ev["h2d"][j].record(cs)
        stream.wait_event(ev["h2d"][j])
        if started[j]:
            stream.wait_event(ev["d2h"][j])  # step i-2's results are read back
        with torch.cuda.stream(stream):
            D.dspark_chain_draft(b["logits"], st.U, st.V, b["last"], b["draft"],
                                 b["score"], st.cws)
            D.dspark_select_step(b["conf"], b["mask"], st.cost, b["T"], 0.0,
                                 st.flags, b["draft"], b["surv"], b["srt"], b["pre"],
                                 b["ne"], b["ns"], b["B"], b["obj"], b["ln"],
                                 b["cu"], b["vi"], b["vt"], st.sws)
            ev["comp"][j].record(stream)
        ds.wait_event(ev["comp"][j])
        with torch.cuda.stream(ds):
            for d_t, h_t in zip(b["outs"], b["h_outs"]):
                h_t.copy_(d_t, non_blocking=True)
            ev["d2h"][j].record(ds)
        started[j] = True

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    cs.wait_event(s)  # the first copy starts after the start stamp
    for i in range(steps):
        one(i)
    for j in range(2):
        stream.wait_event(ev["d2h"][j])
    e.record(stream)
    torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / steps
    return {"value": round(us, 2), "unit": "us/step", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "path": "pinned host -> device copies (copy stream), dspark_chain_draft, "
                    "dspark_select_step, device -> pinned host copies (second copy "
                    "stream); two device buffer sets so step i+1's copy overlaps "
                    "step i's compute"}


# ------------------------------------------------------- CPU oracle leg
def _oracle_data(cfg):
    import workloads
    sel = workloads.make_select_inputs(cfg)
    fac = workloads.make_chain_factors(cfg)
    return dict(logits=workloads.make_logits_rows(cfg), U=fac["U"], V=fac["V"],
                last=workloads.make_last_token(cfg), conf=sel["conf"],
                mask=sel["mask"], cost=sel["cost"], T=sel["T"])


def _flags(cfg):
    import oracle
    return oracle.FORCE_RUNNING_MAX if cfg.cost_kind == "noisy" else 0


def cpu_baseline(cfg):
    """The oracle as it stands, on this host's cores, over one full step
    (all requests, all positions, then the scheduler)."""
    import oracle
    data = _oracle_data(cfg)
    t0 = time.perf_counter()
    ch = oracle.chain(data["logits"], cfg.logits_dtype, data["U"], data["V"],
                      data["last"])
    t1 = time.perf_counter()
    oracle.select_step(data["conf"], data["mask"], data["cost"], data["T"], 0.0,
                       _flags(cfg), ch["draft"])
    t2 = time.perf_counter()
    return {"value": round((t2 - t0) * 1e6, 1), "unit": "us/step",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"one full step of the {cfg.name} workload (all {cfg.N} "
                      f"requests x {cfg.K} positions, then the scheduler): "
                      f"chain {t1 - t0:.2f} s, scheduler {t2 - t1:.3f} s; "
                      f"numpy fp64, BLAS on all cores"}


def run_reference(args):
    """Reference arm: the CPU oracle, timed as it stands on this host.

    Every step, warm-up or timed, is one full oracle step of the workload:
    the chain over all requests and positions, then the scheduler (the same
    work as the GPU arm's step).  Each timed step is measured directly with
    the host clock and ``value`` is their mean.  If the requested steps would
    not fit in the time budget (a few minutes; about 4.4 s per step at the
    headline shape on 16 Grace cores), fewer steps are timed and ``steps``
    says how many."""
    import oracle
    import workloads
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = workloads.get_config(args.workload)
    data = _oracle_data(cfg)

    def one_step():
        t0 = time.perf_counter()
        ch = oracle.chain(data["logits"], cfg.logits_dtype, data["U"], data["V"],
                          data["last"])
        oracle.select_step(data["conf"], data["mask"], data["cost"], data["T"],
                           0.0, _flags(cfg), ch["draft"])
        return time.perf_counter() - t0

    budget_s = float(os.environ.get("DSPARK_REFERENCE_BUDGET_S", "900"))
    t_run0 = time.perf_counter()
    warm = [one_step() for _ in range(args.warmup)]
    per_step = min(warm) if warm else one_step()
    left = budget_s - (time.perf_counter() - t_run0)
    n_timed = int(max(1, min(args.steps, left // max(per_step, 1e-9))))
    t_timed0 = time.perf_counter()
    times = [one_step() for _ in range(n_timed)]
    timed_s = time.perf_counter() - t_timed0
    us = statistics.mean(times) * 1e6
    sample_txt = (f"every step (warm-up and timed) is one full oracle step of the "
                  f"{cfg.name} workload: the chain over all {cfg.N} requests x "
                  f"{cfg.K} positions, then the scheduler; {n_timed} steps timed "
                  f"one by one with the host clock ({timed_s:.1f} s in all)"
                  + ("" if n_timed == args.steps else
                     f", fewer than the {args.steps} requested to stay within "
                     f"{budget_s:.0f} s") + "; numpy fp64, BLAS on all cores")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1),
        "unit": "us/step", "n_gpus": world, "steps": n_timed,
        "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded numpy; shapes and "
                                "distributions of the pages' workloads)",
        "config": {"workload": workload_desc(cfg)},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/step",
                         "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample_txt},
        "e2e": {"value": round(us, 1), "unit": "us/step",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "timed_region_s": round(timed_s, 2),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------ host link (e2e bound)
_LINK_PROBE = r"""
// Host-to-device link probe: pinned copies on S streams, and SMs reading
// mapped pinned memory directly.  Times with CUDA events; returns -1 on error.
#include <cstdint>
#include <cuda_runtime.h>

__global__ void read_mapped(const uint4 *__restrict__ src, size_t n,
                            uint4 *__restrict__ sink) {
  const size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = t; i < n; i += stride) {
    const uint4 v = src[i];
    acc.x ^= v.x; acc.y ^= v.y; acc.z ^= v.z; acc.w ^= v.w;
  }
  sink[t] = acc;
}

static void *g_host = nullptr, *g_dev = nullptr, *g_sink = nullptr;

extern "C" int link_setup(size_t bytes) {
  if (cudaHostAlloc(&g_host, bytes, cudaHostAllocMapped) != cudaSuccess) return -1;
  if (cudaMalloc(&g_dev, bytes) != cudaSuccess) return -1;
  if (cudaMalloc(&g_sink, 1024 * 1024 * 16) != cudaSuccess) return -1;
  unsigned char *h = (unsigned char *)g_host;
  for (size_t i = 0; i < bytes; i += 4096) h[i] = (unsigned char)i;
  return 0;
}

extern "C" float link_copy_ms(size_t bytes, int streams) {
  cudaStream_t st[16];
  cudaEvent_t e0, e1, done[16];
  if (streams < 1 || streams > 16) return -1.0f;
  cudaEventCreate(&e0); cudaEventCreate(&e1);
  for (int s = 0; s < streams; ++s) {
    cudaStreamCreateWithFlags(&st[s], cudaStreamNonBlocking);
    cudaEventCreateWithFlags(&done[s], cudaEventDisableTiming);
  }
  cudaEventRecord(e0, st[0]);
  for (int s = 1; s < streams; ++s) cudaStreamWaitEvent(st[s], e0, 0);
  const size_t part = (bytes / streams) & ~(size_t)4095;
  for (int s = 0; s < streams; ++s) {
    const size_t off = part * s, n = s == streams - 1 ? bytes - off : part;
    cudaMemcpyAsync((char *)g_dev + off, (const char *)g_host + off, n,
                    cudaMemcpyHostToDevice, st[s]);
    cudaEventRecord(done[s], st[s]);
  }
  for (int s = 1; s < streams; ++s) cudaStreamWaitEvent(st[0], done[s], 0);
  cudaEventRecord(e1, st[0]);
  float ms = -1.0f;
  if (cudaEventSynchronize(e1) == cudaSuccess) cudaEventElapsedTime(&ms, e0, e1);
  for (int s = 0; s < streams; ++s) { cudaStreamDestroy(st[s]); cudaEventDestroy(done[s]); }
  cudaEventDestroy(e0); cudaEventDestroy(e1);
  return cudaGetLastError() == cudaSuccess ? ms : -1.0f;
}

extern "C" float link_mapped_ms(size_t bytes, int blocks) {
  void *dptr = nullptr;
  if (cudaHostGetDevicePointer(&dptr, g_host, 0) != cudaSuccess) return -1.0f;
  if (blocks < 1 || (size_t)blocks * 256 * 16 > 1024 * 1024 * 16) return -1.0f;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0, 0);
  read_mapped<<<blocks, 256>>>((const uint4 *)dptr, bytes / 16, (uint4 *)g_sink);
  cudaEventRecord(e1, 0);
  float ms = -1.0f;
  if (cudaEventSynchronize(e1) == cudaSuccess) cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0); cudaEventDestroy(e1);
  return cudaGetLastError() == cudaSuccess ? ms : -1.0f;
}
"""


_L2_PROBE = r"""
// The chain's L2 access pattern without its compute: every sweep (one draft
// position) re-reads a buffer R (the Markov factor V) split into one slice
// per pair of CTAs (the two request tiles of a vocabulary group, which run
// on one TPC), alternating direction, with a fractional evict_last policy,
// and streams a fresh chunk of a buffer S (the position's logits) once with
// evict_first.  DRAM bytes come from ncu; the kernel returns nothing useful.
#include <cstdint>
#include <cuda_runtime.h>

__device__ __forceinline__ uint4 ld_hint(const uint4 *p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__global__ void chain_pattern(const uint4 *__restrict__ R, size_t r_n,
                              const uint4 *__restrict__ S, size_t s_n,
                              int sweeps, float keep, uint4 *__restrict__ sink) {
  uint64_t pk, pf;
  asm volatile("createpolicy.fractional.L2::evict_last.L2::evict_first.b64 %0, %1;"
               : "=l"(pk) : "f"(keep));
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pf));
  const size_t groups = gridDim.x / 2, g = blockIdx.x / 2;
  const size_t lo = r_n * g / groups, hi = r_n * (g + 1) / groups;
  const size_t chunk = s_n / ((size_t)sweeps * gridDim.x);
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  const size_t nt = blockDim.x;
  for (int w = 0; w < sweeps; ++w) {
    // four independent loads in flight per thread and step
    for (size_t t0 = 0; t0 < hi - lo; t0 += 4 * nt) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const size_t t = t0 + u * nt + threadIdx.x;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (t < hi - lo) v[u] = ld_hint(R + ((w & 1) ? hi - 1 - t : lo + t), pk);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x ^= v[u].x; acc.y ^= v[u].y; acc.z ^= v[u].z; acc.w ^= v[u].w;
      }
    }
    const size_t c0 = ((size_t)w * gridDim.x + blockIdx.x) * chunk;
    for (size_t t0 = 0; t0 < chunk; t0 += 4 * nt) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const size_t t = t0 + u * nt + threadIdx.x;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (t < chunk) v[u] = ld_hint(S + c0 + t, pf);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x ^= v[u].x; acc.y ^= v[u].y; acc.z ^= v[u].z; acc.w ^= v[u].w;
      }
    }
  }
  sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

static uint4 *g_R = nullptr, *g_S = nullptr, *g_sink = nullptr;

extern "C" int l2_setup(size_t r_bytes, size_t s_bytes) {
  if (cudaMalloc(&g_R, r_bytes) != cudaSuccess) return -1;
  if (cudaMalloc(&g_S, s_bytes) != cudaSuccess) return -1;
  if (cudaMalloc(&g_sink, 4 << 20) != cudaSuccess) return -1;
  cudaMemset(g_R, 1, r_bytes);
  cudaMemset(g_S, 2, s_bytes);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}

extern "C" float l2_run_ms(size_t r_bytes, size_t s_bytes, int sweeps, float keep,
                           int blocks) {
  if (blocks < 2 || blocks * 512 * 16 > (4 << 20)) return -1.0f;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0, 0);
  chain_pattern<<<blocks, 512>>>(g_R, r_bytes / 16, g_S, s_bytes / 16, sweeps,
                                 keep, g_sink);
  cudaEventRecord(e1, 0);
  float ms = -1.0f;
  if (cudaEventSynchronize(e1) == cudaSuccess) cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0); cudaEventDestroy(e1);
  return cudaGetLastError() == cudaSuccess ? ms : -1.0f;
}
"""


def _build_probe(src_text, name):
    import ctypes
    import tempfile
    tmp = tempfile.mkdtemp(prefix="dspark_probe_")
    src, lib = os.path.join(tmp, name + ".cu"), os.path.join(tmp, name + ".so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
                           "-O3", "-shared", "-Xcompiler", "-fPIC", "-o", lib, src])
    return ctypes.CDLL(lib)


def run_l2(args):
    """The chain's L2 pattern alone (see _L2_PROBE), at the headline's sizes:
    a re-read buffer of 48 MB .. V (134.2 MB) kept with 0.4 .. 1.0 of its
    lines evict_last, and the K = 7 positions' logits (939.5 MB) streamed
    once.  One launch per line of the table, in the printed order; the DRAM
    bytes of each launch come from ncu (one pass: dram__bytes_read.sum)."""
    import ctypes
    import workloads
    cfg = workloads.get_config(args.workload)
    v_bytes = cfg.vocab * cfg.rank * 2
    s_bytes = cfg.N * cfg.K * cfg.vocab * 2
    L = _build_probe(_L2_PROBE, "l2")
    L.l2_setup.argtypes = [ctypes.c_size_t, ctypes.c_size_t]
    L.l2_run_ms.argtypes = [ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
                            ctypes.c_float, ctypes.c_int]
    L.l2_run_ms.restype = ctypes.c_float
    assert L.l2_setup(v_bytes, s_bytes) == 0
    blocks = 150
    L.l2_run_ms(v_bytes, s_bytes, cfg.K, 0.6, blocks)  # warm-up (not a table line)
    rows = []
    for mb in (48, 64, 80, 96, 112, v_bytes / 2**20):
        r = (int(mb * 2**20) // (16 * 150)) * 16 * 150
        for keep in (0.4, 0.6, 0.8, 1.0):
            assert L.l2_run_ms(r, s_bytes, cfg.K, keep, blocks) > 0
            rows.append({"reread_MB": round(r / 1e6, 1), "keep": keep,
                         "algorithmic_if_all_rereads_hit_MB":
                             round((r + s_bytes) / 1e6, 1),
                         "if_no_reread_hits_MB":
                             round((cfg.K * r + s_bytes) / 1e6, 1)})
    print(json.dumps({"probe": "chain L2 pattern", "workload": workload_desc(cfg),
                      "sweeps": cfg.K, "stream_MB": round(s_bytes / 1e6, 1),
                      "blocks": blocks, "launches_after_warmup": rows}), flush=True)


def run_link(args):
    """The host-to-device link alone, for the bytes one headline step copies
    (the logits, 939.5 MB): pinned copies split over 1/2/4/8 streams, and
    SMs reading the mapped pinned buffer themselves.  Best of 5 each."""
    import ctypes
    import workloads
    cfg = workloads.get_config(args.workload)
    nbytes = cfg.N * cfg.K * cfg.vocab * (2 if cfg.logits_dtype == "bf16" else 4)
    L = _build_probe(_LINK_PROBE, "link")
    L.link_setup.argtypes = [ctypes.c_size_t]
    L.link_copy_ms.argtypes = [ctypes.c_size_t, ctypes.c_int]
    L.link_copy_ms.restype = ctypes.c_float
    L.link_mapped_ms.argtypes = [ctypes.c_size_t, ctypes.c_int]
    L.link_mapped_ms.restype = ctypes.c_float
    assert L.link_setup(nbytes) == 0
    out = {"metric": "host-to-device bytes per second for one step's inputs",
           "bytes": nbytes, "workload": workload_desc(cfg), "copies": {},
           "mapped_read": {}}
    for streams in (1, 2, 4, 8):
        L.link_copy_ms(nbytes, streams)  # warm-up
        ms = min(L.link_copy_ms(nbytes, streams) for _ in range(5))
        assert ms > 0
        out["copies"][f"{streams}_streams"] = {"ms": round(ms, 3),
                                               "GB_s": round(nbytes / ms / 1e6, 1)}
    for blocks in (152, 304, 608, 1024):
        L.link_mapped_ms(nbytes, blocks)
        ms = min(L.link_mapped_ms(nbytes, blocks) for _ in range(5))
        assert ms > 0
        out["mapped_read"][f"{blocks}_blocks"] = {"ms": round(ms, 3),
                                                  "GB_s": round(nbytes / ms / 1e6, 1)}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.link:
        run_link(args)
        return
    if args.l2:
        run_l2(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
