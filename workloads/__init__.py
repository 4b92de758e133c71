"""Seeded synthetic inputs for the DSpark draft-and-schedule step.

This module is shared by the CPU oracle (``oracle/``), the tests and
``bench.py``.  It only draws random numbers and lays them out; it holds none
of the method's arithmetic (no bias, no argmax, no survival product, no budget
rule).  Every array is a plain numpy array in the layout the C ABI consumes:

* ``logits``  [N, K, vocab]  bf16 bit patterns (``uint16``) or ``float32``
* ``U``, ``V`` [vocab, rank] bf16 bit patterns (``uint16``), row-major
* ``last_token`` [N] int32, ``conf`` [N, K] float32, ``mask`` [N] uint8
* ``cost`` [L] float32 (microseconds), ``T`` int, ``draft_cost`` float

The workload shapes stand in for the pages' live traffic and datasets, which
are not reproduced here: vocabulary 262144 (a "524 KB row" of bf16 in
"DSpark on MAX", section *Correctness, then 1.3x*), K = 7 draft positions
(DeepSpec defaults, "How DSpark Speeds Up LLM Inference", appendix Part A),
per-position survival falling from >70% to <10% ("Adaptive Verification in
vLLM", *The problem*), batch up to 256 (same page, *Results*) and a cost table
that is a staircase inside the CUDA-graph capture region with a jump past it
(same page, *The cost model*).

Random streams: each component draws from its own child of
``numpy.random.SeedSequence(seed)``; the logits of request ``n`` come from
their own grand-child stream, so any subset of requests can be regenerated
without the others (the oracle uses this to check sampled rows of full-size
workloads).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Config", "CONFIGS", "get_config", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "make_select_inputs", "make_chain_factors", "make_logits_rows",
    "make_last_token", "make_workload", "w1_instance",
]

# child-stream indices of SeedSequence(seed).spawn(_N_STREAMS)
_S_LOGITS, _S_U, _S_V, _S_LAST, _S_CONF, _S_MASK, _S_COST, _S_TIES = range(8)
_N_STREAMS = 8


@dataclass(frozen=True)
class Config:
    """One synthetic workload (shapes, distributions, cost recipe, seed)."""
    name: str
    N: int
    K: int
    vocab: int
    rank: int
    logits_dtype: str            # "bf16" or "f32"
    logit_sd: float              # logits ~ N(0, logit_sd)
    uv_sd: float                 # U, V ~ N(0, uv_sd), rounded to bf16
    conf_kind: str               # "normal_mu" | "logitnormal" | "uniform"
    conf_a: float                # first-position mean (mu or m)
    conf_b: float                # last-position mean
    conf_request_offset_sd: float
    n_nonsampling: int
    prefill_tokens_each: int     # prompt-chunk tokens of each non-sampling request
    cost_kind: str               # "linear" | "stepped" | "noisy"
    cost_a: float                # base(n) = cost_a + cost_b * n
    cost_b: float
    cost_cap: int                # last CUDA-graph capture size (stepped tables)
    cost_jump: float             # multiplier past the capture region
    L: int
    seed: int
    tie_row_fraction: float = 0.0
    tie_pairs: int = 0
    draft_cost: float = 0.0
    notes: str = field(default="", compare=False)

    @property
    def n_sampling(self) -> int:
        return self.N - self.n_nonsampling

    @property
    def T(self) -> int:
        # one non-draft input token per decoding request plus every prompt
        # chunk token scheduled in the same step
        return self.n_sampling + self.n_nonsampling * self.prefill_tokens_each


CONFIGS = {
    "tiny": Config(
        "tiny", N=3, K=7, vocab=1024, rank=16, logits_dtype="f32",
        logit_sd=2.0, uv_sd=0.1, conf_kind="normal_mu", conf_a=1.5,
        conf_b=-2.5, conf_request_offset_sd=0.0, n_nonsampling=0,
        prefill_tokens_each=0, cost_kind="linear", cost_a=10.0, cost_b=0.5,
        cost_cap=0, cost_jump=1.0, L=64, seed=0,
        notes="3 requests, fp32 logits, U/V drawn in fp32 then rounded to bf16"),
    "gemma4_12b": Config(
        "gemma4_12b", N=8, K=7, vocab=262144, rank=256, logits_dtype="bf16",
        logit_sd=2.0, uv_sd=0.02, conf_kind="logitnormal", conf_a=0.7,
        conf_b=0.1, conf_request_offset_sd=0.0, n_nonsampling=0,
        prefill_tokens_each=0, cost_kind="stepped", cost_a=4000.0, cost_b=3.0,
        cost_cap=512, cost_jump=1.4, L=1024, seed=1),
    "conc64": Config(
        "conc64", N=64, K=7, vocab=262144, rank=256, logits_dtype="bf16",
        logit_sd=2.0, uv_sd=0.02, conf_kind="logitnormal", conf_a=0.7,
        conf_b=0.1, conf_request_offset_sd=1.0, n_nonsampling=4,
        prefill_tokens_each=512, cost_kind="stepped", cost_a=4000.0,
        cost_b=3.0, cost_cap=512, cost_jump=1.4, L=4096, seed=2),
    "dsv4": Config(
        "dsv4", N=256, K=7, vocab=129280, rank=256, logits_dtype="bf16",
        logit_sd=2.0, uv_sd=0.02, conf_kind="logitnormal", conf_a=0.7,
        conf_b=0.08, conf_request_offset_sd=0.0, n_nonsampling=16,
        prefill_tokens_each=128, cost_kind="stepped", cost_a=20000.0,
        cost_b=4.0, cost_cap=4096, cost_jump=1.4, L=8192, seed=3,
        notes="2048 prompt tokens in total over the 16 non-sampling requests"),
    "dsv4_alt": Config(
        "dsv4_alt", N=256, K=7, vocab=129280, rank=256, logits_dtype="bf16",
        logit_sd=2.0, uv_sd=0.02, conf_kind="logitnormal", conf_a=0.7,
        conf_b=0.08, conf_request_offset_sd=0.0, n_nonsampling=16,
        prefill_tokens_each=2048, cost_kind="stepped", cost_a=20000.0,
        cost_b=4.0, cost_cap=4096, cost_jump=1.4, L=40960, seed=3,
        notes="2048 prompt tokens for each non-sampling request"),
    "stress": Config(
        "stress", N=1024, K=15, vocab=262144, rank=256, logits_dtype="bf16",
        logit_sd=2.0, uv_sd=0.02, conf_kind="uniform", conf_a=0.0, conf_b=1.0,
        conf_request_offset_sd=0.0, n_nonsampling=102, prefill_tokens_each=32,
        cost_kind="noisy", cost_a=2000.0, cost_b=1.0, cost_cap=0,
        cost_jump=1.0, L=8192, seed=4, tie_row_fraction=0.05, tie_pairs=256,
        notes="cost noise must be forced monotone before use"),
    "headline": Config(
        "headline", N=256, K=7, vocab=262144, rank=256, logits_dtype="bf16",
        logit_sd=2.0, uv_sd=0.02, conf_kind="logitnormal", conf_a=0.7,
        conf_b=0.08, conf_request_offset_sd=0.0, n_nonsampling=16,
        prefill_tokens_each=128, cost_kind="stepped", cost_a=20000.0,
        cost_b=4.0, cost_cap=4096, cost_jump=1.4, L=8192, seed=5,
        notes="batch 256, K=7, vocab 262144, rank 256 with the DeepSeek-V4 "
              "confidence, mask and cost recipe"),
}


def get_config(name: str, **overrides) -> Config:
    cfg = CONFIGS[name]
    if overrides:
        d = {f: getattr(cfg, f) for f in cfg.__dataclass_fields__}
        d.update(overrides)
        cfg = Config(**d)
    return cfg


# --------------------------------------------------------------------------
# bf16 storage helpers (round-to-nearest-even); data-type plumbing only
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return bits."""
    x = np.asarray(x, dtype=np.float32)
    u = np.ascontiguousarray(x).view(np.uint32).reshape(x.shape)
    # finite inputs only: the rounding increment cannot wrap a 32-bit word
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _streams(seed: int):
    return np.random.SeedSequence(seed).spawn(_N_STREAMS)


# --------------------------------------------------------------------------
# scheduler inputs: confidences, sampling mask, cost table, T
# --------------------------------------------------------------------------
def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _logit(p):
    return np.log(p / (1.0 - p))


def make_cost_table(cfg: Config) -> np.ndarray:
    n = np.arange(cfg.L, dtype=np.float64)
    base = lambda m: cfg.cost_a + cfg.cost_b * m  # noqa: E731
    if cfg.cost_kind == "linear":
        c = base(n)
    elif cfg.cost_kind == "stepped":
        # inside the capture region a batch pays for the next captured size
        # (powers of two up to cost_cap); beyond it cost is continuous with a
        # jump of cost_jump
        c = np.empty(cfg.L, dtype=np.float64)
        for i in range(cfg.L):
            if i == 0:
                c[i] = base(1)
            elif i <= cfg.cost_cap:
                p2 = 1 << (i - 1).bit_length()
                c[i] = base(p2)
            else:
                c[i] = cfg.cost_jump * base(i)
    elif cfg.cost_kind == "noisy":
        rng = np.random.default_rng(_streams(cfg.seed)[_S_COST])
        c = base(n) * rng.uniform(0.95, 1.05, size=cfg.L)
    else:
        raise ValueError(cfg.cost_kind)
    return c.astype(np.float32)


def make_select_inputs(cfg: Config) -> dict:
    """Confidences [N,K] f32, sampling mask [N] u8, cost [L] f32, T, draft_cost."""
    st = _streams(cfg.seed)
    N, K = cfg.N, cfg.K
    rc = np.random.default_rng(st[_S_CONF])
    pos = np.arange(K, dtype=np.float64)
    frac = pos / max(K - 1, 1)
    if cfg.conf_kind == "normal_mu":
        mu = cfg.conf_a + (cfg.conf_b - cfg.conf_a) * frac
        z = rc.normal(0.0, 1.0, size=(N, K)) + mu[None, :]
        conf = _sigmoid(z)
    elif cfg.conf_kind == "logitnormal":
        m = cfg.conf_a + (cfg.conf_b - cfg.conf_a) * frac
        z = rc.normal(0.0, 1.0, size=(N, K)) + _logit(m)[None, :]
        if cfg.conf_request_offset_sd > 0:
            z = z + rc.normal(0.0, cfg.conf_request_offset_sd, size=(N, 1))
        conf = _sigmoid(z)
    elif cfg.conf_kind == "uniform":
        conf = rc.uniform(0.0, 1.0, size=(N, K))
    else:
        raise ValueError(cfg.conf_kind)
    mask = np.ones(N, dtype=np.uint8)
    if cfg.n_nonsampling:
        rm = np.random.default_rng(st[_S_MASK])
        mask[rm.choice(N, cfg.n_nonsampling, replace=False)] = 0
    return dict(conf=conf.astype(np.float32), mask=mask,
                cost=make_cost_table(cfg), T=cfg.T,
                draft_cost=np.float32(cfg.draft_cost))


def make_stale_confidences(cfg: Config, steps_back: int = 1) -> np.ndarray:
    """Confidences [N,K] f32 the head gave ``steps_back`` steps earlier: the
    same recipe as make_select_inputs, drawn from a seed of its own (the
    mask, cost table and T of the current step are unchanged)."""
    import dataclasses
    old = dataclasses.replace(cfg, seed=cfg.seed + 7919 * int(steps_back))
    return make_select_inputs(old)["conf"]


# --------------------------------------------------------------------------
# chain inputs: U, V (with planted duplicate rows), last token, logits rows
# --------------------------------------------------------------------------
def _tie_pairs(cfg: Config) -> np.ndarray:
    """[P, 2] vocabulary columns (c < c') whose V rows are made identical."""
    if not cfg.tie_pairs:
        return np.zeros((0, 2), dtype=np.int64)
    rng = np.random.default_rng(_streams(cfg.seed)[_S_TIES])
    cols = rng.choice(cfg.vocab, 2 * cfg.tie_pairs, replace=False)
    pairs = np.sort(cols.reshape(-1, 2), axis=1)
    return pairs


def _normal_bf16_blocked(ss: np.random.SeedSequence, rows: int, cols: int,
                         sd: float, block: int = 8192) -> np.ndarray:
    """N(0, sd) rounded to bf16, drawn in row blocks from spawned streams."""
    nblk = (rows + block - 1) // block
    kids = ss.spawn(nblk)
    out = np.empty((rows, cols), dtype=np.uint16)

    def work(b):
        r0, r1 = b * block, min(rows, (b + 1) * block)
        x = np.random.default_rng(kids[b]).standard_normal((r1 - r0, cols),
                                                             dtype=np.float32)
        out[r0:r1] = f32_to_bf16_bits(x * np.float32(sd))

    with ThreadPoolExecutor(min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(nblk)))
    return out


def make_chain_factors(cfg: Config) -> dict:
    """U, V as bf16 bits [vocab, rank]; V carries the planted duplicate rows."""
    st = _streams(cfg.seed)
    U = _normal_bf16_blocked(st[_S_U], cfg.vocab, cfg.rank, cfg.uv_sd)
    V = _normal_bf16_blocked(st[_S_V], cfg.vocab, cfg.rank, cfg.uv_sd)
    pairs = _tie_pairs(cfg)
    if len(pairs):
        V[pairs[:, 1]] = V[pairs[:, 0]]
    return dict(U=U, V=V, tie_pairs=pairs)


# width of the drafter's output projection for the fused LM-head workloads
# (a drafter of about a billion parameters; the pages give no width)
LMHEAD_D = 2048


def make_lmhead_inputs(cfg: Config, d: int = LMHEAD_D) -> dict:
    """Hidden states h [N, K, d] ~ N(0, 1) and output projection W [vocab, d]
    ~ N(0, logit_sd / sqrt(d)), both bf16 bits, so that h . W^T has the
    workload's logit spread; drawn from a seed sequence of their own."""
    kids = np.random.SeedSequence([cfg.seed, 0x4C4D]).spawn(2)
    h = _normal_bf16_blocked(kids[0], cfg.N * cfg.K, d, 1.0).reshape(cfg.N, cfg.K, d)
    W = _normal_bf16_blocked(kids[1], cfg.vocab, d, cfg.logit_sd / np.sqrt(d))
    return dict(h=h, W=W, d=d)


def make_last_token(cfg: Config) -> np.ndarray:
    rng = np.random.default_rng(_streams(cfg.seed)[_S_LAST])
    return rng.integers(0, cfg.vocab, size=cfg.N, dtype=np.int64).astype(np.int32)


def _logits_one_request(cfg: Config, ss: np.random.SeedSequence,
                        pairs: np.ndarray):
    rng = np.random.default_rng(ss)
    x = rng.standard_normal((cfg.K, cfg.vocab), dtype=np.float32)
    x *= np.float32(cfg.logit_sd)
    if cfg.logits_dtype == "bf16":
        row = f32_to_bf16_bits(x)
        if cfg.tie_row_fraction > 0 and len(pairs):
            # plant exact ties at the row maximum on a duplicated V pair: the
            # Markov bias of the two columns is then identical, so the adjusted
            # values tie exactly whatever the previous token is
            hit = rng.uniform(size=cfg.K) < cfg.tie_row_fraction
            which = rng.integers(0, len(pairs), size=cfg.K)
            for k in np.nonzero(hit)[0]:
                vals = bf16_bits_to_f32(row[k])
                top = f32_to_bf16_bits(np.float32(vals.max() + 0.5)).item()
                c0, c1 = pairs[which[k]]
                row[k, c0] = top
                row[k, c1] = top
        return row
    return x


def make_logits_rows(cfg: Config, rows=None, threads: int | None = None) -> np.ndarray:
    """Logits of the requests in ``rows`` (default: all), shape [len(rows), K, vocab]."""
    rows = np.arange(cfg.N) if rows is None else np.asarray(rows)
    per_req = _streams(cfg.seed)[_S_LOGITS].spawn(cfg.N)
    pairs = _tie_pairs(cfg)
    dt = np.uint16 if cfg.logits_dtype == "bf16" else np.float32
    out = np.empty((len(rows), cfg.K, cfg.vocab), dtype=dt)
    if threads is None:
        threads = min(32, os.cpu_count() or 1)

    def work(i):
        out[i] = _logits_one_request(cfg, per_req[int(rows[i])], pairs)

    if threads > 1 and len(rows) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(len(rows))))
    else:
        for i in range(len(rows)):
            work(i)
    return out


def planted_ties(cfg: Config, logits_rows: np.ndarray, rows=None):
    """(n, k, c, c') for every row whose maximum sits on a duplicated V pair."""
    rows = np.arange(cfg.N) if rows is None else np.asarray(rows)
    pairs = _tie_pairs(cfg)
    found = []
    if cfg.logits_dtype != "bf16" or not len(pairs):
        return found
    for i, n in enumerate(rows):
        for k in range(cfg.K):
            vals = bf16_bits_to_f32(logits_rows[i, k])
            top = vals.max()
            for c0, c1 in pairs:
                if vals[c0] == top and vals[c1] == top:
                    found.append((int(n), k, int(c0), int(c1)))
    return found


def make_workload(name: str, with_logits: bool = True, **overrides) -> dict:
    cfg = get_config(name, **overrides)
    d = dict(cfg=cfg)
    d.update(make_select_inputs(cfg))
    d.update(make_chain_factors(cfg))
    d["last_token"] = make_last_token(cfg)
    if with_logits:
        d["logits"] = make_logits_rows(cfg)
    return d


# --------------------------------------------------------------------------
# the hand-built 3-request x 7-slot instance of the vLLM blog's Figure 1
# --------------------------------------------------------------------------
def w1_instance() -> dict:
    """Three sampling requests, K = 7, T = 3, cost[n] = 10 + 0.5 n us, L = 64.

    The page prints only the caption of its Figure 1 (verify the best B = 11
    of 21 slots); these confidences are constructed so that 11 is the unique
    outcome (survivals are powers of 0.95 until a 0.1 factor).
    """
    hi, lo = 0.95, 0.1
    conf = np.array([
        [hi, hi, hi, hi, hi, lo, lo],
        [hi, hi, hi, hi, lo, lo, lo],
        [hi, hi, lo, lo, lo, lo, lo],
    ], dtype=np.float32)
    return dict(conf=conf, mask=np.ones(3, dtype=np.uint8),
                cost=(10.0 + 0.5 * np.arange(64)).astype(np.float32), T=3,
                draft_cost=np.float32(0.0))
