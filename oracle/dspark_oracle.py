"""Plain CPU oracle of the DSpark draft-and-schedule step (fp64, numpy).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never does, and
this module shares no code, table or helper with it.

What it computes, step by step, with the passage each step follows:

* Chaining ("DSpark on MAX", *What DSpark is*, item 3; "How DSpark Speeds Up
  LLM Inference", *Draft better*): for every draft position k the backbone
  logits are adjusted by a rank-r bias keyed on the previously chosen token,
  bias[v] = U[prev] . V[v], and the token is the argmax of the adjusted row.
  prev is the request's last committed token for k = 0, else the token just
  chosen at k - 1.
* Probabilistic drafting ("Adaptive Verification in vLLM", *Appendix:
  reproducing*, draft_sample_method "probabilistic"): each token is a draw
  from softmax(adj / tau), taken as a two-level Gumbel-max over blocks of 16
  vocabulary entries (sample_position).
* Survival ("Adaptive Verification in vLLM", *Scheduling the budget*): the
  running product of the confidences along each request.
* Global top-B (same section): slots of all sampling requests compete on
  survival; because survival only falls with position the best B slots form
  a contiguous prefix of every request.
* Budget (same section, the paragraph after the formula): B maximises
  (N_sampling + sum of the best B survivals) / cost[T + B], an argmax over a
  cumulative sum; T counts the step's non-draft tokens.
* Cost table (same page, *The cost model*): profiled step costs in
  microseconds, forced monotone; a drafter cost may be added.
* Allocation and compaction (same page, *Scheduling the budget*; "How DSpark
  Speeds Up LLM Inference", appendix Part B): each request gets its selected
  prefix; the verify list is flattened across requests with per-request
  offsets.
* Stale sizing (same page, *Scheduling the budget*, last paragraph: B is
  sized from a double-buffered confidence array one step old while the
  allocation uses current confidences; "How DSpark Speeds Up LLM Inference",
  appendix Part B: capacity from confidences two steps earlier): the budget
  steps run on the older buffer, the order and allocation on the current one.
* Fused LM head ("DSpark on MAX", *What DSpark is*, items 2-3: the block
  drafter emits scores for all K positions in one pass, then the chain adds
  the low-rank bias): the backbone logits are h[n, k] . W^T for hidden
  states h and the drafter's output projection W, computed here in fp64 and
  fed to the same chain.
* Greedy verification ("DSpark on MAX", *The kernel pass*, item 2): a draft
  token is accepted iff it equals the target's best token; the longest
  accepted run is kept and the target's next token is added.

Readings of points the pages leave open: exact cumulative sums (rounded
once), first-index argmax with NaN ranked highest, slot ties broken by slot
id, running-max forcing, b <= L-1-T, confidences clamped into [0, 1]; for
stale sizing the older buffer is aligned slot by slot with the current batch
and the current sampling mask and T apply to both passes.

Every function is pinned by ``tests/test_oracle_*.py`` against values and
properties the pages and the mathematics fix (a worked instance, brute force
over every slot subset, closed forms, exact integer arithmetic).
"""
from __future__ import annotations

import numpy as np

# device-status bits, mirrored from the C header's documented values so the
# tests can compare flags; the numbers are part of the public contract
TOKEN_OOR = 1
NAN_LOGIT = 2
CONF_OOR = 4
TABLE_SHORT = 8
COST_NONPOS = 16

FORCE_RUNNING_MAX = 1
FORCE_SUFFIX_MIN = 2
BUDGET_GREEDY_STOP = 4


# ---------------------------------------------------------------------------
# inputs to fp64
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (the upper half of an IEEE binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_to_f64(x) if dtype == "bf16" else np.asarray(x, np.float64)


# ---------------------------------------------------------------------------
# counter-based random numbers for probabilistic drafting
# ---------------------------------------------------------------------------
# Philox4x32-10 as defined by Salmon, Moraes, Dror and Shaw, "Parallel random
# numbers: as easy as 1, 2, 3" (SC 2011): a 4 x 32-bit counter and a 2 x 32-bit
# key; each of 10 rounds multiplies counter words 0 and 2 by the two round
# multipliers, mixes the high halves with the other words and the key, and
# bumps the key by the two Weyl constants.
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_M32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Four 32-bit output words (uint64 arrays) for counters (c0..c3) and key
    (k0, k1); inputs broadcast."""
    c = [np.asarray(x, dtype=np.uint64) & _M32 for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & _M32
    k1 = np.asarray(k1, dtype=np.uint64) & _M32
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    for _ in range(10):
        p0 = c[0] * m0  # < 2^64: exact in uint64
        p1 = c[2] * m1
        c = [(p1 >> np.uint64(32)) ^ c[1] ^ k0, p1 & _M32,
             (p0 >> np.uint64(32)) ^ c[3] ^ k1, p0 & _M32]
        k0 = (k0 + np.uint64(PHILOX_W0)) & _M32
        k1 = (k1 + np.uint64(PHILOX_W1)) & _M32
    return c


# ---------------------------------------------------------------------------
# probabilistic drafting: a two-level Gumbel-max draw
# ---------------------------------------------------------------------------
# Each draft token is a draw from softmax(adj / tau) ("Adaptive Verification
# in vLLM", *Appendix: reproducing*: draft_sample_method "probabilistic"),
# taken in two steps over blocks of SAMPLE_BLOCK consecutive vocabulary
# entries: the block by the Gumbel-max rule on the blocks' log partition
# functions, then the entry inside the block by inverting its cumulative
# distribution.  Block j is chosen with probability Z_j / sum Z and entry v of
# it with probability exp(s_v) / Z_j, so every entry has exactly its softmax
# probability exp(s_v) / sum Z.
SAMPLE_BLOCK = 16


def word_uniform(x) -> np.ndarray:
    """u = (2 * (x >> 9) + 1) / 2^24 from a 32-bit word: the top 23 bits, an
    odd multiple of 2^-24 in (0, 1) that fp32 and fp64 both hold exactly."""
    x = np.asarray(x, dtype=np.uint64)
    return (2.0 * (x >> np.uint64(9)).astype(np.float64) + 1.0) * 2.0 ** -24


def block_words(seed: int, offset: int, n: int, k: int, n_blocks: int):
    """The two words of every block j of request n, draft position k:
    Philox4x32-10 with counter (j // 2, n, k, offset) and key (low, high 32
    bits of seed); an even block takes words 0 and 1, an odd one words 2 and
    3.  Returns (x_gumbel, x_choice), uint64 arrays of n_blocks."""
    ctr = np.arange((n_blocks + 1) // 2, dtype=np.uint64)
    w = philox4x32_10(ctr, n, k, offset, seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    xg = np.stack([w[0], w[2]], axis=1).reshape(-1)[:n_blocks]
    xc = np.stack([w[1], w[3]], axis=1).reshape(-1)[:n_blocks]
    return xg, xc


def _block_view(s: np.ndarray) -> np.ndarray:
    """s [rows, vocab] as [rows, n_blocks, SAMPLE_BLOCK], -inf past vocab."""
    rows, vocab = s.shape
    nb = -(-vocab // SAMPLE_BLOCK)
    pad = np.full((rows, nb * SAMPLE_BLOCK), -np.inf)
    pad[:, :vocab] = s
    return pad.reshape(rows, nb, SAMPLE_BLOCK)


def _block_log_partition(b: np.ndarray) -> np.ndarray:
    """log sum exp over the last axis: NaN if any entry is NaN, -inf if every
    entry is -inf (max-shifted, fp64)."""
    m = np.max(b, axis=-1)                    # NaN propagates
    finite = np.isfinite(m)
    mm = np.where(finite, m, 0.0)
    with np.errstate(invalid="ignore"):
        z = np.sum(np.exp(b - mm[..., None]), axis=-1)
    return np.where(finite, mm + np.log(np.where(finite, z, 1.0)), m)


def _within_block(b: np.ndarray, u: float) -> int:
    """The entry of one block drawn with u in (0, 1): the first NaN entry if
    there is one, else the first +inf entry if there is one (it holds all
    the weight), the first entry if all are -inf, else the first e with
    sum_{i <= e} exp(b_i - max) > u * sum_i exp(b_i - max)."""
    if np.isnan(b).any():
        return int(np.argmax(np.isnan(b)))
    m = np.max(b)
    if m == np.inf:
        return int(np.argmax(b == np.inf))
    if m == -np.inf:
        return 0
    c = np.cumsum(np.exp(b - m))
    return int(np.argmax(c > u * c[-1]))


def sample_position(adj: np.ndarray, tau: float, seed: int, offset: int,
                    ns, k: int) -> dict:
    """Draws one token per row of adj [rows, vocab] (fp64) from
    softmax(adj / tau); row i uses the random words of request ns[i] and
    draft position k.  Returns the tokens, the score (the winning block's key
    log Z_j + g_j), the top-2 margin and |max| of the block keys, and per row
    the block keys, the winning block's cumulative weights and the choice
    target u * total (for the parity tests' tolerance)."""
    s = np.asarray(adj, dtype=np.float64) / tau
    b = _block_view(s)
    rows, nb, _ = b.shape
    keys = np.empty((rows, nb))
    uc = np.empty((rows, nb))
    for i, n in enumerate(ns):
        xg, xc = block_words(seed, offset, int(n), k, nb)
        keys[i] = _block_log_partition(b[i]) - np.log(-np.log(word_uniform(xg)))
        uc[i] = word_uniform(xc)
    jstar = np.argmax(keys, axis=1)           # first NaN, else first maximum
    r = np.arange(rows)
    best = keys[r, jstar]
    tok = np.array([jstar[i] * SAMPLE_BLOCK + _within_block(b[i, jstar[i]], uc[i, jstar[i]])
                    for i in range(rows)], dtype=np.int64)
    if nb > 1:
        part = np.partition(keys, nb - 2, axis=1)[:, -2:]
        with np.errstate(invalid="ignore"):
            margin = np.where(np.isnan(best), np.nan, part[:, 1] - part[:, 0])
    else:
        margin = np.full(rows, np.inf)
    cum, target = [], []
    for i in range(rows):
        bb = b[i, jstar[i]]
        m = np.max(bb)
        c = np.cumsum(np.exp(bb - m)) if np.isfinite(m) else np.zeros(SAMPLE_BLOCK)
        cum.append(c)
        target.append(uc[i, jstar[i]] * c[-1])
    return dict(tok=tok, score=best, margin=margin, absmax=np.abs(best), keys=keys,
                block=jstar, cum=np.array(cum), target=np.array(target))


# ---------------------------------------------------------------------------
# chaining
# ---------------------------------------------------------------------------
def markov_bias(U64: np.ndarray, V64: np.ndarray, prev: np.ndarray) -> np.ndarray:
    """bias[n, v] = sum_j U[prev_n, j] * V[v, j]  (rank-r factorised head)."""
    return U64[prev] @ V64.T


def chain_position(logits_k64: np.ndarray, U64: np.ndarray, V64: np.ndarray,
                   prev: np.ndarray) -> dict:
    """One draft position: adjusted logits and their first-index argmax.

    numpy's argmax returns the first maximal index and the first NaN if a row
    holds one, which is the tie and NaN rule of the C ABI.
    """
    adj = logits_k64 + markov_bias(U64, V64, prev)
    tok = np.argmax(adj, axis=1)
    rows = np.arange(adj.shape[0])
    best = adj[rows, tok]
    # top-2 margin (for the near-tie tolerance of the parity tests)
    if adj.shape[1] > 1:
        part = np.partition(adj, adj.shape[1] - 2, axis=1)[:, -2:]
        second = np.where(np.isnan(best), np.nan, part[:, 0])
        top = np.where(np.isnan(best), np.nan, part[:, 1])
        with np.errstate(invalid="ignore"):
            margin = top - second
    else:
        margin = np.full(adj.shape[0], np.inf)
    return dict(tok=tok.astype(np.int64), score=best, margin=margin,
                absmax=np.abs(best), adj=adj)


def chain(logits: np.ndarray, logits_dtype: str, U: np.ndarray, V: np.ndarray,
          last_token: np.ndarray, keep_adj: bool = False,
          sample: dict | None = None, rows: np.ndarray | None = None) -> dict:
    """Chain K draft positions for every row of ``logits`` [n, K, vocab].

    U, V are bf16 bit patterns [vocab, rank].  Returns draft [n, K] (int64),
    the adjusted value at the chosen token, the top-2 margin and |max| per
    (row, position), and the status bits a device would raise.

    ``sample`` = dict(seed, offset, tau) draws every token from the softmax
    of the adjusted logits at temperature tau instead of taking the argmax
    (probabilistic drafting: "Adaptive Verification in vLLM", *Appendix:
    reproducing*, draft_sample_method "probabilistic"), by sample_position;
    ``rows`` gives each row's request index n for the random words (default
    0..n-1).  Scores, margins and |max| then refer to the block keys.
    """
    U64 = bf16_to_f64(U)
    V64 = bf16_to_f64(V)
    n, K, vocab = logits.shape
    status = 0
    prev = np.asarray(last_token, dtype=np.int64).copy()
    bad = (prev < 0) | (prev >= vocab)
    if bad.any():
        status |= TOKEN_OOR
        prev[bad] = 0
    draft = np.zeros((n, K), dtype=np.int64)
    score = np.zeros((n, K))
    margin = np.zeros((n, K))
    absmax = np.zeros((n, K))
    adjs = []
    rows = np.arange(n) if rows is None else np.asarray(rows)
    for k in range(K):
        r = chain_position(to_f64(logits[:, k, :], logits_dtype), U64, V64, prev)
        if sample is not None:
            adj = r["adj"]
            r = sample_position(adj, float(sample["tau"]), int(sample["seed"]),
                                int(sample["offset"]), rows, k)
            r["adj"] = adj
        draft[:, k] = r["tok"]
        score[:, k] = r["score"]
        margin[:, k] = r["margin"]
        absmax[:, k] = r["absmax"]
        if np.isnan(r["score"]).any():
            status |= NAN_LOGIT
        if keep_adj:
            adjs.append(r["adj"])
        prev = r["tok"]
    out = dict(draft=draft, score=score, margin=margin, absmax=absmax,
               status=status)
    if keep_adj:
        out["adj"] = adjs
    return out


# ---------------------------------------------------------------------------
# confidence-scheduled verification
# ---------------------------------------------------------------------------
def clamp_confidence(conf: np.ndarray):
    """Confidences as fp64 in [0, 1]; NaN -> 0.  Returns (values, status)."""
    c = np.asarray(conf, dtype=np.float64).copy()
    status = 0
    bad = np.isnan(c) | (c < 0.0) | (c > 1.0)
    if bad.any():
        status |= CONF_OOR
    c[np.isnan(c)] = 0.0
    c = np.minimum(np.maximum(c, 0.0), 1.0)
    return c, status


def survival(conf: np.ndarray, mask: np.ndarray):
    """s[n, k] = prod_{j <= k} c[n, j], left to right; 0 for non-sampling rows."""
    c, status = clamp_confidence(conf)
    s = np.cumprod(c, axis=1)
    s[np.asarray(mask) == 0, :] = 0.0
    return s, status


def order_slots(s: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Eligible slots (rows of sampling requests) by survival desc, slot id asc."""
    N, K = s.shape
    slot = np.arange(N * K).reshape(N, K)
    elig = np.repeat(np.asarray(mask) != 0, K).reshape(N, K)
    ids = slot[elig]
    vals = s[elig]
    order = np.lexsort((ids, -vals))
    return ids[order].astype(np.int64)


def exact_prefix_sums(x: np.ndarray) -> np.ndarray:
    """P_b = x_0 + ... + x_{b-1} for b = 0..len(x), each the exact sum rounded
    once to the nearest double (ties to even).

    Every double is an integer multiple of 2**-1074, so the running sum is
    kept as a Python integer in those units and converted back with integer
    true division, which Python rounds correctly.  The result does not depend
    on the order of the additions.
    """
    out = np.empty(len(x) + 1, dtype=np.float64)
    out[0] = 0.0
    acc = 0
    scale = 1 << 1074
    for i, v in enumerate(np.asarray(x, dtype=np.float64).tolist()):
        num, den = float(v).as_integer_ratio()
        acc += num * (scale // den)
        out[i + 1] = acc / scale
    return out


def force_monotone(cost: np.ndarray, mode: int = FORCE_RUNNING_MAX) -> np.ndarray:
    """Cost table forced monotone non-decreasing.

    FORCE_RUNNING_MAX: cost'[n] = max_{m <= n} cost[m].
    FORCE_SUFFIX_MIN:  cost'[n] = min_{m >= n} cost[m] (a bigger, cheaper
    graph bounds the cost of a smaller batch).  NaN propagates in both.
    """
    c = np.asarray(cost, dtype=np.float32)
    if mode == FORCE_RUNNING_MAX:
        return np.maximum.accumulate(c)
    if mode == FORCE_SUFFIX_MIN:
        return np.minimum.accumulate(c[::-1])[::-1].copy()
    return c.copy()


def budget(sorted_s: np.ndarray, n_sampling: int, cost: np.ndarray, T: int,
           draft_cost: float = 0.0, greedy_stop: bool = False) -> dict:
    """Verify budget B from the sorted survivals and a (forced) cost table.

    f(b) = (N_sampling + P_b) / (cost[T + b] + draft_cost) for
    b = 0..b_max, b_max = min(S, L - 1 - T); B = first argmax (NaN ranks
    highest).  With greedy_stop, slots are admitted one at a time while f
    strictly rises.  T outside [0, L) gives B = 0 and TABLE_SHORT.
    """
    cost = np.asarray(cost, dtype=np.float32)
    L = len(cost)
    S = len(sorted_s)
    status = 0
    if T < 0 or T >= L:
        return dict(B=0, objective=0.0, b_max=0, P=np.zeros(1),
                    f=np.zeros(1), status=TABLE_SHORT)
    b_max = min(S, L - 1 - T)
    P = exact_prefix_sums(np.asarray(sorted_s[:b_max], dtype=np.float64))
    num = np.float64(n_sampling) + P
    den = cost[T:T + b_max + 1].astype(np.float64) + np.float64(np.float32(draft_cost))
    if not np.all(den > 0):
        status |= COST_NONPOS
    with np.errstate(divide="ignore", invalid="ignore"):
        f = num / den
    if greedy_stop:
        B = 0
        while B < b_max and f[B + 1] > f[B]:
            B += 1
    else:
        B = int(np.argmax(f))
    return dict(B=int(B), objective=float(f[B]), b_max=int(b_max), P=P, f=f,
                status=status)


def allocate(order: np.ndarray, B: int, N: int, K: int) -> np.ndarray:
    """len[n] = number of request n's slots among the first B of the order."""
    sel = np.asarray(order[:B], dtype=np.int64)
    return np.bincount(sel // K, minlength=N).astype(np.int64)


def compact(draft_len: np.ndarray, K: int, draft: np.ndarray | None = None) -> dict:
    """Request-major flattened verify list: offsets, slot ids, draft tokens."""
    draft_len = np.asarray(draft_len, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(draft_len)]).astype(np.int64)
    parts = [n * K + np.arange(draft_len[n]) for n in range(len(draft_len))]
    idx = np.concatenate(parts).astype(np.int64) if parts else np.zeros(0, np.int64)
    tok = None if draft is None else np.asarray(draft).reshape(-1)[idx]
    return dict(cu_len=cu, verify_idx=idx, verify_tok=tok)


# ---------------------------------------------------------------------------
# greedy verification of the compacted list
# ---------------------------------------------------------------------------
def verify_rows(draft_len: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """First target row of every request: each sampling request has
    draft_len[n] + 1 target rows (one per verified draft token plus the
    bonus position), request-major; non-sampling requests have none."""
    per = np.where(np.asarray(mask) != 0, np.asarray(draft_len) + 1, 0)
    return np.concatenate([[0], np.cumsum(per)]).astype(np.int64)


def greedy_verify(target_logits: np.ndarray, logits_dtype: str,
                  draft: np.ndarray, draft_len: np.ndarray,
                  mask: np.ndarray) -> dict:
    """Compare-only acceptance ("DSpark on MAX", *The kernel pass*, item 2:
    under greedy sampling a draft token is accepted iff it equals the
    target's best token; "How DSpark Speeds Up LLM Inference", *Context*:
    keep the longest matching run plus the target's next token).

    target_logits: [R, vocab], R = sum over sampling requests of len + 1.
    Returns the per-row target argmax (first index, NaN first), the accepted
    length and the bonus token per request (-1 for non-sampling requests).
    """
    N, K = np.asarray(draft).shape
    rows = verify_rows(draft_len, mask)
    R = int(rows[-1])
    tl = to_f64(target_logits[:R], logits_dtype)
    tgt = np.argmax(tl, axis=1).astype(np.int64) if R else np.zeros(0, np.int64)
    acc = np.full(N, -1, np.int64)
    bonus = np.full(N, -1, np.int64)
    for n in range(N):
        if mask[n] == 0:
            continue
        r0, ln = int(rows[n]), int(draft_len[n])
        a = 0
        while a < ln and draft[n, a] == tgt[r0 + a]:
            a += 1
        acc[n] = a
        bonus[n] = tgt[r0 + a]
    return dict(target_argmax=tgt, accepted=acc, bonus=bonus, rows=rows)


def select_step(conf, mask, cost, T, draft_cost=0.0, flags=0, draft=None) -> dict:
    """Survival -> order -> budget -> allocation -> compaction in one call."""
    conf = np.asarray(conf)
    N, K = conf.shape
    mask = np.ones(N, np.uint8) if mask is None else np.asarray(mask)
    s, st = survival(conf, mask)
    order = order_slots(s, mask)
    mode = (FORCE_RUNNING_MAX if flags & FORCE_RUNNING_MAX else
            FORCE_SUFFIX_MIN if flags & FORCE_SUFFIX_MIN else 0)
    cost_used = force_monotone(cost, mode)
    n_s = int((mask != 0).sum())
    bud = budget(s.reshape(-1)[order], n_s, cost_used, int(T), draft_cost,
                 greedy_stop=bool(flags & BUDGET_GREEDY_STOP))
    ln = allocate(order, bud["B"], N, K)
    cp = compact(ln, K, draft)
    return dict(survival=s, order=order, n_sampling=n_s, n_eligible=len(order),
                prefix=exact_prefix_sums(s.reshape(-1)[order]),
                B=bud["B"], objective=bud["objective"], b_max=bud["b_max"],
                f=bud["f"], draft_len=ln, cu_len=cp["cu_len"],
                verify_idx=cp["verify_idx"], verify_tok=cp["verify_tok"],
                cost_used=cost_used, status=st | bud["status"])


def select_step_stale(conf_size, conf, mask, cost, T, draft_cost=0.0, flags=0,
                      draft=None) -> dict:
    """Stale sizing ("Adaptive Verification in vLLM", *Scheduling the budget*,
    last paragraph; "How DSpark Speeds Up LLM Inference", appendix Part B).

    B (and the prefix sums and objective behind it) comes from ``conf_size``,
    an older confidence buffer aligned slot by slot with the current batch;
    the survival, the order and the allocation of those B slots come from the
    current ``conf``.  The current mask and T serve both passes, so both have
    the same number of eligible slots and B never exceeds it.
    """
    sized = select_step(conf_size, mask, cost, T, draft_cost, flags)
    conf = np.asarray(conf)
    N, K = conf.shape
    mask = np.ones(N, np.uint8) if mask is None else np.asarray(mask)
    s, st = survival(conf, mask)
    order = order_slots(s, mask)
    B = min(sized["B"], len(order))
    ln = allocate(order, B, N, K)
    cp = compact(ln, K, draft)
    return dict(survival=s, order=order, n_sampling=sized["n_sampling"],
                n_eligible=len(order), prefix=sized["prefix"], B=B,
                objective=sized["objective"], b_max=sized["b_max"],
                f=sized["f"], draft_len=ln, cu_len=cp["cu_len"],
                verify_idx=cp["verify_idx"], verify_tok=cp["verify_tok"],
                cost_used=sized["cost_used"], status=st | sized["status"])


def lmhead_logits(h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Backbone logits [n, K, vocab] (fp64) from bf16 hidden states h
    [n, K, d] and the bf16 output projection W [vocab, d]."""
    h64 = bf16_to_f64(h)
    W64 = bf16_to_f64(W)
    return h64 @ W64.T


def chain_lmhead(h: np.ndarray, W: np.ndarray, U: np.ndarray, V: np.ndarray,
                 last_token: np.ndarray, rows: np.ndarray | None = None) -> dict:
    """The chain over adj = h . W^T + U[prev] . V^T ("DSpark on MAX", *What
    DSpark is*, items 2-3): the drafter's output projection and the Markov
    bias as one score, the backbone logits never stored on the device.  All
    of h, W, U, V are bf16 bit patterns; ``rows`` as for chain()."""
    return chain(lmhead_logits(h, W), "f64", U, V, last_token, rows=rows)
