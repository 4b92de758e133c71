"""ctypes binding of libdspark.so (argument marshalling only).

Every function here has the name of the C entry point it calls and passes
``torch`` tensors as raw device pointers together with the current CUDA
stream.  All arithmetic happens in the library's kernels: there is no CPU or
PyTorch fallback, and a missing library raises at the first call.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdspark.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dspark.h")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_WORKSPACE = 4
BF16 = 0
F32 = 1
DEV_TOKEN_OOR = 1
DEV_NAN_LOGIT = 2
DEV_CONF_OOR = 4
DEV_TABLE_SHORT = 8
DEV_COST_NONPOS = 16
DEV_TIMEOUT = 32
COST_FORCE_MONOTONE = 1
COST_FORCE_SUFFIX_MIN = 2
BUDGET_GREEDY_STOP = 4

_ERR_NAMES = {1: "DSPARK_ERR_INVALID_ARG", 2: "DSPARK_ERR_UNSUPPORTED",
              3: "DSPARK_ERR_CUDA", 4: "DSPARK_ERR_WORKSPACE"}

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_U32 = ctypes.c_uint32
_F = ctypes.c_float

_SIGS = {
    "dspark_version": (_I32, []),
    "dspark_sm_count": (_I32, []),
    "dspark_chain_workspace_size": (_SZ, [_I32, _I32]),
    "dspark_chain_draft": (_I32, [_P, _I32, _I64, _I64, _P, _P, _P, _I32, _I32,
                                  _I32, _I32, _P, _P, _P, _SZ, _P]),
    "dspark_chain_sample": (_I32, [_P, _I32, _I64, _I64, _P, _P, _P, _I32, _I32,
                                   _I32, _I32, ctypes.c_uint64, _U32, _F, _P,
                                   _P, _P, _SZ, _P]),
    "dspark_chain_lmhead": (_I32, [_P, _I64, _I64, _P, _P, _P, _P, _I32, _I32,
                                   _I32, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "dspark_chain_draft_noalloc": (_I32, [_P, _I32, _I64, _I64, _P, _P, _P,
                                          _I32, _I32, _I32, _I32, _P, _P, _P,
                                          _P]),
    "dspark_select_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "dspark_survival_topb": (_I32, [_P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                    _SZ, _P]),
    "dspark_choose_budget": (_I32, [_P, _P, _P, _P, _I32, _P, _F, _U32, _P, _P,
                                    _P, _SZ, _P]),
    "dspark_allocate_prefix": (_I32, [_P, _P, _I32, _I32, _P, _P, _SZ, _P]),
    "dspark_compact_verify": (_I32, [_P, _P, _I32, _I32, _P, _P, _P, _P, _SZ,
                                     _P]),
    "dspark_select_step": (_I32, [_P, _P, _I32, _I32, _P, _I32, _P, _F, _U32,
                                  _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _P, _P, _SZ, _P]),
    "dspark_select_step_stale": (_I32, [_P, _P, _P, _I32, _I32, _P, _I32, _P,
                                        _F, _U32, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "dspark_gather_verify_tokens": (_I32, [_P, _P, _P, _I32, _I32, _P, _P]),
    "dspark_greedy_verify": (_I32, [_P, _I32, _I64, _I32, _P, _P, _P, _P, _I32,
                                    _I32, _P, _P, _P, _P, _SZ, _P]),
    "dspark_force_monotone": (_I32, [_P, _P, _I32, _U32, _P]),
    "dspark_read_status": (_I32, [_P, _P, _P]),
    "dspark_clear_status": (_I32, [_P, _P]),
}

_lib = None


class DsparkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {_ERR_NAMES.get(code, code)}")
        self.code = code


def header_functions() -> list[str]:
    """Names of the entry points declared in include/dspark.h."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"DSPARK_API\s+[\w\s\*]+?\b(dspark_\w+)\s*\(", txt)))


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "speculative_decoding_draft_dspark_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, code, raise_on_error):
    if code != OK and raise_on_error:
        raise DsparkError(name, code)
    return code


def _nbytes(t):
    return t.numel() * t.element_size()


# ------------------------------------------------------------------ chain
def dspark_chain_workspace_size(N: int, K: int) -> int:
    return int(load().dspark_chain_workspace_size(N, K))


def dspark_chain_draft(logits, U, V, last_token, draft_tokens, draft_score,
                       workspace, *, N=None, K=None, vocab=None, rank=None,
                       stride_n=None, stride_k=None, logits_dtype=None,
                       stream=None, raise_on_error=True) -> int:
    """logits [N, K, vocab] (bf16 or fp32), U/V [vocab, rank] bf16,
    last_token [N] int32, draft_tokens [N, K] int32 (out), draft_score
    [N, K] fp32 (out) or None, workspace uint8 tensor (zero-filled once)."""
    import torch
    if logits_dtype is None:
        logits_dtype = BF16 if logits.dtype == torch.bfloat16 else F32
    N = logits.shape[0] if N is None else N
    K = logits.shape[1] if K is None else K
    vocab = logits.shape[2] if vocab is None else vocab
    rank = U.shape[1] if rank is None else rank
    stride_n = logits.stride(0) if stride_n is None else stride_n
    stride_k = logits.stride(1) if stride_k is None else stride_k
    code = load().dspark_chain_draft(
        _ptr(logits), logits_dtype, stride_n, stride_k, _ptr(U), _ptr(V),
        _ptr(last_token), N, K, vocab, rank, _ptr(draft_tokens),
        _ptr(draft_score), _ptr(workspace), _nbytes(workspace),
        _stream(stream))
    return _check("dspark_chain_draft", code, raise_on_error)


def dspark_chain_sample(logits, U, V, last_token, draft_tokens, draft_score,
                        workspace, *, seed, offset, temperature=1.0, N=None,
                        K=None, vocab=None, rank=None, stride_n=None,
                        stride_k=None, logits_dtype=None, stream=None,
                        raise_on_error=True) -> int:
    """dspark_chain_draft drawing each token from softmax(adj / temperature)
    (probabilistic drafting: a Gumbel-max draw over 16-entry blocks, then the
    entry inside the block); seed (uint64), offset (uint32) and temperature
    as in include/dspark.h."""
    import torch
    if logits_dtype is None:
        logits_dtype = BF16 if logits.dtype == torch.bfloat16 else F32
    N = logits.shape[0] if N is None else N
    K = logits.shape[1] if K is None else K
    vocab = logits.shape[2] if vocab is None else vocab
    rank = U.shape[1] if rank is None else rank
    stride_n = logits.stride(0) if stride_n is None else stride_n
    stride_k = logits.stride(1) if stride_k is None else stride_k
    code = load().dspark_chain_sample(
        _ptr(logits), logits_dtype, stride_n, stride_k, _ptr(U), _ptr(V),
        _ptr(last_token), N, K, vocab, rank, int(seed), int(offset),
        float(temperature), _ptr(draft_tokens), _ptr(draft_score),
        _ptr(workspace), _nbytes(workspace), _stream(stream))
    return _check("dspark_chain_sample", code, raise_on_error)


def dspark_chain_lmhead(h, W, U, V, last_token, draft_tokens, draft_score,
                        workspace, *, N=None, K=None, d=None, stride_n=None,
                        stride_k=None, stream=None, raise_on_error=True) -> int:
    """Chain over h . W^T + U[prev] . V^T: h [N, K, d] bf16 hidden states
    (or any layout given by N, K, d and the element strides), W [vocab, d]
    bf16 output projection, U/V [vocab, rank] bf16."""
    N = h.shape[0] if N is None else N
    K = h.shape[1] if K is None else K
    d = W.shape[1] if d is None else d
    vocab, rank = W.shape[0], U.shape[1]
    stride_n = h.stride(0) if stride_n is None else stride_n
    stride_k = h.stride(1) if stride_k is None else stride_k
    code = load().dspark_chain_lmhead(
        _ptr(h), stride_n, stride_k, _ptr(W), _ptr(U), _ptr(V),
        _ptr(last_token), N, K, vocab, d, rank, _ptr(draft_tokens),
        _ptr(draft_score), _ptr(workspace), _nbytes(workspace), _stream(stream))
    return _check("dspark_chain_lmhead", code, raise_on_error)


def dspark_chain_draft_noalloc(logits, U, V, last_token, draft_tokens,
                               draft_score, device_status=None, *, N=None,
                               K=None, vocab=None, rank=None, stride_n=None,
                               stride_k=None, logits_dtype=None, stream=None,
                               raise_on_error=True) -> int:
    """dspark_chain_draft without a workspace, for callers that cannot
    allocate device memory (scratch lives in the library's own fixed device
    array; see include/dspark.h).  device_status: optional uint32 device
    tensor that receives this call's status bits."""
    import torch
    if logits_dtype is None:
        logits_dtype = BF16 if logits.dtype == torch.bfloat16 else F32
    N = logits.shape[0] if N is None else N
    K = logits.shape[1] if K is None else K
    vocab = logits.shape[2] if vocab is None else vocab
    rank = U.shape[1] if rank is None else rank
    stride_n = logits.stride(0) if stride_n is None else stride_n
    stride_k = logits.stride(1) if stride_k is None else stride_k
    code = load().dspark_chain_draft_noalloc(
        _ptr(logits), logits_dtype, stride_n, stride_k, _ptr(U), _ptr(V),
        _ptr(last_token), N, K, vocab, rank, _ptr(draft_tokens),
        _ptr(draft_score), _ptr(device_status), _stream(stream))
    return _check("dspark_chain_draft_noalloc", code, raise_on_error)


# -------------------------------------------------------------- scheduler
def dspark_select_workspace_size(N: int, K: int, cost_len: int) -> int:
    return int(load().dspark_select_workspace_size(N, K, cost_len))


def dspark_survival_topb(conf, sampling_mask, survival, sorted_slots,
                         prefix_sum, n_eligible, n_sampling, workspace, *,
                         stream=None, raise_on_error=True) -> int:
    N, K = conf.shape
    code = load().dspark_survival_topb(
        _ptr(conf), _ptr(sampling_mask), N, K, _ptr(survival),
        _ptr(sorted_slots), _ptr(prefix_sum), _ptr(n_eligible),
        _ptr(n_sampling), _ptr(workspace), _nbytes(workspace), _stream(stream))
    return _check("dspark_survival_topb", code, raise_on_error)


def dspark_choose_budget(prefix_sum, n_eligible, n_sampling, cost, T_dev,
                         draft_cost, flags, B, objective, workspace, *,
                         stream=None, raise_on_error=True) -> int:
    code = load().dspark_choose_budget(
        _ptr(prefix_sum), _ptr(n_eligible), _ptr(n_sampling), _ptr(cost),
        cost.numel(), _ptr(T_dev), float(draft_cost), int(flags), _ptr(B),
        _ptr(objective), _ptr(workspace), _nbytes(workspace), _stream(stream))
    return _check("dspark_choose_budget", code, raise_on_error)


def dspark_allocate_prefix(sorted_slots, B, N, K, draft_len, workspace, *,
                           stream=None, raise_on_error=True) -> int:
    code = load().dspark_allocate_prefix(
        _ptr(sorted_slots), _ptr(B), N, K, _ptr(draft_len), _ptr(workspace),
        _nbytes(workspace), _stream(stream))
    return _check("dspark_allocate_prefix", code, raise_on_error)


def dspark_compact_verify(draft_len, draft_tokens, N, K, cu_len, verify_idx,
                          verify_tok, workspace, *, stream=None,
                          raise_on_error=True) -> int:
    code = load().dspark_compact_verify(
        _ptr(draft_len), _ptr(draft_tokens), N, K, _ptr(cu_len),
        _ptr(verify_idx), _ptr(verify_tok), _ptr(workspace),
        _nbytes(workspace), _stream(stream))
    return _check("dspark_compact_verify", code, raise_on_error)


def dspark_select_step(conf, sampling_mask, cost, T_dev, draft_cost, flags,
                       draft_tokens, survival, sorted_slots, prefix_sum,
                       n_eligible, n_sampling, B, objective, draft_len, cu_len,
                       verify_idx, verify_tok, workspace, *, stream=None,
                       raise_on_error=True) -> int:
    N, K = conf.shape
    code = load().dspark_select_step(
        _ptr(conf), _ptr(sampling_mask), N, K, _ptr(cost), cost.numel(),
        _ptr(T_dev), float(draft_cost), int(flags), _ptr(draft_tokens),
        _ptr(survival), _ptr(sorted_slots), _ptr(prefix_sum), _ptr(n_eligible),
        _ptr(n_sampling), _ptr(B), _ptr(objective), _ptr(draft_len),
        _ptr(cu_len), _ptr(verify_idx), _ptr(verify_tok), _ptr(workspace),
        _nbytes(workspace), _stream(stream))
    return _check("dspark_select_step", code, raise_on_error)


def dspark_select_step_stale(conf_size, conf, sampling_mask, cost, T_dev,
                             draft_cost, flags, draft_tokens, survival,
                             sorted_slots, prefix_sum, n_eligible, n_sampling,
                             B, objective, draft_len, cu_len, verify_idx,
                             verify_tok, workspace, *, stream=None,
                             raise_on_error=True) -> int:
    N, K = conf.shape
    if tuple(conf_size.shape) != (N, K):
        raise ValueError("conf_size and conf must have the same [N, K] shape")
    code = load().dspark_select_step_stale(
        _ptr(conf_size), _ptr(conf), _ptr(sampling_mask), N, K, _ptr(cost),
        cost.numel(), _ptr(T_dev), float(draft_cost), int(flags),
        _ptr(draft_tokens), _ptr(survival), _ptr(sorted_slots),
        _ptr(prefix_sum), _ptr(n_eligible), _ptr(n_sampling), _ptr(B),
        _ptr(objective), _ptr(draft_len), _ptr(cu_len), _ptr(verify_idx),
        _ptr(verify_tok), _ptr(workspace), _nbytes(workspace), _stream(stream))
    return _check("dspark_select_step_stale", code, raise_on_error)


def dspark_gather_verify_tokens(verify_idx, B, draft_tokens, verify_tok, *,
                                stream=None, raise_on_error=True) -> int:
    N, K = draft_tokens.shape
    code = load().dspark_gather_verify_tokens(
        _ptr(verify_idx), _ptr(B), _ptr(draft_tokens), N, K, _ptr(verify_tok),
        _stream(stream))
    return _check("dspark_gather_verify_tokens", code, raise_on_error)


def dspark_greedy_verify(target_logits, draft_tokens, draft_len, cu_len,
                         sampling_mask, target_argmax, accepted, bonus,
                         workspace, *, vocab=None, row_stride=None,
                         logits_dtype=None, stream=None,
                         raise_on_error=True) -> int:
    import torch
    if logits_dtype is None:
        logits_dtype = BF16 if target_logits.dtype == torch.bfloat16 else F32
    vocab = target_logits.shape[-1] if vocab is None else vocab
    row_stride = target_logits.stride(0) if row_stride is None else row_stride
    N, K = draft_tokens.shape
    code = load().dspark_greedy_verify(
        _ptr(target_logits), logits_dtype, row_stride, vocab,
        _ptr(draft_tokens), _ptr(draft_len), _ptr(cu_len), _ptr(sampling_mask),
        N, K, _ptr(target_argmax), _ptr(accepted), _ptr(bonus),
        _ptr(workspace), _nbytes(workspace), _stream(stream))
    return _check("dspark_greedy_verify", code, raise_on_error)


def dspark_force_monotone(cost_in, cost_out, mode=COST_FORCE_MONOTONE, *,
                          stream=None, raise_on_error=True) -> int:
    code = load().dspark_force_monotone(_ptr(cost_in), _ptr(cost_out),
                                        cost_in.numel(), int(mode),
                                        _stream(stream))
    return _check("dspark_force_monotone", code, raise_on_error)


def dspark_read_status(workspace, *, stream=None) -> int:
    out = ctypes.c_uint32(0)
    code = load().dspark_read_status(_ptr(workspace), ctypes.byref(out),
                                     _stream(stream))
    _check("dspark_read_status", code, True)
    return int(out.value)


def dspark_clear_status(workspace, *, stream=None) -> int:
    code = load().dspark_clear_status(_ptr(workspace), _stream(stream))
    return _check("dspark_clear_status", code, True)


def dspark_sm_count() -> int:
    return int(load().dspark_sm_count())


def dspark_version() -> int:
    return int(load().dspark_version())


# ------------------------------------------------------- buffer helpers
def new_workspace(nbytes: int, device="cuda"):
    """Zero-filled uint8 device buffer, 256-byte aligned by the allocator."""
    import torch
    return torch.zeros(max(256, int(nbytes)), dtype=torch.uint8, device=device)
