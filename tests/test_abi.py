"""The C-ABI library builds, loads and exports every declared entry point,
and its host-side validation rejects bad arguments before any CUDA call (so
these run without a GPU)."""
import ctypes

import pytest

import __graft_entry__
from speculative_decoding_draft_dspark_gb300 import dspark as D


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return D.load()


def test_exports_every_header_function(lib):
    names = D.header_functions()
    assert len(names) == 19
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(D._SIGS)


def test_version_and_sizes(lib):
    assert lib.dspark_version() == 100
    assert lib.dspark_chain_workspace_size(256, 7) >= 256 + 256 * 7 * 8
    assert lib.dspark_chain_workspace_size(0, 7) == 0
    assert lib.dspark_select_workspace_size(256, 7, 8192) >= 4
    assert lib.dspark_select_workspace_size(256, 0, 8192) == 0


FAKE = 1 << 20  # aligned, never dereferenced: validation fails first


def _chain(lib, **kw):
    a = dict(logits=FAKE, dt=0, sn=7 * 1024, sk=1024, U=FAKE, V=FAKE,
             last=FAKE, N=4, K=7, vocab=1024, rank=16, draft=FAKE, score=None,
             ws=FAKE * 2, wsb=1 << 16, stream=None)
    a.update(kw)
    return lib.dspark_chain_draft(a["logits"], a["dt"], a["sn"], a["sk"], a["U"],
                                  a["V"], a["last"], a["N"], a["K"], a["vocab"],
                                  a["rank"], a["draft"], a["score"], a["ws"],
                                  a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(logits=None), D.ERR_INVALID_ARG),
    (dict(U=None), D.ERR_INVALID_ARG),
    (dict(draft=None), D.ERR_INVALID_ARG),
    (dict(dt=7), D.ERR_INVALID_ARG),
    (dict(N=0), D.ERR_INVALID_ARG),
    (dict(K=33), D.ERR_UNSUPPORTED),
    (dict(rank=24), D.ERR_UNSUPPORTED),
    (dict(rank=272), D.ERR_UNSUPPORTED),
    (dict(vocab=1020, sn=7 * 1020, sk=1020), D.ERR_UNSUPPORTED),
    (dict(sn=7 * 1024 + 4), D.ERR_INVALID_ARG),
    (dict(sk=1000), D.ERR_INVALID_ARG),
    (dict(logits=FAKE + 8), D.ERR_INVALID_ARG),
    (dict(ws=None), D.ERR_WORKSPACE),
    (dict(wsb=64), D.ERR_WORKSPACE),
    (dict(ws=FAKE * 2 + 16), D.ERR_WORKSPACE),
])
def test_chain_validation(lib, kw, code):
    assert _chain(lib, **kw) == code


def test_chain_sample_validation(lib):
    f = lib.dspark_chain_sample
    ok = dict(logits=FAKE, dt=D.BF16, sn=1024 * 7, sk=1024, U=FAKE, V=FAKE,
              last=FAKE, N=4, K=7, vocab=1024, rank=16, seed=1, offset=0,
              tau=1.0, draft=FAKE, score=None, ws=FAKE * 2, wsb=1 << 16,
              stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*a.values())

    for tau in (0.0, -1.0, float("nan"), float("inf"), 1e-45):
        assert call(tau=tau) == D.ERR_INVALID_ARG, tau
    assert call(logits=None) == D.ERR_INVALID_ARG
    assert call(K=40) == D.ERR_UNSUPPORTED
    assert call(rank=24) == D.ERR_UNSUPPORTED
    assert call(wsb=16) == D.ERR_WORKSPACE


def test_chain_lmhead_validation(lib):
    f = lib.dspark_chain_lmhead
    ok = dict(h=FAKE, sn=7 * 2048, sk=2048, W=FAKE, U=FAKE, V=FAKE, last=FAKE,
              N=4, K=7, vocab=1024, d=2048, rank=16, draft=FAKE, score=None,
              ws=FAKE * 2, wsb=1 << 16, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*a.values())

    assert call(h=None) == D.ERR_INVALID_ARG
    assert call(W=None) == D.ERR_INVALID_ARG
    assert call(d=100) == D.ERR_UNSUPPORTED           # not a multiple of 64
    assert call(d=0) == D.ERR_INVALID_ARG
    assert call(rank=300) == D.ERR_UNSUPPORTED
    assert call(vocab=1020) == D.ERR_UNSUPPORTED
    assert call(sn=2047) == D.ERR_INVALID_ARG
    assert call(sk=2044) == D.ERR_INVALID_ARG
    assert call(h=FAKE + 8) == D.ERR_INVALID_ARG       # misaligned
    assert call(wsb=16) == D.ERR_WORKSPACE


def test_select_validation(lib):
    f = lib.dspark_select_step
    ok = dict(conf=FAKE, mask=None, N=4, K=7, cost=FAKE, L=64, T=FAKE, dc=0.0,
              flags=0, draft=None, surv=None, srt=None, pre=None, ne=None,
              ns=None, B=FAKE, obj=None, ln=FAKE, cu=FAKE, vi=FAKE, vt=None,
              ws=FAKE * 2, wsb=256, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*a.values())

    assert call(conf=None) == D.ERR_INVALID_ARG
    assert call(N=0) == D.ERR_INVALID_ARG
    assert call(K=40) == D.ERR_UNSUPPORTED
    assert call(N=4096, K=5) == D.ERR_UNSUPPORTED      # N*K > 16384
    assert call(L=0) == D.ERR_INVALID_ARG
    assert call(flags=64) == D.ERR_INVALID_ARG
    assert call(B=None) == D.ERR_INVALID_ARG
    assert call(ws=None) == D.ERR_WORKSPACE
    assert call(wsb=16) == D.ERR_WORKSPACE
    assert lib.dspark_force_monotone(FAKE, FAKE, 64, 9, None) == D.ERR_INVALID_ARG
    assert lib.dspark_force_monotone(None, FAKE, 64, 1, None) == D.ERR_INVALID_ARG
    assert lib.dspark_read_status(None, ctypes.byref(ctypes.c_uint32()), None) \
        == D.ERR_INVALID_ARG


def test_select_stale_validation(lib):
    f = lib.dspark_select_step_stale
    ok = dict(conf_size=FAKE, conf=FAKE, mask=None, N=4, K=7, cost=FAKE, L=64,
              T=FAKE, dc=0.0, flags=0, draft=None, surv=None, srt=None,
              pre=None, ne=None, ns=None, B=FAKE, obj=None, ln=FAKE, cu=FAKE,
              vi=FAKE, vt=None, ws=FAKE * 2, wsb=256, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*a.values())

    assert call(conf_size=None) == D.ERR_INVALID_ARG
    assert call(conf=None) == D.ERR_INVALID_ARG
    assert call(K=40) == D.ERR_UNSUPPORTED
    assert call(flags=64) == D.ERR_INVALID_ARG
    assert call(wsb=16) == D.ERR_WORKSPACE


def test_product_path_never_touches_the_oracle():
    import os
    import re
    pkg = os.path.dirname(D.__file__)
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(root, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), fn
                assert "oracle/" not in src, fn


def _noalloc(lib, **kw):
    a = dict(logits=FAKE, dt=0, sn=7 * 1024, sk=1024, U=FAKE, V=FAKE,
             last=FAKE, N=4, K=7, vocab=1024, rank=16, draft=FAKE, score=None,
             status=None, stream=None)
    a.update(kw)
    return lib.dspark_chain_draft_noalloc(
        a["logits"], a["dt"], a["sn"], a["sk"], a["U"], a["V"], a["last"],
        a["N"], a["K"], a["vocab"], a["rank"], a["draft"], a["score"],
        a["status"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(logits=None), D.ERR_INVALID_ARG),
    (dict(last=None), D.ERR_INVALID_ARG),
    (dict(dt=7), D.ERR_INVALID_ARG),
    (dict(N=0), D.ERR_INVALID_ARG),
    (dict(K=33), D.ERR_UNSUPPORTED),
    (dict(rank=24), D.ERR_UNSUPPORTED),
    (dict(sk=1000), D.ERR_INVALID_ARG),
    (dict(V=FAKE + 8), D.ERR_INVALID_ARG),
    # 4096 x 8 slots need about 262 KB of scratch, over the 256 KiB array
    (dict(N=4096, K=8, sn=8 * 1024), D.ERR_UNSUPPORTED),
])
def test_noalloc_checks_before_any_cuda_call(lib, kw, code):
    """Every check of the no-allocation entry point runs before its first
    CUDA call, so a rejected call enqueues nothing.  Without a GPU any CUDA
    call would fail with DSPARK_ERR_CUDA, so the argument error itself shows
    the order; with one, the call returns before touching the stream."""
    assert _noalloc(lib, **kw) == code
