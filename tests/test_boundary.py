"""C-ABI boundary checks that need no GPU: the library loads, exports every
symbol the header declares, computes tree masks on the host, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import long_context_attention_tree_b300 as ts
import oracle
from long_context_attention_tree_b300 import build as ts_build
from long_context_attention_tree_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    ts_build.build()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "ts.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = header_symbols()
    assert len(names) >= 8
    L = ts.lib()
    for n in names:
        assert hasattr(L, n), n
    assert "sm_103a" in ts.ts_version()


@pytest.mark.parametrize("parent", [
    W.verify_parents(), W.tree_parents([1, 3, 3, 3]), W.tree_parents([3, 3, 3, 3]),
    W.chain_parents(32, 4), [-1] * 128, [-1] + list(range(127)), [],
    W.verify_parents((1, 9, 9, 9)), W.verify_parents((3, 3, 3, 3)), [-1] + list(range(1023)), [-1] * 129,
])
def test_mask_matches_oracle_visibility(parent):
    mask = ts.ts_tree_mask_from_parents(parent)
    T = len(parent)
    if T == 0:
        return
    mw = max(2, (T + 63) // 64)
    assert mask.shape == (T, mw)
    vis = oracle.visible(parent)
    for i in range(0, T, max(1, T // 97)):
        bits = [(int(mask[i, u // 64]) >> (u % 64)) & 1 for u in range(T)]
        assert bits == vis[i].astype(int).tolist()
        assert all(((int(mask[i, u // 64]) >> (u % 64)) & 1) == 0 for u in range(T, 64 * mw))


@pytest.mark.parametrize("parent", [[-1, 1], [0], [-1, -2], [-1, 0, 5]])
def test_mask_rejects_bad_parents(parent):
    with pytest.raises(ts.TSError) as e:
        ts.ts_tree_mask_from_parents(parent)
    assert e.value.status == ts.TS_ERR_INVALID_ARG


def test_mask_rejects_too_many_rows():
    with pytest.raises(ts.TSError):
        ts.ts_tree_mask_from_parents([-1] * 1025)
    assert ts.lib().ts_tree_mask_words(128) == 2 and ts.lib().ts_tree_mask_words(129) == 3
    assert ts.lib().ts_tree_mask_words(820) == 13 and ts.lib().ts_tree_mask_words(1) == 2


def _attn(**kw):
    """Call ts_tree_attn with fake (never dereferenced) aligned pointers."""
    L = ts.lib()
    P = 0x10000
    a = dict(q=P, k=P, v=P, ld=5000, N=4096, T=40, Hq=4, Hkv=1, d=64, scale=0.125, mask=P, out=P,
             lse=None, scores=None, score_row=0, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return L.ts_tree_attn(a["q"], a["k"], a["v"], a["ld"], a["N"], a["T"], a["Hq"], a["Hkv"], a["d"], a["scale"],
                          a["mask"], a["out"], a["lse"], a["scores"], a["score_row"], a["ws"], a["ws_bytes"],
                          a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), ts.TS_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), ts.TS_ERR_INVALID_ARG),
    (dict(Hq=66, Hkv=1), ts.TS_ERR_UNSUPPORTED),
    (dict(T=1025, ld=6000), ts.TS_ERR_UNSUPPORTED),
    (dict(N=-1), ts.TS_ERR_INVALID_ARG),
    (dict(q=None), ts.TS_ERR_INVALID_ARG),
    (dict(mask=None), ts.TS_ERR_INVALID_ARG),
    (dict(k=0x10008), ts.TS_ERR_INVALID_ARG),
    (dict(ld=4100), ts.TS_ERR_INVALID_ARG),
    (dict(scale=0.0), ts.TS_ERR_INVALID_ARG),
    (dict(scores=0x10000, score_row=40), ts.TS_ERR_INVALID_ARG),
    (dict(ws=None), ts.TS_ERR_INVALID_ARG),
    (dict(ws_bytes=16), ts.TS_ERR_INVALID_ARG),
])
def test_tree_attn_rejects_before_launch(kw, status):
    assert _attn(**kw) == status
    assert ts.lib().ts_last_error()


def test_tree_attn_empty_batch_is_noop():
    assert _attn(T=0, q=None, mask=None) == ts.TS_OK


def test_workspace_size_is_consistent():
    for (T, Hq, Hkv, d, N) in [(40, 4, 1, 64, 4096), (120, 32, 8, 128, 20480), (4, 40, 8, 128, 4096)]:
        need = ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N)
        assert need % 4 == 0
        if need:
            assert _attn(T=T, Hq=Hq, Hkv=Hkv, d=d, N=N, ld=N + T, ws_bytes=need - 4) == ts.TS_ERR_INVALID_ARG


def test_select_gather_rejects():
    L = ts.lib()
    P = 0x10000
    # budget not a multiple of the chunk
    assert L.ts_select_gather(P, 8, 4096, 100, 64, 0, 0, P, P, 5000, 128, P, None, P, P, 4096, None) == ts.TS_ERR_INVALID_ARG
    # partial cache too short
    assert L.ts_select_gather(P, 8, 8192, 4096, 64, 0, 0, P, P, 8192, 128, P, None, P, P, 4000, None) == ts.TS_ERR_INVALID_ARG
    # chunk other than 64
    assert L.ts_select_gather(P, 8, 8192, 4096, 32, 0, 0, P, P, 8192, 128, P, None, P, P, 4096, None) == ts.TS_ERR_UNSUPPORTED
    # ld_kv below N (a ragged N is accepted: the last chunk is short)
    assert L.ts_select_gather(P, 8, 4100, 4096, 64, 0, 0, P, P, 4099, 128, P, None, P, P, 4096, None) == ts.TS_ERR_INVALID_ARG
    # misaligned part_len
    assert L.ts_select_gather(P, 8, 4100, 4096, 64, 0, 0, P, P, 4100, 128, P, P + 2, P, P, 4096, None) == ts.TS_ERR_INVALID_ARG
    # always-kept chunks beyond the budget, negative counts
    assert L.ts_select_gather(P, 8, 8192, 4096, 64, 40, 30, P, P, 8192, 128, P, None, P, P, 4096, None) == ts.TS_ERR_INVALID_ARG
    assert L.ts_select_gather(P, 8, 8192, 4096, 64, -1, 0, P, P, 8192, 128, P, None, P, P, 4096, None) == ts.TS_ERR_INVALID_ARG
    # more than 16384 chunks
    assert L.ts_select_gather(P, 8, 16384 * 64 + 1, 4096, 64, 0, 0, P, P, 1 << 21, 128, P, None, P, P, 4096,
                              None) == ts.TS_ERR_UNSUPPORTED


def test_select_chunks_rejects():
    L = ts.lib()
    P = 0x10000
    assert L.ts_select_chunks(P, 8, 4096, 100, 64, 0, 0, P, None, None) == ts.TS_ERR_INVALID_ARG   # budget % chunk
    assert L.ts_select_chunks(P, 8, 8192, 4096, 32, 0, 0, P, None, None) == ts.TS_ERR_UNSUPPORTED  # chunk != 64
    assert L.ts_select_chunks(P, 8, 4100, 4096, 64, 0, 0, P, P + 2, None) == ts.TS_ERR_INVALID_ARG  # part_len
    assert L.ts_select_chunks(P, 8, 8192, 4096, 64, 40, 30, P, None, None) == ts.TS_ERR_INVALID_ARG
    assert L.ts_select_chunks(None, 8, 8192, 4096, 64, 0, 0, P, None, None) == ts.TS_ERR_INVALID_ARG
    assert L.ts_select_chunks(P, 8, 0, 4096, 64, 0, 0, P, None, None) == ts.TS_OK  # nothing to select


def _gather_attn(N=20480, k_sel=64, ld_part=64 * 64 + 4, T=4, Hq=40, Hkv=8, d=128, sel=0x10000):
    P = 0x10000
    return ts.lib().ts_gather_tree_attn(P, P, P, N + 8, N, sel, k_sel, P, P, ld_part, T, Hq, Hkv, d, 0.088, P, P,
                                        None, P, 1 << 30, None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=5, ld_part=64 * 64 + 8), ts.TS_ERR_UNSUPPORTED),  # 5 rows x 5 heads > 24 pairs per KV head
    (dict(T=64, Hq=8, Hkv=8, ld_part=64 * 64 + 64), ts.TS_ERR_UNSUPPORTED),  # a tensor-core sized batch
    (dict(d=64), ts.TS_ERR_UNSUPPORTED),
    (dict(k_sel=0), ts.TS_ERR_INVALID_ARG),
    (dict(k_sel=321), ts.TS_ERR_INVALID_ARG),               # more chunks than the cache holds
    (dict(ld_part=64 * 64 + 3), ts.TS_ERR_INVALID_ARG),     # no room for the batch's own rows
    (dict(sel=None), ts.TS_ERR_INVALID_ARG),
    (dict(N=0), ts.TS_ERR_INVALID_ARG),
])
def test_gather_tree_attn_rejects(kw, status):
    assert _gather_attn(**kw) == status
    assert ts.lib().ts_last_error()


def test_tree_attn_merge_host_checks():
    L = ts.lib()
    P = 0x10000
    # a multi-split plan needs the workspace the unmerged half filled
    assert L.ts_tree_attn_merge(20480, 120, 40, 8, 128, P, None, P, 16, None) == ts.TS_ERR_INVALID_ARG
    assert L.ts_tree_attn_merge(20480, 120, 40, 8, 128, None, None, P, 1 << 30, None) == ts.TS_ERR_INVALID_ARG
    # one split (the kernel wrote the output) and an empty batch: nothing to do
    assert L.ts_tree_attn_merge(60, 4, 8, 8, 128, P, None, None, 0, None) == ts.TS_OK
    assert L.ts_tree_attn_merge(4096, 0, 40, 8, 128, None, None, None, 0, None) == ts.TS_OK
    assert L.ts_tree_attn_merge(4096, 4, 40, 7, 128, P, None, P, 1 << 30, None) == ts.TS_ERR_INVALID_ARG


def _select_gather_attn(scores=0x10000, N=20480, budget=4096, chunk=64, sink=0, recent=0, sel=0x10000,
                        ld_part=64 * 64 + 4, T=4, Hq=40, Hkv=8, d=128):
    P = 0x10000
    return ts.lib().ts_select_gather_tree_attn(scores, N, budget, chunk, sink, recent, sel, None, P, P, P, N + 8, P, P,
                                               ld_part, T, Hq, Hkv, d, 0.088, P, P, None, P, 1 << 30, None)


@pytest.mark.parametrize("kw,status", [
    (dict(budget=100), ts.TS_ERR_INVALID_ARG),               # budget not a multiple of the chunk
    (dict(chunk=32), ts.TS_ERR_UNSUPPORTED),
    (dict(scores=None), ts.TS_ERR_INVALID_ARG),
    (dict(sel=None), ts.TS_ERR_INVALID_ARG),
    (dict(N=0), ts.TS_ERR_INVALID_ARG),                       # nothing to select
    (dict(sink=40, recent=30), ts.TS_ERR_INVALID_ARG),        # always-kept chunks beyond the budget
    (dict(T=5, ld_part=64 * 64 + 8), ts.TS_ERR_UNSUPPORTED),  # 25 (row, head) pairs per KV head
    (dict(d=64), ts.TS_ERR_UNSUPPORTED),
    (dict(ld_part=64 * 64 + 3), ts.TS_ERR_INVALID_ARG),       # no room for the batch's own rows
    (dict(N=16384 * 64 + 1), ts.TS_ERR_UNSUPPORTED),          # 16385 chunks: the keys would overflow the K/V buffers
])
def test_select_gather_tree_attn_rejects(kw, status):
    assert _select_gather_attn(**kw) == status
    assert ts.lib().ts_last_error()


def test_rescore_tail_rejects():
    L = ts.lib()
    P = 0x10000
    # N_old above N_new
    assert L.ts_rescore_tail(P, 200, P, P, 300, 100, 8, 2, 128, 64, P + 4096, None) == ts.TS_ERR_INVALID_ARG
    # in place across a change of the chunk count
    assert L.ts_rescore_tail(P, 100, P, P, 300, 200, 8, 2, 128, 64, P, None) == ts.TS_ERR_INVALID_ARG
    # overlapping buffers
    assert L.ts_rescore_tail(P, 100, P, P, 300, 200, 8, 2, 128, 64, P + 4, None) == ts.TS_ERR_INVALID_ARG
    # chunk other than 64, ld_kv below N_new
    assert L.ts_rescore_tail(P, 100, P, P, 300, 200, 8, 2, 128, 32, P + 4096, None) == ts.TS_ERR_UNSUPPORTED
    assert L.ts_rescore_tail(P, 100, P, P, 150, 200, 8, 2, 128, 64, P + 4096, None) == ts.TS_ERR_INVALID_ARG
    # nothing to do
    assert L.ts_rescore_tail(None, 0, P, P, 300, 0, 8, 2, 128, 64, P, None) == ts.TS_OK


def test_partial_attention_needs_part_len():
    L = ts.lib()
    P = 0x10000
    st = L.ts_tree_attn_partial(P, P, P, 4100, 4096, 4, 40, 8, 128, 0.088, P, None, P, None, P, 1 << 30, None)
    assert st == ts.TS_ERR_INVALID_ARG and b"part_len" in L.ts_last_error()


def test_vocab_rejects():
    L = ts.lib()
    P = 0x10000
    f = L.ts_penalty_minp_verify
    ok = dict(logits=P, T=120, V=152064, history=P, W=1024, theta=1.2, min_p=0.1, temp=1.0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["logits"], a["T"], a["V"], a["history"], a["W"], a["theta"], a["min_p"], a["temp"],
                 P, P, 0, P, P, P, P, None, 0, None)
    assert call(T=0) == ts.TS_ERR_UNSUPPORTED
    assert call(V=200000) == ts.TS_ERR_UNSUPPORTED
    assert call(theta=0.0) == ts.TS_ERR_INVALID_ARG
    assert call(temp=-1.0) == ts.TS_ERR_INVALID_ARG
    assert call(min_p=1.5) == ts.TS_ERR_INVALID_ARG
    assert call(history=None) == ts.TS_ERR_INVALID_ARG
    assert call(logits=0x10002) == ts.TS_ERR_INVALID_ARG


def test_sampled_vocab_rejects():
    """The sampled entry point validates exactly like the greedy one."""
    L = ts.lib()
    P = 0x10000
    f = L.ts_penalty_minp_sample_verify
    ok = dict(logits=P, T=120, V=152064, history=P, W=1024, theta=1.2, min_p=0.1, temp=1.0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["logits"], a["T"], a["V"], a["history"], a["W"], a["theta"], a["min_p"], a["temp"],
                 2**64 - 1, 7, P, P, 0, P, P, P, P, None)
    assert call(T=0) == ts.TS_ERR_UNSUPPORTED
    assert call(T=1025) == ts.TS_ERR_UNSUPPORTED
    assert call(V=200000) == ts.TS_ERR_UNSUPPORTED
    assert call(theta=float("nan")) == ts.TS_ERR_INVALID_ARG
    assert call(temp=0.0) == ts.TS_ERR_INVALID_ARG
    assert call(min_p=-0.1) == ts.TS_ERR_INVALID_ARG
    assert call(W=-1) == ts.TS_ERR_INVALID_ARG
    assert call(history=None) == ts.TS_ERR_INVALID_ARG
    assert call(logits=0x10002) == ts.TS_ERR_INVALID_ARG


def test_product_does_not_import_oracle():
    """The product package and its sources never reference the oracle."""
    pkg = os.path.join(ROOT, "long_context_attention_tree_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "liboracle" not in text, fn


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), ts.TS_ERR_UNSUPPORTED),
    (dict(T=1025, ld=6000), ts.TS_ERR_UNSUPPORTED),
    (dict(d=96), ts.TS_ERR_UNSUPPORTED),
    (dict(Hkv=0), ts.TS_ERR_INVALID_ARG),
    (dict(N=-1), ts.TS_ERR_INVALID_ARG),
    (dict(ld=100), ts.TS_ERR_INVALID_ARG),
    (dict(k=0x10008), ts.TS_ERR_INVALID_ARG),
    (dict(path=0x10002), ts.TS_ERR_INVALID_ARG),
    (dict(result=None), ts.TS_ERR_INVALID_ARG),
])
def test_commit_path_rejects_bad_arguments(kw, status):
    """ts_commit_path validates on the host (fake, never dereferenced pointers)."""
    P = 0x10000
    a = dict(k=P, v=P, ld=4096 + 120, N=4096, T=120, Hkv=8, d=128, result=P, path=P)
    a.update(kw)
    rc = ts.lib().ts_commit_path(a["k"], a["v"], a["ld"], a["N"], a["T"], a["Hkv"], a["d"], a["result"], a["path"],
                                 None)
    assert rc == status, ts.lib().ts_last_error()
