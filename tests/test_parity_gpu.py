"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Bars: bit-exact for chunk scores on integer data, selected indices, gathered
caches, targets, min-p counts and acceptance; bf16 attention outputs within
max-abs 2e-2 and relative L2 1e-2 of the fp64 result; LSE within 1e-3.

The tensor-core path rounds every softmax weight to bf16 for the P.V product
and normalises the output by the sum of those rounded weights; when the call
asks for the log-sum-exp it also sums the unrounded weights, so the LSE keeps
fp32 accuracy (well inside 1e-3)."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_tree_b300 as ts
import oracle
from long_context_attention_tree_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 1e-2
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from long_context_attention_tree_b300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    torch.cuda.init()


def dev_mask(parent):
    return torch.from_numpy(ts.ts_tree_mask_from_parents(parent).view(np.int64)).cuda()


def run_attn(q, k, v, N, parent, scale, scores=False, score_row=0, stream=None):
    T, Hq, d = q.shape
    Hkv = k.shape[0]
    out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    nc = (N + 63) // 64
    sc = torch.full((Hkv, max(nc, 1)), float("nan"), dtype=torch.float32, device="cuda") if scores else None
    ws_n = ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    ts.ts_tree_attn(q, k, v, N, dev_mask(parent), out, lse=lse, chunk_scores=sc, score_row=score_row,
                    workspace=ws, scale=scale, stream=stream)
    torch.cuda.synchronize()
    # no bounded device-side wait may have given up
    assert ts.ts_device_error(True) == ts.TS_OK
    return out, lse, sc


def check_attn(out, lse, ref_o, ref_lse, what=""):
    o = out.float().cpu().double().numpy().reshape(ref_o.shape)
    err = np.abs(o - ref_o)
    rel = np.linalg.norm(o - ref_o) / max(np.linalg.norm(ref_o), 1e-30)
    assert err.max() <= MAX_ABS, f"{what}: max abs {err.max():.3e}"
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e}"
    l = lse.cpu().double().numpy().reshape(ref_lse.shape)
    assert np.abs(l - ref_lse).max() <= LSE_ABS, f"{what}: lse err {np.abs(l - ref_lse).max():.3e}"


def verify_parent(T):
    p = W.verify_parents()[:T] if T <= 120 else W.verify_parents() + W.chain_parents((T - 120) // 4 + 1, 4, 120)
    return p[:T]


CASES = [
    # T, Hq, Hkv, d, N, kind
    (1, 4, 1, 64, 0, "int"),
    (1, 8, 8, 128, 1, "normal"),
    (4, 32, 8, 128, 63, "int"),
    (4, 40, 8, 128, 4096, "int"),
    (40, 4, 1, 64, 4096, "int"),
    (40, 5, 1, 64, 65, "normal"),
    (64, 8, 2, 128, 64, "int"),
    (64, 16, 4, 128, 1000, "normal"),
    (120, 32, 8, 128, 2111, "int"),
    (120, 40, 8, 128, 640, "normal"),
    (128, 8, 8, 128, 777, "int"),
    (128, 4, 1, 64, 300, "normal"),
    (13, 20, 4, 128, 5000, "normal"),
    (120, 32, 1, 128, 129, "int"),   # group 32
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}_Hq{}_Hkv{}_d{}_N{}_{}".format(*c))
def test_tree_attn_matches_oracle(case):
    T, Hq, Hkv, d, N, kind = case
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=100 + T + N, device="cuda", value_kind=kind, ld_extra=5)
    parent = verify_parent(T)
    scale = 1.0 / math.sqrt(d)
    out, lse, _ = run_attn(q, k, v, N, parent, scale)
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, scale)
    check_attn(out, lse, ro, rl, str(case))


@pytest.mark.parametrize("branching,chains,Hq,Hkv,d,N", [
    ((3, 3, 3, 3), 20, 40, 8, 128, 3000),   # 200 rows, GQA group 5
    ((1, 9, 9, 9), 0, 8, 2, 128, 1500),     # 820 rows, group 4
    ((1, 9, 9, 9), 20, 10, 2, 128, 701),    # 900 rows, group 5
    ((3, 3, 3, 3), 20, 8, 8, 128, 2000),    # 200 rows, MHA
    ((1, 9, 9, 9), 20, 4, 1, 64, 500),      # 900 rows, head dim 64 (CUDA cores)
])
def test_wide_trees_beyond_128_rows(branching, chains, Hq, Hkv, d, N):
    """The tree ablations of the pages ([3,3,3,3], [1,9,9,9]) with and without
    the n-gram chains: multi-word masks, many M-tiles per KV head."""
    parent = W.verify_parents(branching, chains)
    T = len(parent)
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=T + N, device="cuda", value_kind="normal", ld_extra=2)
    scale = 1 / math.sqrt(d)
    out, lse, sc = run_attn(q, k, v, N, parent, scale, scores=True, score_row=T - 1)
    assert ts.ts_tree_attn_uses_tensor_cores(T, Hq, Hkv, d, N) == (d == 128)
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, scale)
    check_attn(out, lse, ro, rl, f"T{T}")
    rs = oracle.score_chunks(q[T - 1].cpu(), k.cpu(), N)
    np.testing.assert_allclose(sc.cpu().numpy(), rs, rtol=1e-4, atol=1e-2)


def test_wide_tree_cuda_core_path_matches(monkeypatch):
    monkeypatch.setenv("TS_FORCE_SIMT", "1")
    parent = W.verify_parents((1, 9, 9, 9), 20)
    T, Hq, Hkv, d, N = len(parent), 10, 2, 128, 333
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=4, device="cuda")
    out, lse, sc = run_attn(q, k, v, N, parent, 1 / math.sqrt(d), scores=True, score_row=5)
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, 1 / math.sqrt(d))
    check_attn(out, lse, ro, rl)
    np.testing.assert_array_equal(sc.cpu().numpy(), oracle.score_chunks(q[5].cpu(), k.cpu(), N).astype(np.float32))


def test_tensor_core_path_is_selected_and_status_clean():
    assert ts.ts_tree_attn_uses_tensor_cores(120, 32, 8, 128, 20480)
    assert ts.ts_tree_attn_uses_tensor_cores(64, 40, 8, 128, 1)
    assert not ts.ts_tree_attn_uses_tensor_cores(63, 32, 8, 128, 20480)
    assert not ts.ts_tree_attn_uses_tensor_cores(120, 4, 1, 64, 4096)
    assert ts.ts_device_error(True) == ts.TS_OK


@pytest.mark.parametrize("T", [64, 65, 100, 120, 128])
@pytest.mark.parametrize("G", [1, 3, 4, 5, 8, 32])
def test_tensor_core_group_sizes(T, G):
    Hkv = 2 if G < 32 else 1
    Hq, d, N = G * Hkv, 128, 1000 + 7 * T
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=T * 100 + G, device="cuda", value_kind="normal", ld_extra=3)
    parent = verify_parent(T)
    assert ts.ts_tree_attn_uses_tensor_cores(T, Hq, Hkv, d, N)
    out, lse, sc = run_attn(q, k, v, N, parent, 1 / math.sqrt(d), scores=True, score_row=T - 1)
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, 1 / math.sqrt(d))
    check_attn(out, lse, ro, rl, f"T{T} G{G}")
    rs = oracle.score_chunks(q[T - 1].cpu(), k.cpu(), N)
    np.testing.assert_allclose(sc.cpu().numpy(), rs, rtol=1e-4, atol=1e-2)
    assert ts.ts_device_error(True) == ts.TS_OK


def test_tree_attn_forced_cuda_core_path_matches(monkeypatch):
    """Force the CUDA-core kernel at T=120 (cross-check of the tensor-core path)."""
    monkeypatch.setenv("TS_FORCE_SIMT", "1")
    T, Hq, Hkv, d, N = 120, 32, 8, 128, 3000
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=5, device="cuda")
    parent = W.verify_parents()
    out, lse, _ = run_attn(q, k, v, N, parent, 1 / math.sqrt(d))
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, 1 / math.sqrt(d))
    check_attn(out, lse, ro, rl)


@pytest.mark.parametrize("name", ["tiny", "llama8b-20k"])
def test_workload_full_parity(name):
    """The tiny workload and the LLaMA3.1-8B 20K layer, every output row."""
    cfg = W.WORKLOADS[name]
    x = W.make_layer_inputs(cfg, 0, device="cuda")
    out, lse, sc = run_attn(x.q, x.k, x.v, cfg.N, cfg.parents, cfg.scale, scores=True)
    ro, rl = oracle.tree_attn(x.q.cpu(), x.k.cpu(), x.v.cpu(), cfg.N, cfg.parents, cfg.scale)
    check_attn(out, lse, ro, rl, cfg.name)
    rs = oracle.score_chunks(x.q[0].cpu(), x.k.cpu(), cfg.N)
    np.testing.assert_array_equal(sc.cpu().numpy(), rs.astype(np.float32))


@pytest.mark.parametrize("N", [1, 63, 64, 65, 4096, 20480])
def test_score_chunks_bit_exact(N):
    Hq, Hkv, d = 32, 8, 128
    q, k, _ = W.make_qkv(120, Hq, Hkv, d, N, seed=N, device="cuda")
    nc = (N + 63) // 64
    sc = torch.full((Hkv, nc), float("nan"), dtype=torch.float32, device="cuda")
    ts.ts_score_chunks(q[0], k, N, sc)
    torch.cuda.synchronize()
    rs = oracle.score_chunks(q[0].cpu(), k.cpu(), N)
    np.testing.assert_array_equal(sc.cpu().numpy(), rs.astype(np.float32))
    # the fused scores of the attention pass agree bit for bit
    _, _, fs = run_attn(q, k, _dummy_v(k), N, W.verify_parents(), 1 / math.sqrt(d), scores=True, score_row=0)
    np.testing.assert_array_equal(fs.cpu().numpy(), sc.cpu().numpy())


def _dummy_v(k):
    return torch.zeros_like(k)


@pytest.mark.parametrize("score_row", [0, 7, 119])
def test_fused_scores_any_row(score_row):
    Hq, Hkv, d, N = 40, 8, 128, 1280
    q, k, v = W.make_qkv(120, Hq, Hkv, d, N, seed=score_row, device="cuda")
    _, _, fs = run_attn(q, k, v, N, W.verify_parents(), 1 / math.sqrt(d), scores=True, score_row=score_row)
    rs = oracle.score_chunks(q[score_row].cpu(), k.cpu(), N)
    np.testing.assert_array_equal(fs.cpu().numpy(), rs.astype(np.float32))


@pytest.mark.parametrize("T,Hq,Hkv,N,score_row", [(4, 40, 8, 4100, 3), (4, 32, 8, 1000, 0), (1, 8, 8, 63, 0),
                                                   (6, 16, 4, 130, 5), (4, 32, 32, 257, 2),
                                                   (2, 40, 8, 4090, 1),    # 10 pairs; batch rows straddle a block
                                                   (3, 24, 8, 31, 2),      # 9 pairs; one block holds all of it
                                                   (12, 16, 8, 6000, 11)])  # 24 pairs; 12-row tail
def test_small_batch_fused_scores_and_attention(T, Hq, Hkv, N, score_row):
    """Batches of at most 24 (row, head) pairs per KV head run on the CUDA-core
    small-batch kernel: its fused chunk scores are bit-exact, its output within
    the attention bars, including a ragged last KV range."""
    d = 128
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=300 + N, device="cuda")
    parent = verify_parent(T)
    out, lse, fs = run_attn(q, k, v, N, parent, 1 / math.sqrt(d), scores=True, score_row=score_row)
    rs = oracle.score_chunks(q[score_row].cpu(), k.cpu(), N)
    np.testing.assert_array_equal(fs.cpu().numpy(), rs.astype(np.float32))
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, 1 / math.sqrt(d))
    check_attn(out, lse, ro, rl, "small batch")


@pytest.mark.parametrize("N,budget,d", [(4096, 1024, 64), (20480, 4096, 128), (64 * 70, 4096, 128),
                                        (102400, 4096, 128), (640, 4096, 128), (4100, 4096, 128),
                                        (20483, 4096, 128), (102403, 4096, 128), (1000, 1024, 64), (37, 4096, 128)])
def test_select_gather_bit_exact(N, budget, d):
    """Selection, gathered caches and gathered lengths, including a short last
    chunk (N not a multiple of 64): its rows past N stay untouched."""
    Hq, Hkv = 32, 8
    q, k, v = W.make_qkv(1, Hq, Hkv, d, N, seed=N + budget, device="cuda")
    nc = (N + 63) // 64
    sc = torch.empty((Hkv, nc), dtype=torch.float32, device="cuda")
    ts.ts_score_chunks(q[0], k, N, sc)
    kk = min(budget // 64, nc)
    sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
    plen = torch.full((Hkv,), -1, dtype=torch.int32, device="cuda")
    ld_part = kk * 64 + 4
    fill = torch.full((Hkv, ld_part, d), 3.0, dtype=torch.bfloat16)
    kp, vp = fill.cuda(), fill.cuda()
    ts.ts_select_gather(sc, N, budget, k, v, sel, kp, vp, part_len=plen)
    torch.cuda.synchronize()
    scores = sc.cpu().numpy()
    np.testing.assert_array_equal(scores, oracle.score_chunks(q[0].cpu(), k.cpu(), N).astype(np.float32))
    rsel = oracle.select(scores, budget // 64)
    np.testing.assert_array_equal(sel.cpu().numpy(), rsel)
    rk, rl = oracle.gather(rsel, k.cpu(), N, 64, ld_part, fill=fill, return_len=True)
    assert torch.equal(kp.cpu(), rk)
    assert torch.equal(vp.cpu(), oracle.gather(rsel, v.cpu(), N, 64, ld_part, fill=fill))
    np.testing.assert_array_equal(plen.cpu().numpy(), rl)


@pytest.mark.parametrize("N,Hq,Hkv,d", [(4100, 40, 8, 128), (1000, 32, 32, 128), (130, 8, 2, 64), (4096, 40, 8, 128)])
def test_partial_cache_drafting_with_a_short_last_chunk(N, Hq, Hkv, d):
    """Heads that selected the short last chunk hold fewer gathered tokens; the
    drafting attention over the compact cache sees exactly those."""
    Td, budget = 4, 1024
    q, k, v = W.make_qkv(Td, Hq, Hkv, d, N, seed=N + Hkv, device="cuda", value_kind="normal")
    nc = (N + 63) // 64
    rng = np.random.default_rng(N)
    s = rng.integers(-50, 50, size=(Hkv, nc)).astype(np.float32)
    s[::2, nc - 1] = 1000.0   # every other head keeps the last chunk,
    s[1::2, nc - 1] = -1000.0  # the others drop it
    kk = min(budget // 64, nc)
    B = kk * 64
    sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
    plen = torch.empty((Hkv,), dtype=torch.int32, device="cuda")
    kp = torch.full((Hkv, B + Td, d), 7.0, dtype=torch.bfloat16, device="cuda")  # stale rows stand out
    vp = torch.full_like(kp, -7.0)
    kp[:, B:] = k[:, N:N + Td]
    vp[:, B:] = v[:, N:N + Td]
    ts.ts_select_gather(torch.from_numpy(s).cuda(), N, budget, k, v, sel, kp, vp, part_len=plen)
    parent = [-1, 0, 1, 2]
    out = torch.empty((Td, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Td, Hq), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(Td, Hq, Hkv, d, B)), dtype=torch.uint8, device="cuda")
    ts.ts_tree_attn_partial(q, kp, vp, B, dev_mask(parent), plen, out, lse=lse, workspace=ws, scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK
    rsel = oracle.select(s, budget // 64)
    np.testing.assert_array_equal(sel.cpu().numpy(), rsel)
    _, rl = oracle.gather(rsel, k.cpu(), N, 64, B + Td, return_len=True)
    np.testing.assert_array_equal(plen.cpu().numpy(), rl)
    if N % 64 and nc > kk:  # (when every chunk fits the budget, every head holds all N tokens)
        assert (rl[::2] < B).all() and (rl[1::2] == B).all()
    ro, rlse = oracle.tree_attn(q.cpu(), kp.cpu(), vp.cpu(), B, parent, 1 / math.sqrt(d), prefix_len=rl)
    check_attn(out, lse, ro, rlse, "partial")


@pytest.mark.parametrize("N,Hq,Hkv,Td,budget", [
    (4100, 40, 8, 4, 1024),     # 20 (row, head) pairs per KV head, short last chunk
    (20480, 40, 8, 4, 4096),
    (20483, 32, 8, 4, 4096),    # 16 pairs
    (102403, 40, 8, 4, 4096),
    (1000, 32, 32, 4, 1024),    # 4 pairs; the budget covers every chunk, the short one last
    (300, 8, 8, 24, 256),       # 24 pairs (the largest batch of the kernel)
    (4096, 16, 4, 6, 4096),     # 24 pairs, no short chunk
    (5000, 40, 8, 1, 2048),     # one row
    (2000, 40, 8, 3, 1024),     # 15 pairs (a padding row)
    (3000, 40, 8, 2, 2048),     # 10 pairs
    (64, 40, 8, 4, 4096),       # one chunk: the gathered cache is a single block pair
])
def test_gather_tree_attn_matches_oracle_and_the_two_calls(N, Hq, Hkv, Td, budget):
    """The gather fused with the drafting pass: the compact cache bit-exact
    against the oracle's gather (rows a selected short last chunk lacks keep
    their old contents), the output within the bars against the oracle over the
    gathered cache, and bit-identical to ts_select_gather followed by
    ts_tree_attn_partial, and to the one-pass call that also selects."""
    d = 128
    q, k, v = W.make_qkv(Td, Hq, Hkv, d, N, seed=N + 7 * Td, device="cuda", value_kind="normal")
    nc = (N + 63) // 64
    rng = np.random.default_rng(N + Td)
    s = rng.integers(-50, 50, size=(Hkv, nc)).astype(np.float32)
    s[::2, nc - 1] = 1000.0    # every other head keeps the short last chunk,
    s[1::2, nc - 1] = -1000.0  # the others drop it
    scores = torch.from_numpy(s).cuda()
    kk = min(budget // 64, nc)
    B = kk * 64
    fill_k = torch.full((Hkv, B + Td, d), 7.0, dtype=torch.bfloat16, device="cuda")  # stale rows stand out
    fill_v = torch.full_like(fill_k, -7.0)
    fill_k[:, B:] = k[:, N:N + Td]
    fill_v[:, B:] = v[:, N:N + Td]
    parent = list(range(-1, Td - 1))
    mask = dev_mask(parent)
    ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(Td, Hq, Hkv, d, B)), dtype=torch.uint8, device="cuda")
    scale = 1 / math.sqrt(d)

    sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
    plen = torch.empty((Hkv,), dtype=torch.int32, device="cuda")
    kp, vp = fill_k.clone(), fill_v.clone()
    out = torch.empty((Td, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Td, Hq), dtype=torch.float32, device="cuda")
    ts.ts_select_chunks(scores, N, budget, sel, part_len=plen)
    ts.ts_gather_tree_attn(q, k, v, N, sel, kp, vp, mask, out, lse=lse, workspace=ws, scale=scale)

    sel2 = torch.empty_like(sel)
    plen2 = torch.empty_like(plen)
    kp2, vp2 = fill_k.clone(), fill_v.clone()
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    ts.ts_select_gather(scores, N, budget, k, v, sel2, kp2, vp2, part_len=plen2)
    ts.ts_tree_attn_partial(q, kp2, vp2, B, mask, plen2, out2, lse=lse2, workspace=ws, scale=scale)
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK

    rsel = oracle.select(s, budget // 64)
    np.testing.assert_array_equal(sel.cpu().numpy(), rsel)
    rk, rl = oracle.gather(rsel, k.cpu(), N, 64, B + Td, fill=fill_k.cpu(), return_len=True)
    assert torch.equal(kp.cpu(), rk)
    assert torch.equal(vp.cpu(), oracle.gather(rsel, v.cpu(), N, 64, B + Td, fill=fill_v.cpu()))
    np.testing.assert_array_equal(plen.cpu().numpy(), rl)
    ro, rlse = oracle.tree_attn(q.cpu(), kp.cpu(), vp.cpu(), B, parent, scale, prefix_len=rl)
    check_attn(out, lse, ro, rlse, "gather + draft")
    # the two-call path: same selection, same caches, same output bits
    assert torch.equal(sel, sel2) and torch.equal(plen, plen2)
    assert torch.equal(kp, kp2) and torch.equal(vp, vp2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # and the one-pass call that also selects: the same bits again
    sel3 = torch.full_like(sel, -1)
    plen3 = torch.full_like(plen, -1)
    kp3, vp3 = fill_k.clone(), fill_v.clone()
    out3, lse3 = torch.empty_like(out), torch.empty_like(lse)
    ts.ts_select_gather_tree_attn(scores, q, k, v, N, budget, sel3, kp3, vp3, mask, out3, part_len=plen3, lse=lse3,
                                  workspace=ws, scale=scale)
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK
    assert torch.equal(sel3, sel) and torch.equal(plen3, plen)
    assert torch.equal(kp3, kp) and torch.equal(vp3, vp)
    assert torch.equal(out3, out) and torch.equal(lse3, lse)


@pytest.mark.parametrize("N,Hq,Hkv,Td,budget,sink,recent,kind", [
    (102400, 40, 8, 4, 4096, 1, 4, "normal"),        # the drafting shape with always-kept chunks
    (16384 * 64 - 5, 4, 1, 4, 4096, 0, 0, "normal"),  # the most chunks a call takes (keys over both K/V buffers)
    (16384 * 64, 8, 1, 2, 64 * 300, 2, 3, "ties"),
    (5000, 40, 8, 4, 2048, 3, 2, "constant"),          # every score equal: the lowest indices complete k
    (3000, 16, 4, 3, 64 * 47, 0, 0, "normal"),         # the budget covers every chunk
])
def test_one_pass_select_sink_recent_and_most_chunks(N, Hq, Hkv, Td, budget, sink, recent, kind):
    """The one-pass call (each CTA selects its head's chunks) with always-kept
    first/last chunks, continuous, tied and constant scores, up to 16384
    chunks: indices and gathered lengths bit-exact against the oracle's
    selection, and every output bit-identical to ts_select_gather followed by
    ts_tree_attn_partial (whose gather and attention other tests pin to the
    oracle); at the smaller sizes the attention against the oracle too."""
    d = 128
    q, k, v = W.make_qkv(Td, Hq, Hkv, d, N, seed=N + Td + sink, device="cuda", value_kind="normal")
    nc = (N + 63) // 64
    rng = np.random.default_rng(N + 3 * Td)
    if kind == "normal":
        s = rng.standard_normal((Hkv, nc)).astype(np.float32)
    elif kind == "ties":
        s = rng.integers(-3, 4, size=(Hkv, nc)).astype(np.float32)
    else:
        s = np.full((Hkv, nc), 1.5, dtype=np.float32)
    scores = torch.from_numpy(s).cuda()
    kk = min(budget // 64, nc)
    B = kk * 64
    fill_k = torch.full((Hkv, B + Td, d), 7.0, dtype=torch.bfloat16, device="cuda")
    fill_v = torch.full_like(fill_k, -7.0)
    fill_k[:, B:] = k[:, N:N + Td]
    fill_v[:, B:] = v[:, N:N + Td]
    parent = list(range(-1, Td - 1))
    mask = dev_mask(parent)
    ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(Td, Hq, Hkv, d, B)), dtype=torch.uint8, device="cuda")
    scale = 1 / math.sqrt(d)

    sel = torch.full((Hkv, kk), -1, dtype=torch.int32, device="cuda")
    plen = torch.full((Hkv,), -1, dtype=torch.int32, device="cuda")
    kp, vp = fill_k.clone(), fill_v.clone()
    out = torch.empty((Td, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Td, Hq), dtype=torch.float32, device="cuda")
    ts.ts_select_gather_tree_attn(scores, q, k, v, N, budget, sel, kp, vp, mask, out, part_len=plen, lse=lse,
                                  workspace=ws, sink_chunks=sink, recent_chunks=recent, scale=scale)
    sel2 = torch.empty_like(sel)
    plen2 = torch.empty_like(plen)
    kp2, vp2 = fill_k.clone(), fill_v.clone()
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    ts.ts_select_gather(scores, N, budget, k, v, sel2, kp2, vp2, part_len=plen2, sink_chunks=sink,
                        recent_chunks=recent)
    ts.ts_tree_attn_partial(q, kp2, vp2, B, mask, plen2, out2, lse=lse2, workspace=ws, scale=scale)
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK

    rsel = oracle.select(s, budget // 64, sink=sink, recent=recent)
    np.testing.assert_array_equal(sel.cpu().numpy(), rsel)
    last = (rsel == nc - 1).any(axis=1)
    tail = N - (nc - 1) * 64
    np.testing.assert_array_equal(plen.cpu().numpy(), kk * 64 - np.where(last, 64 - tail, 0))
    if nc > kk:
        assert (sel[:, :sink].cpu() == torch.arange(sink, dtype=torch.int32)).all()
        assert (sel[:, kk - recent:].cpu() == torch.arange(nc - recent, nc, dtype=torch.int32)).all()
    assert torch.equal(sel, sel2) and torch.equal(plen, plen2)
    assert torch.equal(kp, kp2) and torch.equal(vp, vp2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    if N <= 102400:
        rk, rl = oracle.gather(rsel, k.cpu(), N, 64, B + Td, fill=fill_k.cpu(), return_len=True)
        assert torch.equal(kp.cpu(), rk)
        ro, rlse = oracle.tree_attn(q.cpu(), kp.cpu(), vp.cpu(), B, parent, scale, prefix_len=rl)
        check_attn(out, lse, ro, rlse, "one-pass select + gather + draft")


@pytest.mark.parametrize("T,Hq,Hkv,N", [(120, 40, 8, 20480), (4, 40, 8, 4100), (30, 32, 8, 5000), (4, 8, 8, 60)])
def test_unmerged_then_merge_equals_one_call(T, Hq, Hkv, N):
    """ts_tree_attn_unmerged, then ts_tree_attn_merge on another stream after
    an event: bit for bit what one ts_tree_attn call produces (tensor-core,
    small-batch and CUDA-core plans, and a one-split plan)."""
    d = 128
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=T + N, device="cuda", value_kind="normal")
    parent = verify_parent(T)
    o1, l1, s1 = run_attn(q, k, v, N, parent, 1 / math.sqrt(d), scores=True)
    out = torch.empty_like(o1)
    lse = torch.empty_like(l1)
    sc = torch.full_like(s1, float("nan"))
    ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N)), dtype=torch.uint8, device="cuda")
    s_main, s_side = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    ts.ts_tree_attn_unmerged(q, k, v, N, dev_mask(parent), out, lse=lse, chunk_scores=sc, workspace=ws,
                             scale=1 / math.sqrt(d), stream=s_main)
    ev.record(s_main)
    s_side.wait_event(ev)
    ts.ts_tree_attn_merge(out, Hkv, N, lse=lse, workspace=ws, stream=s_side)
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK
    assert torch.equal(out, o1) and torch.equal(lse, l1) and torch.equal(sc, s1)


@pytest.mark.parametrize("N_old,N_new", [(4094, 4098), (4096, 4100), (4100, 4100), (0, 37), (20480, 20483),
                                         (130, 135), (63, 64), (102400, 102404)])
def test_rescore_tail_equals_full_scoring(N_old, N_new):
    """Scores after a commit: the untouched chunks keep their old values, the
    touched ones are scored again; bit-exact against scoring all of N_new."""
    Hq, Hkv, d = 40, 8, 128
    q, k, _ = W.make_qkv(1, Hq, Hkv, d, N_new, seed=N_old + N_new, device="cuda")
    nc_old, nc_new = (N_old + 63) // 64, (N_new + 63) // 64
    old = torch.empty((Hkv, max(nc_old, 1)), dtype=torch.float32, device="cuda")
    if N_old:
        ts.ts_score_chunks(q[0], k, N_old, old)
    new = torch.full((Hkv, nc_new), float("nan"), dtype=torch.float32, device="cuda")
    ts.ts_rescore_tail(old if N_old else None, N_old, q[0], k, N_new, new)
    torch.cuda.synchronize()
    want = oracle.score_chunks(q[0].cpu(), k.cpu(), N_new).astype(np.float32)
    np.testing.assert_array_equal(new.cpu().numpy(), want)
    if nc_old == nc_new and N_old:
        ts.ts_rescore_tail(old, N_old, q[0], k, N_new, old)   # in place
        torch.cuda.synchronize()
        np.testing.assert_array_equal(old.cpu().numpy(), want)


@pytest.mark.parametrize("N,sink,recent", [(102400, 1, 4), (4100, 2, 2), (20480, 0, 3), (640, 5, 5)])
def test_select_gather_keeps_sink_and_recent_chunks(N, sink, recent):
    Hq, Hkv, d, budget = 32, 8, 128, 4096
    q, k, v = W.make_qkv(1, Hq, Hkv, d, N, seed=N + sink, device="cuda")
    nc = (N + 63) // 64
    sc = torch.empty((Hkv, nc), dtype=torch.float32, device="cuda")
    ts.ts_score_chunks(q[0], k, N, sc)
    kk = min(budget // 64, nc)
    sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
    plen = torch.empty((Hkv,), dtype=torch.int32, device="cuda")
    kp = torch.zeros((Hkv, kk * 64, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    ts.ts_select_gather(sc, N, budget, k, v, sel, kp, vp, part_len=plen, sink_chunks=sink, recent_chunks=recent)
    torch.cuda.synchronize()
    rsel = oracle.select(sc.cpu().numpy(), budget // 64, sink=sink, recent=recent)
    np.testing.assert_array_equal(sel.cpu().numpy(), rsel)
    rk, rl = oracle.gather(rsel, k.cpu(), N, 64, kk * 64, return_len=True)
    assert torch.equal(kp.cpu(), rk)
    np.testing.assert_array_equal(plen.cpu().numpy(), rl)
    if nc > kk:
        assert (sel[:, :sink].cpu() == torch.arange(sink, dtype=torch.int32)).all()
        assert (sel[:, kk - recent:].cpu() == torch.arange(nc - recent, nc, dtype=torch.int32)).all()


@pytest.mark.parametrize("nc", [1, 63, 5000, 16384])
@pytest.mark.parametrize("kind", ["normal", "ties", "constant"])
def test_select_chunks_sizes_and_ties(nc, kind):
    """The selection alone up to the largest chunk count, budgets from one
    chunk to all of them, with many equal scores: bit-exact indices and
    gathered lengths (lowest indices win ties)."""
    Hkv = 2
    rng = np.random.default_rng(nc)
    if kind == "normal":
        s = rng.standard_normal((Hkv, nc)).astype(np.float32)
    elif kind == "ties":
        s = rng.integers(-2, 3, size=(Hkv, nc)).astype(np.float32)
        s[:, ::3] = -0.0
    else:
        s = np.full((Hkv, nc), 1.5, dtype=np.float32)
    scores = torch.from_numpy(s).cuda()
    N = nc * 64 - 17 if nc > 1 else 5
    for k in sorted({1, 64, 300, 1024, nc}):
        kk = min(k, nc)
        sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
        plen = torch.empty((Hkv,), dtype=torch.int32, device="cuda")
        ts.ts_select_chunks(scores, N, k * 64, sel, part_len=plen)
        torch.cuda.synchronize()
        rsel = oracle.select(s, k)
        np.testing.assert_array_equal(sel.cpu().numpy(), rsel, err_msg=f"k={k}")
        last = (rsel == nc - 1).any(axis=1)
        tail = N - (nc - 1) * 64
        np.testing.assert_array_equal(plen.cpu().numpy(), kk * 64 - np.where(last, 64 - tail, 0))


def test_select_ties_and_signed_zero():
    Hkv, nc = 3, 300
    rng = np.random.default_rng(1)
    s = rng.integers(-3, 4, size=(Hkv, nc)).astype(np.float32)
    s[1, ::2] = -0.0
    s[1, 1::2] = 0.0
    s[2, :] = 5.0
    d = 64
    k = torch.randn((Hkv, nc * 64, d), device="cuda").to(torch.bfloat16)
    v = torch.randn((Hkv, nc * 64, d), device="cuda").to(torch.bfloat16)
    for budget in (64, 64 * 17, 64 * 150, 64 * 300, 64 * 400):
        kk = min(budget // 64, nc)
        sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
        kp = torch.zeros((Hkv, kk * 64, d), dtype=torch.bfloat16, device="cuda")
        ts.ts_select_gather(torch.from_numpy(s).cuda(), nc * 64, budget, k, v, sel, kp, torch.zeros_like(kp))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(sel.cpu().numpy(), oracle.select(s, budget // 64))


def test_draft_attention_over_partial_cache():
    cfg = W.WORKLOADS["llama8b-20k"]
    x = W.make_layer_inputs(cfg, 0, device="cuda")
    N = cfg.N
    sc = torch.empty((cfg.Hkv, cfg.n_chunks), dtype=torch.float32, device="cuda")
    ts.ts_score_chunks(x.q[0], x.k, N, sc)
    B = cfg.k_sel * 64
    sel = torch.empty((cfg.Hkv, cfg.k_sel), dtype=torch.int32, device="cuda")
    kp = torch.zeros((cfg.Hkv, B + 4, cfg.d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    kp[:, B:] = x.k_draft_tail
    vp[:, B:] = x.v_draft_tail
    plen = torch.empty((cfg.Hkv,), dtype=torch.int32, device="cuda")
    ts.ts_select_gather(sc, N, cfg.budget, x.k, x.v, sel, kp, vp, part_len=plen)
    assert (plen.cpu() == B).all()
    parent = [-1, 0, 1, 2]
    out, lse, _ = run_attn(x.q_draft, kp, vp, B, parent, cfg.scale)
    rsel = oracle.select(sc.cpu().numpy(), cfg.k_sel)
    rkp = oracle.gather(rsel, x.k.cpu(), N, 64, B + 4, fill=kp.cpu())
    rvp = oracle.gather(rsel, x.v.cpu(), N, 64, B + 4, fill=vp.cpu())
    ro, rl = oracle.tree_attn(x.q_draft.cpu(), rkp, rvp, B, parent, cfg.scale)
    check_attn(out, lse, ro, rl, "draft")


def test_budget_covering_cache_gives_full_attention_bitwise():
    """Budget >= N: the partial cache is the full cache and draft attention
    over it equals attention over the full cache bit for bit."""
    Hq, Hkv, d, N, T = 32, 8, 128, 4096, 4
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=77, device="cuda")
    sc = torch.empty((Hkv, N // 64), dtype=torch.float32, device="cuda")
    ts.ts_score_chunks(q[0], k, N, sc)
    sel = torch.empty((Hkv, N // 64), dtype=torch.int32, device="cuda")
    kp = torch.zeros((Hkv, N + T, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    kp[:, N:] = k[:, N:N + T]
    vp[:, N:] = v[:, N:N + T]
    ts.ts_select_gather(sc, N, 8192, k, v, sel, kp, vp)
    parent = [-1, 0, 1, 2]
    o1, l1, _ = run_attn(q, k, v, N, parent, 1 / math.sqrt(d))
    o2, l2, _ = run_attn(q, kp, vp, N, parent, 1 / math.sqrt(d))
    assert torch.equal(sel.cpu(), torch.arange(N // 64, dtype=torch.int32).repeat(Hkv, 1))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_non_default_stream():
    T, Hq, Hkv, d, N = 40, 4, 1, 64, 999
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=3, device="cuda")
    s = torch.cuda.Stream()
    parent = W.tree_parents([1, 3, 3, 3])
    with torch.cuda.stream(s):
        out, lse, _ = run_attn(q, k, v, N, parent, 0.125, stream=s)
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, 0.125)
    check_attn(out, lse, ro, rl)


# ----------------------------------------------------------------------------- vocab stage
def run_vocab(logits, history, parent, draft, anchor, theta=1.2, min_p=0.1, temp=1.0):
    T = logits.shape[0]
    target = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    kept = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    result = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    ts.ts_penalty_minp_verify(logits, history, theta, min_p, temp, draft, parent, anchor, target, kept, result,
                              path)
    torch.cuda.synchronize()
    return target.cpu().numpy(), kept.cpu().numpy(), result.cpu().numpy(), path.cpu().numpy()


@pytest.mark.parametrize("V,W_,flip,seed", [(152064, 1024, 0.25, 0), (152064, 1024, 0.0, 1), (1000, 50, 0.5, 2),
                                            (33, 5, 0.0, 3), (152064, 0, 0.0, 4), (163840, 2048, 0.3, 5)])
def test_vocab_stage_bit_exact(V, W_, flip, seed):
    parent = W.verify_parents()
    vi = W.make_vocab_inputs(parent, V, W_, seed=seed, device="cuda", flip_rows=flip)
    t, kp, r, p = run_vocab(vi.logits, vi.history, vi.parent, vi.draft, vi.anchor)
    rt, rk = oracle.penalty_minp(vi.logits.cpu().numpy(), vi.history.cpu().numpy(), 1.2, 0.1, 1.0)
    np.testing.assert_array_equal(t, rt)
    np.testing.assert_array_equal(kp, rk)
    rr, rp = oracle.accept(vi.draft.cpu().numpy(), parent, rt, vi.anchor)
    np.testing.assert_array_equal(r, rr)
    np.testing.assert_array_equal(p, rp)


@pytest.mark.parametrize("theta,min_p,temp", [(1.0, 0.1, 1.0), (1.2, 0.0, 1.0), (1.2, 1.0, 1.0), (1.5, 0.05, 0.7),
                                              (1.2, 0.1, 2.0)])
def test_vocab_parameters(theta, min_p, temp):
    parent = W.verify_parents()
    vi = W.make_vocab_inputs(parent, 5000, 300, seed=9, device="cuda", flip_rows=0.3)
    t, kp, r, p = run_vocab(vi.logits, vi.history, vi.parent, vi.draft, vi.anchor, theta, min_p, temp)
    rt, rk = oracle.penalty_minp(vi.logits.cpu().numpy(), vi.history.cpu().numpy(), theta, min_p, temp)
    np.testing.assert_array_equal(t, rt)
    np.testing.assert_array_equal(kp, rk)
    rr, rp = oracle.accept(vi.draft.cpu().numpy(), parent, rt, vi.anchor)
    np.testing.assert_array_equal(r, rr)


def test_vocab_hand_examples(golden_dir):
    import os
    from tests.test_oracle_pins import _nums, _parse
    for name, lg, hist, theta, mp, temp, final, tgt, kept in _parse(os.path.join(golden_dir, "penalty_minp_hand.txt")):
        logits = torch.tensor([_nums(lg, float)], dtype=torch.float32, device="cuda")
        h = torch.tensor(_nums(hist, int), dtype=torch.int32, device="cuda")
        one = torch.tensor([-1], dtype=torch.int32, device="cuda")
        t, k, _, _ = run_vocab(logits, h if h.numel() else None, one, torch.tensor([0], dtype=torch.int32, device="cuda"),
                               0, float(theta), float(mp), float(temp))
        assert t[0] == int(tgt) and k[0] == int(kept), name


def test_accept_hand_examples(golden_dir):
    import os
    from tests.test_oracle_pins import _nums, _parse
    for name, par, dr, tg, anc, res, path in _parse(os.path.join(golden_dir, "accept_hand.txt")):
        T = len(_nums(par, int))
        # logits whose greedy tokens are the example's targets
        V = 16
        logits = torch.zeros((T, V), dtype=torch.float32)
        for i, x in enumerate(_nums(tg, int)):
            logits[i, x] = 5.0
        _, _, r, p = run_vocab(logits.cuda(), None, torch.tensor(_nums(par, int), dtype=torch.int32, device="cuda"),
                               torch.tensor(_nums(dr, int), dtype=torch.int32, device="cuda"), int(anc))
        L, best, bonus = _nums(res, int)
        assert (r[0], r[1], r[2], r[3]) == (L, best, bonus, 0), name
        want = _nums(path, int)
        assert p[:len(want)].tolist() == want and all(x == -1 for x in p[len(want):]), name


def test_vocab_data_errors_reported_not_trapped():
    parent = W.verify_parents()
    vi = W.make_vocab_inputs(parent, 1000, 20, seed=4, device="cuda")
    bad_hist = vi.history.clone()
    bad_hist[3] = 1000
    _, _, r, _ = run_vocab(vi.logits, bad_hist, vi.parent, vi.draft, vi.anchor)
    assert r[3] == ts.TS_ERR_DATA
    bad_parent = vi.parent.clone()
    bad_parent[5] = 7
    _, _, r, p = run_vocab(vi.logits, vi.history, bad_parent, vi.draft, vi.anchor)
    assert r[3] == ts.TS_ERR_DATA and r[0] == 0 and (p == -1).all()
    # the context is still usable
    t, _, r, _ = run_vocab(vi.logits, vi.history, vi.parent, vi.draft, vi.anchor)
    assert r[3] == 0


@pytest.mark.parametrize("Hq,Hkv,N", [(40, 8, 20480), (4, 4, 40960), (32, 8, 4000), (40, 8, 1000)])
def test_tree_attn_without_lse_matches_oracle(Hq, Hkv, N):
    """Without a log-sum-exp output the tensor-core kernel skips the sum of the
    unrounded weights and the split merge weighs the ranges by the rounded sums;
    O stays within the bars (pair and single streams, split and direct)."""
    T, d = 120, 128
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=7 * N + Hq, device="cuda")
    parent = W.verify_parents()
    scale = 1 / math.sqrt(d)
    out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N)), dtype=torch.uint8, device="cuda")
    ts.ts_tree_attn(q, k, v, N, dev_mask(parent), out, workspace=ws, scale=scale)
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK
    o_lse, _, _ = run_attn(q, k, v, N, parent, scale)
    assert (out.float() - o_lse.float()).abs().max().item() <= MAX_ABS
    rows = np.unique(np.concatenate([np.arange(Hq), np.arange(T * Hq - Hq, T * Hq),
                                     np.random.default_rng(N + 1).integers(0, T * Hq, 40)])).astype(np.int32)
    ro, _ = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, scale, rows=rows)
    o = out.reshape(-1, d)[rows].float().cpu().double().numpy()
    assert np.abs(o - ro).max() <= MAX_ABS
    assert np.linalg.norm(o - ro) / np.linalg.norm(ro) <= REL_L2


@pytest.mark.parametrize("Hq,Hkv,N", [(4, 4, 102400), (10, 2, 40960)])
def test_fused_scores_leave_attention_bitwise_unchanged(Hq, Hkv, N):
    """The fused chunk scoring only reads S: outputs with and without it must be
    bit-identical, on long KV ranges where warps drift apart (one-tile streams
    with double-buffered S, and two-tile plus one-tile streams for group 5)."""
    T, d = 120, 128
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=N + Hq, device="cuda")
    parent = W.verify_parents()
    scale = 1 / math.sqrt(d)
    o1, l1, _ = run_attn(q, k, v, N, parent, scale)
    for score_row in (0, 64, T - 1):
        o2, l2, sc = run_attn(q, k, v, N, parent, scale, scores=True, score_row=score_row)
        assert torch.equal(o1, o2) and torch.equal(l1, l2), f"score_row {score_row}"
    rows = np.unique(np.concatenate([np.arange(Hq), np.arange(T * Hq - Hq, T * Hq),
                                     np.random.default_rng(N).integers(0, T * Hq, 24)])).astype(np.int32)
    ro, rl = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, scale, rows=rows)
    o = o1.reshape(-1, d)[rows].float().cpu().double().numpy()
    assert np.abs(o - ro).max() <= MAX_ABS
    assert np.abs(l1.reshape(-1)[rows].cpu().double().numpy() - rl).max() <= LSE_ABS


# --------------------------------------------------------------------------
# commit of the accepted path (next row: the step after verification)
# --------------------------------------------------------------------------
def _ancestors(parent, row):
    out = []
    while row >= 0:
        out.append(int(row))
        row = parent[row]
    return out[::-1]


@pytest.mark.parametrize("Hkv,d,N,T,seed", [(8, 128, 20480, 120, 0), (2, 64, 4096, 40, 1), (32, 128, 1000, 64, 2),
                                            (1, 128, 0, 1, 3), (8, 128, 2048, 900, 4), (2, 64, 100, 300, 5)])
def test_commit_path_bit_exact(Hkv, d, N, T, seed):
    """Includes a 900-row batch of the [1,9,9,9] tree and a 300-row chain whose
    accepted path (300 rows) is moved in several shared-memory rounds."""
    parent = verify_parent(T) if T <= 120 else (W.verify_parents((1, 9, 9, 9), 20) if T == 900
                                                else [-1] + list(range(T - 1)))
    _, k, v = W.make_qkv(T, Hkv, Hkv, d, N, seed=500 + seed, device="cuda", value_kind="normal", ld_extra=3)
    rng = np.random.default_rng(seed)
    for best in list(rng.choice(T, size=min(T, 4), replace=False)) + [T - 1]:
        path = _ancestors(parent, int(best))
        L = len(path)
        pth = np.full(T, -1, dtype=np.int32)
        pth[:L] = path
        res = np.array([L, best, 0, 0], dtype=np.int32)
        kr, vr, st = oracle.commit_path(k.cpu(), v.cpu(), N, res, pth)
        kg, vg = k.clone(), v.clone()
        rd = torch.from_numpy(res).cuda()
        ts.ts_commit_path(kg, vg, N, rd, torch.from_numpy(pth).cuda())
        torch.cuda.synchronize()
        assert st == 0 and int(rd[3]) == 0
        assert torch.equal(kg.cpu(), kr) and torch.equal(vg.cpu(), vr)


def test_commit_path_from_the_vocab_stage_on_device():
    """Verify then commit with no host round trip: L and the path come from the
    vocab stage's device outputs."""
    parent = W.verify_parents()
    T, Hkv, d, N = len(parent), 8, 128, 4096
    vi = W.make_vocab_inputs(parent, 152064, 1024, seed=11, device="cuda", flip_rows=0.25)
    target = torch.empty((T,), dtype=torch.int32, device="cuda")
    kept = torch.empty_like(target)
    result = torch.empty((4,), dtype=torch.int32, device="cuda")
    path = torch.empty_like(target)
    _, k, v = W.make_qkv(T, Hkv, Hkv, d, N, seed=12, device="cuda", value_kind="normal")
    kg, vg = k.clone(), v.clone()
    ts.ts_penalty_minp_verify(vi.logits, vi.history, 1.2, 0.1, 1.0, vi.draft, vi.parent, vi.anchor, target, kept,
                              result, path)
    ts.ts_commit_path(kg, vg, N, result, path)
    torch.cuda.synchronize()
    res, pth = result.cpu().numpy(), path.cpu().numpy()
    assert res[0] > 0 and res[3] == 0
    kr, vr, st = oracle.commit_path(k.cpu(), v.cpu(), N, res, pth)
    assert st == 0 and torch.equal(kg.cpu(), kr) and torch.equal(vg.cpu(), vr)


def test_commit_path_data_errors_reported_not_trapped():
    T, Hkv, d, N = 16, 2, 128, 256
    _, k, v = W.make_qkv(T, Hkv, Hkv, d, N, seed=13, device="cuda", value_kind="normal")
    for res, pth in (([3, 0, 0, 0], [0, 4, 4]), ([2, 0, 0, 0], [1, T]), ([T + 1, 0, 0, 0], list(range(T))),
                     ([0, -1, 0, 0], [])):
        p = np.full(T, -1, dtype=np.int32)
        p[:len(pth)] = pth
        kg, vg = k.clone(), v.clone()
        rd = torch.tensor(res, dtype=torch.int32, device="cuda")
        ts.ts_commit_path(kg, vg, N, rd, torch.from_numpy(p).cuda())
        torch.cuda.synchronize()
        assert int(rd[3]) == (0 if res[0] == 0 else 5)
        assert torch.equal(kg, k) and torch.equal(vg, v)
    assert ts.ts_device_error(True) == 0


# --------------------------------------------------------------------------
# min-p sampled targets (next row): Gumbel-max with Philox4x64-10
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V,W_,flip,seed,min_p,temp", [(152064, 1024, 0.25, 0, 0.1, 1.0),
                                                       (152064, 1024, 0.0, 1, 0.02, 1.0),
                                                       (1000, 50, 0.5, 2, 0.0, 1.0),
                                                       (33, 5, 0.0, 3, 0.3, 0.7),
                                                       (163840, 2048, 0.3, 5, 0.1, 2.0)])
def test_sampled_vocab_stage_bit_exact(V, W_, flip, seed, min_p, temp):
    """Sampled targets, kept counts, accepted length and path agree bit for bit
    with the oracle's Gumbel-max draw from the same Philox stream."""
    parent = W.verify_parents()
    T = len(parent)
    vi = W.make_vocab_inputs(parent, V, W_, seed=seed, device="cuda", flip_rows=flip)
    target = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    kept = torch.full_like(target, -7)
    result = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    path = torch.full_like(target, -7)
    ts.ts_penalty_minp_sample_verify(vi.logits, vi.history, 1.2, min_p, temp, 77 + seed, 5, vi.draft, vi.parent,
                                     vi.anchor, target, kept, result, path)
    torch.cuda.synchronize()
    _, rk, pen = oracle.penalty_minp(vi.logits.cpu().numpy(), vi.history.cpu().numpy(), 1.2, min_p, temp,
                                     return_logits=True)
    rs = oracle.sample(pen, min_p, 77 + seed, 5)
    np.testing.assert_array_equal(target.cpu().numpy(), rs)
    np.testing.assert_array_equal(kept.cpu().numpy(), rk)
    rr, rp = oracle.accept(vi.draft.cpu().numpy(), parent, rs, vi.anchor, seed=77 + seed, offset=5)
    np.testing.assert_array_equal(result.cpu().numpy(), rr)
    np.testing.assert_array_equal(path.cpu().numpy(), rp)


def test_sampled_stage_draws_among_the_longest_paths():
    """Rows tie for the longest accepted path (every chain repeats a path of the
    sampled targets); the kept row is the oracle's seeded uniform draw, offset
    by offset, and over many offsets every tied row is drawn."""
    parent = W.verify_parents()
    T = len(parent)
    V = 64
    vi = W.make_vocab_inputs(parent, V, 8, seed=21, device="cuda")
    logits = torch.full((T, V), -20.0, dtype=torch.float32)
    logits[:, 7] = 5.0   # every sampled target is token 7 (min-p keeps only it)
    draft = torch.full((T,), 7, dtype=torch.int32)
    draft[40::4] = 3     # chain heads match the anchor 3, the rest match target 7
    for c in range(0, 20, 3):
        draft[40 + 4 * c + 2] = 1   # some chains break at depth 3
    target = torch.empty((T,), dtype=torch.int32, device="cuda")
    kept = torch.empty_like(target)
    result = torch.empty((4,), dtype=torch.int32, device="cuda")
    path = torch.empty_like(target)
    seen = set()
    hist = torch.zeros(1, dtype=torch.int32, device="cuda")
    for off in range(40):
        ts.ts_penalty_minp_sample_verify(logits.cuda(), hist, 1.2, 0.1, 1.0, 9, off, draft.cuda(), vi.parent, 3,
                                         target, kept, result, path)
        torch.cuda.synchronize()
        rr, rp = oracle.accept(draft.numpy(), parent, np.full(T, 7, np.int32), 3, seed=9, offset=off)
        np.testing.assert_array_equal(result.cpu().numpy(), rr)
        np.testing.assert_array_equal(path.cpu().numpy(), rp)
        assert rr[0] == 4
        seen.add(int(rr[1]))
    assert len(seen) >= 8


# --------------------------------------------------------------------------
# path-aware penalty window (each row's window ends with the drafts on its path)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V,W_,sample,branching", [(152064, 1024, False, (1, 3, 3, 3)), (5000, 40, False, (1, 3, 3, 3)),
                                                   (4096, 8, True, (3, 3, 3, 3)), (1000, 3, False, (1, 9, 9, 9))])
def test_path_window_vocab_stage_bit_exact(V, W_, sample, branching):
    parent = W.verify_parents(branching)
    T = len(parent)
    vi = W.make_vocab_inputs(parent, V, W_, seed=V + W_, device="cuda", flip_rows=0.3)
    # drafts that sit inside the windows of their descendants: raise their logits
    lg = vi.logits.clone()
    dr = vi.draft.cpu().numpy()
    for i, p in enumerate(parent):
        if p >= 0:
            lg[i, int(dr[p])] = lg[i].max() + 0.7
    target = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    kept = torch.full_like(target, -7)
    result = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    path = torch.full_like(target, -7)
    flags = ts.TS_VOCAB_PATH_WINDOW | (ts.TS_VOCAB_SAMPLE if sample else 0)
    ts.ts_vocab_verify(lg, vi.history, 1.2, 0.1, 1.0, flags, 31, 2, vi.draft, vi.parent, vi.anchor, target, kept,
                       result, path)
    torch.cuda.synchronize()
    rt, rk, pen = oracle.penalty_minp(lg.cpu().numpy(), vi.history.cpu().numpy(), 1.2, 0.1, 1.0, return_logits=True,
                                      path_parent=parent, path_draft=dr)
    if sample:
        rt = oracle.sample(pen, 0.1, 31, 2)
    np.testing.assert_array_equal(target.cpu().numpy(), rt)
    np.testing.assert_array_equal(kept.cpu().numpy(), rk)
    rr, rp = oracle.accept(dr, parent, rt, vi.anchor, seed=31 if sample else None, offset=2)
    np.testing.assert_array_equal(result.cpu().numpy(), rr)
    np.testing.assert_array_equal(path.cpu().numpy(), rp)
    # the path-aware window changes some targets against the shared window
    if not sample:
        t0, _ = oracle.penalty_minp(lg.cpu().numpy(), vi.history.cpu().numpy(), 1.2, 0.1, 1.0)
        assert (t0 != rt).any()
