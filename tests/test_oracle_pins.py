"""Pins of the fp64 oracle to things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong index, a transposed operand, a wrong mask bit, a wrong tie rule) fails:
  * attention: torch's scaled_dot_product_attention in fp64 with a mask built
    by boolean transitive closure (a different algorithm from the oracle's
    parent walk); closed forms (zero query -> mean of visible values, constant
    values, a lone visible key); the chain-is-causal and all-roots-is-decode
    special cases; invariance under permuting prefix tokens and under a
    topological relabelling of the batch;
  * chunk scores: exact int64 brute force by a different association
    (sum over tokens of q.k instead of q . sum k), and a closed form;
  * selection: numpy lexsort, plus hand-made tie and signed-zero cases;
  * gather: identity when the budget covers the cache;
  * penalty/min-p and acceptance: hand-worked examples in tests/golden, plus
    min-p checked against a scipy softmax, and acceptance against path
    enumeration with networkx.
"""
import math
import os

import networkx as nx
import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch
import torch.nn.functional as F

import oracle
from long_context_attention_tree_b300 import workloads as W


# ---------------------------------------------------------------- helpers
def closure_mask(parent):
    """Ancestor-or-self relation by repeated boolean matrix products."""
    T = len(parent)
    A = np.zeros((T, T), dtype=bool)
    for i, p in enumerate(parent):
        if p >= 0:
            A[i, p] = True
    R = np.eye(T, dtype=bool) | A
    while True:
        R2 = R | ((R.astype(np.int64) @ R.astype(np.int64)) > 0)
        if (R2 == R).all():
            return R
        R = R2


def sdpa_reference(q, k, v, N, vis, scale):
    """torch SDPA in fp64 with an explicit boolean mask (GQA by repeat)."""
    T, Hq, d = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    L = N + T
    kk = k[:, :L].double().repeat_interleave(G, dim=0)  # [Hq][L][d]
    vv = v[:, :L].double().repeat_interleave(G, dim=0)
    qq = q.double().permute(1, 0, 2)  # [Hq][T][d]
    mask = torch.zeros((T, L), dtype=torch.bool)
    mask[:, :N] = True
    mask[:, N:] = torch.from_numpy(vis)
    out = F.scaled_dot_product_attention(qq.unsqueeze(0), kk.unsqueeze(0), vv.unsqueeze(0),
                                         attn_mask=mask, scale=scale)[0]
    scores = torch.einsum("htd,hld->htl", qq, kk) * scale
    scores = scores.masked_fill(~mask, -math.inf)
    lse = torch.from_numpy(scipy.special.logsumexp(scores.numpy(), axis=-1))
    return out.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


def run_oracle(q, k, v, N, parent, scale):
    return oracle.tree_attn(q, k, v, N, parent, scale)


SHAPES = [
    # (T, Hq, Hkv, d, N, value_kind)
    (40, 4, 1, 64, 200, "int"),
    (13, 8, 2, 64, 77, "normal"),
    (7, 6, 3, 128, 0, "normal"),
    (20, 5, 5, 32, 65, "int"),
]


# ---------------------------------------------------------------- visibility
@pytest.mark.parametrize("parent", [
    W.tree_parents([1, 3, 3, 3]),
    W.verify_parents(),
    W.tree_parents([3, 3, 3]),
    W.chain_parents(5, 4),
    [-1] * 9,
])
def test_visible_matches_networkx_ancestors(parent):
    vis = oracle.visible(parent)
    g = nx.DiGraph()
    g.add_nodes_from(range(len(parent)))
    g.add_edges_from((p, i) for i, p in enumerate(parent) if p >= 0)
    for i in range(len(parent)):
        want = nx.ancestors(g, i) | {i}
        assert set(np.nonzero(vis[i])[0].tolist()) == want


def test_visible_rejects_bad_parents():
    with pytest.raises(ValueError):
        oracle.visible([-1, 1])      # parent[i] >= i
    with pytest.raises(ValueError):
        oracle.visible([-1, -2])     # below -1


def test_tree_shapes_from_ablation_table():
    assert len(W.tree_parents([1, 3, 3, 3])) == 40
    assert len(W.tree_parents([3, 3, 3, 3])) == 120
    assert len(W.tree_parents([1, 9, 9, 9])) == 1 + 9 + 81 + 729
    assert W.tree_parents([1, 3, 3, 3])[:13] == [-1, 0, 0, 0, 1, 1, 1, 2, 2, 2, 3, 3, 3]
    assert len(W.verify_parents()) == 120


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("tree", ["verify", "chain", "roots"])
def test_attention_matches_torch_sdpa(shape, tree):
    T, Hq, Hkv, d, N, kind = shape
    if tree == "verify":
        parent = (W.tree_parents([1, 3, 3, 3]) + W.chain_parents(20, 4, offset=40))[:T]
        parent = [p if p < T else -1 for p in parent]
    elif tree == "chain":
        parent = [-1] + list(range(T - 1))
    else:
        parent = [-1] * T
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=7 + T + N, value_kind=kind, ld_extra=3)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_oracle(q, k, v, N, parent, scale)
    ro, rlse = sdpa_reference(q, k, v, N, closure_mask(parent), scale)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lse, rlse, rtol=0, atol=1e-10)


def test_chain_equals_causal_attention():
    """A chain batch is plain causal attention over prefix + batch."""
    T, Hq, Hkv, d, N = 9, 4, 2, 64, 50
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=3, value_kind="normal")
    o, _ = run_oracle(q, k, v, N, [-1] + list(range(T - 1)), 0.125)
    G = Hq // Hkv
    kk = k.double().repeat_interleave(G, 0)
    vv = v.double().repeat_interleave(G, 0)
    # causal over the full N+T sequence, keep the last T query positions
    qfull = torch.zeros((Hq, N + T, d), dtype=torch.float64)
    qfull[:, N:] = q.double().permute(1, 0, 2)
    ref = F.scaled_dot_product_attention(qfull[None], kk[None], vv[None], is_causal=True, scale=0.125)[0, :, N:]
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), atol=1e-10, rtol=0)


def test_zero_query_gives_mean_of_visible_values():
    T, Hq, Hkv, d, N = 40, 4, 1, 64, 33
    parent = W.tree_parents([1, 3, 3, 3])
    _, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=11, value_kind="normal")
    q = torch.zeros((T, Hq, d), dtype=torch.bfloat16)
    o, lse = run_oracle(q, k, v, N, parent, 0.125)
    vis = closure_mask(parent)
    vd = v.double().numpy()
    for t in range(T):
        idx = list(range(N)) + [N + u for u in range(T) if vis[t, u]]
        want = vd[0, idx].mean(axis=0)
        for h in range(Hq):
            np.testing.assert_allclose(o[t, h], want, atol=1e-12)
            assert abs(lse[t, h] - math.log(len(idx))) < 1e-12


def test_constant_values_and_lone_key():
    T, Hq, Hkv, d = 6, 2, 1, 64
    q, k, _ = W.make_qkv(T, Hq, Hkv, d, 0, seed=5, value_kind="normal")
    v = torch.full((Hkv, T, d), 1.5, dtype=torch.bfloat16)
    o, _ = run_oracle(q, k, v, 0, [-1, 0, 1, 2, 3, 4], 0.125)
    np.testing.assert_allclose(o, 1.5, atol=1e-12)
    # N = 0 and every row a root: each row sees only its own key
    v2 = torch.randn((Hkv, T, d)).to(torch.bfloat16)
    o2, lse2 = run_oracle(q, k, v2, 0, [-1] * T, 0.125)
    for t in range(T):
        for h in range(Hq):
            np.testing.assert_array_equal(o2[t, h], v2[0, t].double().numpy())
            s = 0.125 * float((q[t, h].double() * k[0, t].double()).sum())
            assert abs(lse2[t, h] - s) < 1e-12


def test_prefix_permutation_invariance():
    T, Hq, Hkv, d, N = 40, 4, 2, 64, 130
    parent = W.tree_parents([1, 3, 3, 3])
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=21, value_kind="normal")
    o, lse = run_oracle(q, k, v, N, parent, 0.125)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(1))
    k2, v2 = k.clone(), v.clone()
    k2[:, :N] = k[:, perm]
    v2[:, :N] = v[:, perm]
    o2, lse2 = run_oracle(q, k2, v2, N, parent, 0.125)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)


def test_topological_relabel_permutes_outputs():
    """Listing the batch in DFS order instead of BFS permutes the output rows."""
    parent = W.tree_parents([1, 3, 3])
    T = len(parent)
    kids = {}
    for i, p in enumerate(parent):
        kids.setdefault(p, []).append(i)
    order = []

    def dfs(n):
        order.append(n)
        for c in kids.get(n, []):
            dfs(c)
    dfs(0)
    new_of = {old: new for new, old in enumerate(order)}
    parent2 = [-1 if parent[old] < 0 else new_of[parent[old]] for old in order]
    Hq, Hkv, d, N = 4, 2, 64, 40
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=9, value_kind="normal")
    o, _ = run_oracle(q, k, v, N, parent, 0.125)
    idx = torch.tensor(order)
    q2 = q[idx]
    k2 = torch.cat([k[:, :N], k[:, N:N + T][:, idx]], dim=1)
    v2 = torch.cat([v[:, :N], v[:, N:N + T][:, idx]], dim=1)
    o2, _ = run_oracle(q2, k2, v2, N, parent2, 0.125)
    np.testing.assert_allclose(o2, o[order], atol=1e-12)


def test_sampled_rows_equal_full():
    T, Hq, Hkv, d, N = 40, 4, 2, 64, 100
    parent = W.tree_parents([1, 3, 3, 3])
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=2)
    o, lse = oracle.tree_attn(q, k, v, N, parent, 0.125)
    rows = np.array([0, 5, 77, 159])
    os_, ls_ = oracle.tree_attn(q, k, v, N, parent, 0.125, rows=rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, d)[rows])
    np.testing.assert_array_equal(ls_, lse.reshape(-1)[rows])


@pytest.mark.parametrize("prefix_len", [[0, 5, 77], [77, 77, 77], [64, 1, 30]])
def test_ragged_prefix_matches_sdpa_per_head(prefix_len):
    """KV head g sees prefix rows [0, prefix_len[g]) only: torch SDPA per KV head
    with a mask that hides the rest of the prefix."""
    T, Hq, Hkv, d, N = 4, 6, 3, 64, 77
    parent = [-1, 0, 1, 2]
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=31, value_kind="normal")
    o, lse = oracle.tree_attn(q, k, v, N, parent, 0.125, prefix_len=prefix_len)
    G = Hq // Hkv
    vis = closure_mask(parent)
    for g in range(Hkv):
        mask = torch.zeros((T, N + T), dtype=torch.bool)
        mask[:, :prefix_len[g]] = True
        mask[:, N:] = torch.from_numpy(vis)
        qq = q[:, g * G:(g + 1) * G].double().permute(1, 0, 2)
        kk = k[g:g + 1, :N + T].double().expand(G, -1, -1)
        vv = v[g:g + 1, :N + T].double().expand(G, -1, -1)
        ref = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], attn_mask=mask, scale=0.125)[0]
        np.testing.assert_allclose(o[:, g * G:(g + 1) * G], ref.permute(1, 0, 2).numpy(), atol=1e-10, rtol=0)
        sc = (torch.einsum("htd,hld->htl", qq, kk) * 0.125).masked_fill(~mask, -math.inf).numpy()
        np.testing.assert_allclose(lse[:, g * G:(g + 1) * G], scipy.special.logsumexp(sc, axis=-1).T,
                                   atol=1e-10, rtol=0)


def test_ragged_prefix_rejects_out_of_range():
    q, k, v = W.make_qkv(1, 2, 2, 64, 10, seed=1)
    with pytest.raises(ValueError):
        oracle.tree_attn(q, k, v, 10, [-1], 0.125, prefix_len=[3, 11])


# ---------------------------------------------------------------- chunk scores
@pytest.mark.parametrize("N", [1, 63, 64, 65, 300])
def test_chunk_scores_int64_brute_force(N):
    Hq, Hkv, d = 8, 2, 64
    q, k, _ = W.make_qkv(1, Hq, Hkv, d, N, seed=N)
    s = oracle.score_chunks(q[0], k, N, 64)
    qi = q[0].to(torch.int64).numpy()
    ki = k[:, :N].to(torch.int64).numpy()
    G = Hq // Hkv
    nc = (N + 63) // 64
    for g in range(Hkv):
        per_tok = qi[g * G:(g + 1) * G] @ ki[g].T       # [G][N] exact q.k per token
        for c in range(nc):
            want = per_tok[:, c * 64:(c + 1) * 64].sum(axis=1).max()
            assert s[g, c] == float(want)


def test_chunk_scores_closed_form_ones():
    Hq, Hkv, d, N = 4, 1, 64, 100
    q, _, _ = W.make_qkv(1, Hq, Hkv, d, 0, seed=4)
    k = torch.ones((Hkv, N, d), dtype=torch.bfloat16)
    s = oracle.score_chunks(q[0], k, N, 64)
    qsum = q[0].double().sum(dim=1).max().item()
    assert s[0, 0] == 64 * qsum and s[0, 1] == 36 * qsum


# ---------------------------------------------------------------- selection
def test_select_matches_lexsort():
    rng = np.random.default_rng(0)
    s = rng.integers(-5, 6, size=(3, 300)).astype(np.float32)  # many ties
    sel = oracle.select(s, 64)
    for g in range(3):
        order = np.lexsort((np.arange(300), -s[g]))[:64]
        np.testing.assert_array_equal(sel[g], np.sort(order))


def test_select_hand_cases():
    s = np.array([[5, 5, 3, 5, 1]], dtype=np.float32)
    np.testing.assert_array_equal(oracle.select(s, 2)[0], [0, 1])
    np.testing.assert_array_equal(oracle.select(s, 3)[0], [0, 1, 3])
    np.testing.assert_array_equal(oracle.select(s, 4)[0], [0, 1, 2, 3])
    np.testing.assert_array_equal(oracle.select(s, 9)[0], [0, 1, 2, 3, 4])
    z = np.array([[-0.0, 0.0, -1.0]], dtype=np.float32)   # -0 equals +0: lower index wins
    np.testing.assert_array_equal(oracle.select(z, 1)[0], [0])
    z2 = np.array([[0.0, -0.0, 2.0]], dtype=np.float32)
    np.testing.assert_array_equal(oracle.select(z2, 2)[0], [0, 2])


def test_select_keeps_sink_and_recent_chunks():
    """Always-kept first / last chunks: equal to a lexsort in which those
    chunks score +inf; and a hand case."""
    rng = np.random.default_rng(7)
    s = rng.integers(-5, 6, size=(3, 200)).astype(np.float32)
    for sink, recent, k in ((1, 1, 16), (2, 3, 16), (0, 4, 4), (3, 0, 10), (5, 5, 10)):
        sel = oracle.select(s, k, sink=sink, recent=recent)
        for g in range(3):
            f = s[g].astype(np.float64).copy()
            f[:sink] = np.inf
            if recent:
                f[200 - recent:] = np.inf
            order = np.lexsort((np.arange(200), -f))[:k]
            np.testing.assert_array_equal(sel[g], np.sort(order))
    h = np.array([[5, 5, 3, 5, 1]], dtype=np.float32)
    np.testing.assert_array_equal(oracle.select(h, 3, sink=1, recent=1)[0], [0, 1, 4])
    np.testing.assert_array_equal(oracle.select(h, 2, sink=0, recent=2)[0], [3, 4])
    with pytest.raises(ValueError):
        oracle.select(h, 2, sink=2, recent=1)


# ---------------------------------------------------------------- gather
def test_gather_identity_when_budget_covers_cache():
    Hkv, d, N = 2, 64, 192
    _, k, _ = W.make_qkv(1, 2, Hkv, d, N, seed=8)
    sel = np.tile(np.arange(3, dtype=np.int32), (Hkv, 1))
    kp = oracle.gather(sel, k, N, 64, ld_dst=N + 4)
    assert torch.equal(kp[:, :N], k[:, :N])


def test_gather_moves_the_named_chunk():
    Hkv, d, N = 1, 64, 256
    _, k, _ = W.make_qkv(1, 1, Hkv, d, N, seed=12)
    kp = oracle.gather(np.array([[3, 1]], dtype=np.int32), k, N, 64, ld_dst=128)
    assert torch.equal(kp[0, :64], k[0, 192:256]) and torch.equal(kp[0, 64:128], k[0, 64:128])


@pytest.mark.parametrize("N", [4100, 130, 64 * 9])
def test_partial_cache_attention_equals_attention_over_the_selected_tokens(N):
    """A ragged last chunk: the gathered rows [0, part_len[g]) of head g, with the
    draft batch's own rows after the budget, give the same attention as the
    selected token positions indexed straight out of the full cache."""
    Hq, Hkv, d, Td, chunk, kk = 4, 2, 64, 3, 64, 3
    q, k, v = W.make_qkv(Td, Hq, Hkv, d, N, seed=N, value_kind="normal")
    nc = (N + chunk - 1) // chunk
    rng = np.random.default_rng(N)
    sel = np.stack([np.sort(rng.choice(nc, size=kk, replace=False)) for _ in range(Hkv)]).astype(np.int32)
    sel[0, -1] = nc - 1   # head 0 always holds the (possibly short) last chunk
    B = kk * chunk
    kp, plen = oracle.gather(sel, k, N, chunk, B + Td, return_len=True)
    vp = oracle.gather(sel, v, N, chunk, B + Td)
    kp[:, B:] = k[:, N:N + Td]
    vp[:, B:] = v[:, N:N + Td]
    parent = [-1] + list(range(Td - 1))
    o, lse = oracle.tree_attn(q, kp, vp, B, parent, 0.125, prefix_len=plen)
    G = Hq // Hkv
    for g in range(Hkv):
        idx = np.concatenate([np.arange(c * chunk, min((c + 1) * chunk, N)) for c in sel[g]])
        assert plen[g] == idx.size
        for t in range(Td):
            keys = np.concatenate([idx, N + np.arange(t + 1)])
            kk_ = k[g, keys].double()
            vv_ = v[g, keys].double()
            for j in range(G):
                s_ = 0.125 * (kk_ @ q[t, g * G + j].double())
                p_ = torch.softmax(s_, 0)
                np.testing.assert_allclose(o[t, g * G + j], (p_ @ vv_).numpy(), atol=1e-10, rtol=0)
                assert abs(lse[t, g * G + j] - torch.logsumexp(s_, 0).item()) < 1e-10


# ---------------------------------------------------------------- penalty / min-p
def _parse(path):
    rows = []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append([f.strip() for f in line.split("|")])
    return rows


def _nums(s, typ):
    return [] if s.strip() == "-" else [typ(x) for x in s.split()]


def test_penalty_minp_hand_examples(golden_dir):
    rows = _parse(os.path.join(golden_dir, "penalty_minp_hand.txt"))
    assert len(rows) >= 8
    for name, lg, hist, theta, mp, temp, final, tgt, kept in rows:
        logits = np.array([_nums(lg, float)], dtype=np.float32)
        t, kp, pen = oracle.penalty_minp(logits, np.array(_nums(hist, int), dtype=np.int32),
                                         float(theta), float(mp), float(temp), return_logits=True)
        np.testing.assert_array_equal(pen[0], np.array(_nums(final, float), dtype=np.float32), err_msg=name)
        assert t[0] == int(tgt), name
        assert kp[0] == int(kept), name


def test_minp_count_matches_softmax_definition():
    rng = np.random.default_rng(3)
    logits = (rng.standard_normal((6, 5000)) * 3).astype(np.float32)
    hist = rng.integers(0, 5000, size=300).astype(np.int32)
    t, kp, pen = oracle.penalty_minp(logits, hist, 1.2, 0.1, 1.0, return_logits=True)
    p = scipy.special.softmax(pen.astype(np.float64), axis=1)
    for i in range(6):
        ratio = p[i] / p[i].max()
        assert not np.any(np.abs(ratio - np.float32(0.1)) < 1e-9)   # no boundary case
        assert kp[i] == int((ratio >= np.float64(np.float32(0.1))).sum())
        assert t[i] == int(np.argmax(pen[i]))


def _path_window_brute(logits, history, parent, draft, theta, min_p, temp):
    """Each row's window built as an explicit token list, the penalty in numpy fp32."""
    T, V = logits.shape
    W_ = len(history)
    out = logits.astype(np.float32).copy()
    for i in range(T):
        path = []
        j = i
        while j >= 0:
            path.append(int(draft[j]))
            j = parent[j]
        ctx = list(history) + path[::-1]
        win = {t for t in (ctx[-W_:] if W_ else []) if 0 <= t < V}
        for t in win:
            x = out[i, t]
            out[i, t] = x / np.float32(theta) if x > 0 else x * np.float32(theta)
        out[i] = out[i] / np.float32(temp)
    m = out.max(axis=1)
    thr = m.astype(np.float64) + math.log(float(np.float32(min_p)))
    kept = (out.astype(np.float64) >= thr[:, None]).sum(axis=1)
    return out.argmax(axis=1), kept, out


def test_path_window_hand_example():
    """history [0 1 2], W = 3; tree 0 <- {1, 2} with drafts 3, 4, 5: row 0's
    window is {1, 2, 3}, row 1's {2, 3, 4}, row 2's {2, 3, 5}."""
    logits = np.full((3, 6), 1.0, dtype=np.float32)
    t, _, pen = oracle.penalty_minp(logits, np.array([0, 1, 2], np.int32), 2.0, 0.1, 1.0, return_logits=True,
                                    path_parent=[-1, 0, 0], path_draft=[3, 4, 5])
    np.testing.assert_array_equal(pen, np.array([[1, .5, .5, .5, 1, 1], [1, 1, .5, .5, .5, 1],
                                                 [1, 1, .5, .5, 1, .5]], dtype=np.float32))
    np.testing.assert_array_equal(t, [0, 0, 0])


@pytest.mark.parametrize("seed,W_", [(0, 16), (1, 3), (2, 0), (3, 64)])
def test_path_window_matches_explicit_windows(seed, W_):
    rng = np.random.default_rng(seed)
    parent = W.verify_parents((1, 3, 3, 3), 5)
    T, V = len(parent), 40
    logits = (rng.standard_normal((T, V)) * 3).astype(np.float32)
    history = rng.integers(0, V, W_).astype(np.int32)
    draft = rng.integers(0, V, T).astype(np.int32)
    draft[-3] = -1   # an unused n-gram row adds no token
    t, kp, pen = oracle.penalty_minp(logits, history, 1.2, 0.1, 1.0, return_logits=True, path_parent=parent,
                                     path_draft=draft)
    bt, bk, bpen = _path_window_brute(logits, history.tolist(), parent, draft, 1.2, 0.1, 1.0)
    np.testing.assert_array_equal(pen, bpen)
    np.testing.assert_array_equal(t, bt)
    np.testing.assert_array_equal(kp, bk)


def test_penalty_empty_window_is_plain_argmax():
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal((3, 777)) * 3).astype(np.float32)
    t, _ = oracle.penalty_minp(logits, np.zeros(0, dtype=np.int32), 1.2, 0.1, 1.0)
    np.testing.assert_array_equal(t, logits.argmax(axis=1))


def test_penalty_rejects_out_of_range_history():
    with pytest.raises(ValueError):
        oracle.penalty_minp(np.zeros((1, 4), np.float32), np.array([4], np.int32), 1.2, 0.1, 1.0)


# ---------------------------------------------------------------- acceptance
def test_accept_hand_examples(golden_dir):
    rows = _parse(os.path.join(golden_dir, "accept_hand.txt"))
    assert len(rows) >= 5
    for name, par, dr, tg, anc, res, path in rows:
        r, p = oracle.accept(_nums(dr, int), _nums(par, int), _nums(tg, int), int(anc))
        L, best, bonus = _nums(res, int)
        assert (r[0], r[1], r[2], r[3]) == (L, best, bonus, 0), name
        want = _nums(path, int)
        assert p[:len(want)].tolist() == want and all(x == -1 for x in p[len(want):]), name


def _accept_by_enumeration(draft, parent, target, anchor):
    g = nx.DiGraph()
    g.add_node("r")
    for i, p in enumerate(parent):
        g.add_edge("r" if p < 0 else p, i)
    best_len, best_row = 0, -1
    for i in range(len(parent)):
        path = nx.shortest_path(g, "r", i)[1:]
        ok = all(draft[n] == (anchor if parent[n] < 0 else target[parent[n]]) for n in path)
        if ok and len(path) > best_len:
            best_len, best_row = len(path), i
    return best_len, best_row


@pytest.mark.parametrize("seed", range(6))
def test_accept_matches_path_enumeration(seed):
    parent = W.verify_parents()
    vi = W.make_vocab_inputs(parent, V=500, W=50, seed=seed)
    target = vi.designed_target.numpy()
    r, path = oracle.accept(vi.draft.numpy(), parent, target, vi.anchor)
    L, best = _accept_by_enumeration(vi.draft.tolist(), parent, target.tolist(), vi.anchor)
    assert (r[0], r[1]) == (L, best)
    assert r[2] == (target[best] if L > 0 else vi.anchor)
    if L:
        assert path[L - 1] == best


def _longest_rows(draft, parent, target, anchor):
    """Rows of the longest accepted paths, ascending, by networkx path enumeration."""
    g = nx.DiGraph()
    g.add_node("r")
    for i, p in enumerate(parent):
        g.add_edge("r" if p < 0 else p, i)
    ok = {}
    for i in range(len(parent)):
        path = nx.shortest_path(g, "r", i)[1:]
        if all(draft[n] == (anchor if parent[n] < 0 else target[parent[n]]) for n in path):
            ok[i] = len(path)
    L = max(ok.values(), default=0)
    return L, sorted(i for i, n in ok.items() if n == L and L > 0)


def test_random_longest_choice_follows_numpy_philox():
    """The kept row is S[floor(x m / 2^64)], S the longest accepted rows in
    ascending order (networkx), x word 0 of numpy's Philox4x64 at counter
    (0, 0, offset, 1) under key (seed, 0)."""
    parent = [-1, 0, 0, 0, 1, 2, 3, -1, 7, 8]
    target = [5, 6, 6, 6, 9, 9, 9, 1, 2, 3]
    draft = [4, 5, 5, 5, 6, 6, 6, 4, 1, 2]     # rows 4, 5, 6 and 9 end paths of depth 3
    L, S = _longest_rows(draft, parent, target, 4)
    assert L == 3 and S == [4, 5, 6, 9]
    picks = []
    for seed, offset in [(1, 0), (1, 1), (99, 7), (2**63 + 5, 2**40)]:
        c = (offset << 128) + (1 << 192) - 1   # numpy adds 1 to the 256-bit counter before each block
        ctr = np.array([(c >> (64 * i)) & (2**64 - 1) for i in range(4)], dtype=np.uint64)
        bg = np.random.Philox(counter=ctr, key=np.array([seed, 0], dtype=np.uint64))
        x = int(bg.random_raw(1)[0])
        want = S[(x * len(S)) >> 64]
        r, path = oracle.accept(draft, parent, target, 4, seed=seed, offset=offset)
        assert (r[0], r[1], r[2]) == (3, want, target[want])
        assert path[:3].tolist() == nx.shortest_path(
            nx.DiGraph([("r" if p < 0 else p, i) for i, p in enumerate(parent)]), "r", want)[1:]
        picks.append(want)
    assert len(set(picks)) > 1


def test_random_longest_choice_is_uniform_and_valid():
    parent = W.verify_parents()
    vi = W.make_vocab_inputs(parent, V=300, W=20, seed=12)
    target = vi.designed_target.numpy()
    # every chain repeats the tree's path so that several rows tie for the longest
    draft = vi.draft.numpy().copy()
    L0, S0 = _longest_rows(draft.tolist(), parent, target.tolist(), vi.anchor)
    for c in range(20):
        rows = [40 + 4 * c + j for j in range(4)]
        draft[rows[0]] = vi.anchor
        for j in range(1, 4):
            draft[rows[j]] = target[rows[j - 1]]
    L, S = _longest_rows(draft.tolist(), parent, target.tolist(), vi.anchor)
    assert L == 4 and len(S) >= 20
    R = 6000
    counts = np.zeros(len(S))
    for o in range(R):
        r, _ = oracle.accept(draft, parent, target, vi.anchor, seed=2024, offset=o)
        assert r[0] == L and r[1] in S
        counts[S.index(r[1])] += 1
    chi2 = (((counts - R / len(S)) ** 2) / (R / len(S))).sum()
    assert scipy.stats.chi2.sf(chi2, len(S) - 1) > 1e-4
    # one longest row: the draw has nothing to choose
    if len(S0) == 1:
        r, _ = oracle.accept(vi.draft.numpy(), parent, target, vi.anchor, seed=5)
        assert r[1] == S0[0]


def test_planted_targets_are_the_oracle_targets():
    """The input generator's designed tokens are what the greedy step picks."""
    parent = W.verify_parents()
    vi = W.make_vocab_inputs(parent, V=4000, W=256, seed=1, flip_rows=0.5)
    t, _ = oracle.penalty_minp(vi.logits.numpy(), vi.history.numpy(), 1.2, 0.1, 1.0)
    np.testing.assert_array_equal(t, vi.designed_target.numpy())
    # without the penalty the flipped rows pick the history token instead
    t0, _ = oracle.penalty_minp(vi.logits.numpy(), vi.history.numpy(), 1.0, 0.1, 1.0)
    assert (t0 != t).sum() > 10


# --------------------------------------------------------------------------
# commit of the accepted path
# --------------------------------------------------------------------------
def _ancestors(parent, row):
    out = []
    while row >= 0:
        out.append(row)
        row = parent[row]
    return out[::-1]


@pytest.mark.parametrize("best", [0, 5, 20, 39, 41, 119])
def test_commit_makes_the_path_the_sequence(best):
    """After the commit, plain attention of the accepted row over the first
    N + L cache rows equals its tree attention before the commit: the row saw
    exactly the prefix and its ancestors, which the commit lays out in order."""
    parent = W.verify_parents()
    T, Hq, Hkv, d, N = len(parent), 4, 2, 64, 100
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=best, value_kind="normal")
    scale = 1.0 / math.sqrt(d)
    path = _ancestors(parent, best)
    L = len(path)
    pth = np.full(T, -1, dtype=np.int32)
    pth[:L] = path
    k2, v2, st = oracle.commit_path(k, v, N, [L, best, 0, 0], pth)
    assert st == 0
    before, lse_b = oracle.tree_attn(q, k, v, N, parent, scale, rows=list(range(best * Hq, best * Hq + Hq)))
    after, lse_a = oracle.tree_attn(q[best:best + 1], k2, v2, N + L - 1, [-1], scale)
    np.testing.assert_allclose(after.reshape(-1), before.reshape(-1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_a.reshape(-1), lse_b.reshape(-1), rtol=0, atol=1e-12)
    # rows past the committed ones are untouched
    assert torch.equal(k2[:, N + L:], k[:, N + L:]) and torch.equal(v2[:, :N], v[:, :N])


def test_commit_identity_and_data_errors():
    T, Hkv, d, N = 12, 2, 64, 8
    _, k, v = W.make_qkv(T, 2, Hkv, d, N, seed=3)
    chain = np.arange(T, dtype=np.int32)
    for L in (0, 1, 5, T):  # a path 0, 1, ..., L-1 leaves the cache as it is
        k2, v2, st = oracle.commit_path(k, v, N, [L, L - 1, 0, 0], chain)
        assert st == 0 and torch.equal(k2, k) and torch.equal(v2, v)
    for res, pth in (([3, 0, 0, 0], [0, 2, 2] + [-1] * 9),     # not increasing
                     ([2, 0, 0, 0], [0, T] + [-1] * 10),       # outside the batch
                     ([T + 1, 0, 0, 0], list(range(T))),       # L > T
                     ([-1, 0, 0, 0], list(range(T)))):
        k2, v2, st = oracle.commit_path(k, v, N, res, np.asarray(pth, dtype=np.int32))
        assert st == 5 and torch.equal(k2, k) and torch.equal(v2, v)


# --------------------------------------------------------------------------
# min-p sampling: Philox4x64-10, the fp32 logarithm, the Gumbel-max draw
# --------------------------------------------------------------------------
def test_philox_matches_numpy():
    """numpy's Philox bit generator is Philox4x64-10; it advances its counter
    before each block, so its block from counter c - 1 is ours at counter c."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        c = [int(rng.integers(1, 2**63)), int(rng.integers(0, 2**63)), int(rng.integers(0, 2**63)), 0]
        k = [int(rng.integers(0, 2**63)), int(rng.integers(0, 2**63))]
        bg = np.random.Philox(counter=[c[0] - 1, c[1], c[2], c[3]], key=k)
        np.testing.assert_array_equal(oracle.philox4x64(c, k), bg.random_raw(4).astype(np.uint64))


def test_ln_f32_within_four_ulp():
    rng = np.random.default_rng(6)
    xs = np.concatenate([np.exp(rng.uniform(-60, 60, 4000)), 1 + rng.uniform(-0.3, 0.3, 2000),
                         (2.0 * np.arange(1, 2000) + 1) * 2.0 ** -24]).astype(np.float32)
    for x in xs:
        got = oracle.ln_f32(float(x))
        ref = math.log(float(x))
        ulp = np.spacing(np.float32(abs(ref))) if ref != 0 else np.float32(2.0 ** -149)
        assert abs(got - ref) <= 4 * float(ulp), (x, got, ref)


@pytest.mark.parametrize("min_p", [0.0, 0.3])
def test_gumbel_max_draws_the_min_p_distribution(min_p):
    """Each row draws independently (its own counter); over many rows the
    frequencies match softmax(l) renormalised over the min-p kept set."""
    logits = np.array([0.0, 0.5, 1.0, 1.5, -3.0, 2.0, 1.9], dtype=np.float32)
    R = 40000
    s = oracle.sample(np.tile(logits, (R, 1)), min_p, seed=1234)
    p = np.exp(logits - logits.max())
    keep = p >= min_p * p.max()
    p = np.where(keep, p, 0.0)
    p /= p.sum()
    counts = np.bincount(s, minlength=logits.size)
    assert counts[~keep].sum() == 0
    exp = p[keep] * R
    chi2 = (((counts[keep] - exp) ** 2) / exp).sum()
    assert scipy.stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4, (counts, exp)


def test_sampling_edge_cases():
    lg = np.array([[0.0, 5.0, 1.0], [3.0, 3.0, -1.0]], dtype=np.float32)
    # min_p = 1: only the maximum is kept, so the draw is the argmax (ties: both kept)
    s = oracle.sample(lg, 1.0, seed=9)
    assert s[0] == 1 and s[1] in (0, 1)
    # the same seed and offset reproduce; another offset draws anew
    big = np.random.default_rng(0).normal(0, 3, (64, 1000)).astype(np.float32)
    a, b, c = (oracle.sample(big, 0.0, seed=3, offset=o) for o in (0, 0, 1))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


# --------------------------------------------------------------------------
# n-gram table: top-k 4-grams of the generated text that start with the anchor
# --------------------------------------------------------------------------
def _ngram_brute(seq, anchor, k):
    from collections import Counter
    c = Counter(tuple(seq[p - 3:p + 1]) for p in range(3, len(seq)))
    cand = sorted(((-n, w[1:], w) for w, n in c.items() if w[0] == anchor))
    return [list(w) for _, _, w in cand[:k]], [-n for n, _, _ in cand[:k]]


def test_ngram_hand_examples(golden_dir):
    for line in open(os.path.join(golden_dir, "ngram_hand.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, seq, anchor, k, want = [x.strip() for x in line.split("|")]
        chains, counts = oracle.ngram_topk([int(x) for x in seq.split()], int(anchor), int(k))
        got = "-" if len(chains) == 0 else " ; ".join(
            " ".join(str(int(x)) for x in c) + f" : {int(n)}" for c, n in zip(chains, counts))
        assert got == want, name


@pytest.mark.parametrize("vocab,n,k", [(3, 200, 5), (6, 1000, 20), (50, 3000, 20), (2, 40, 30)])
def test_ngram_topk_matches_a_counter(vocab, n, k):
    """Against collections.Counter over every window, for every anchor."""
    seq = np.random.default_rng(vocab * n).integers(0, vocab, n).tolist()
    total = 0
    for a in range(vocab + 1):
        chains, counts = oracle.ngram_topk(seq, a, k)
        want_c, want_n = _ngram_brute(seq, a, k)
        assert chains.tolist() == want_c and counts.tolist() == want_n
        total += oracle.ngram_topk(seq, a, 10 ** 6)[1].sum()
    assert total == n - 3  # every window counted once


def test_ngram_update_adds_exactly_the_new_window():
    seq = [3, 1, 4, 1, 5, 9, 2, 6, 5, 3, 5, 8, 9, 7, 9, 3, 2, 3, 8, 4]
    for n in range(4, len(seq)):
        before = {tuple(c): m for c, m in zip(*oracle.ngram_topk(seq[:n], seq[n - 3], 10 ** 6))}
        after = {tuple(c): m for c, m in zip(*oracle.ngram_topk(seq[:n + 1], seq[n - 3], 10 ** 6))}
        w = tuple(seq[n - 3:n + 1])
        assert after[w] == before.get(w, 0) + 1
        assert all(after[x] == before[x] for x in before if x != w)
