"""The speculative loop over several steps on one layer, through the C ABI.

Each step follows "How it works" on the TokenSwift tool listing: draft over
the partial cache, verify the tree + n-gram batch over the full cache (chunk
importance fused), accept the longest exact-match path, commit its K/V rows
(N grows by the accepted length L), then refresh the partial cache for the next
step: re-score only the chunks the commit touched and re-select / re-gather at
the new N.  The prefix starts two tokens short of a chunk boundary so that the
last chunk is short and the chunk count changes within the first steps.

Every step is checked against the fp64 oracle from the same device state:
scores, selections, gathered caches and lengths, committed caches and the
vocab stage bit for bit; attention outputs within the bars."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_tree_b300 as ts
import oracle
from long_context_attention_tree_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 2e-2, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from long_context_attention_tree_b300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def _mask(parent):
    return torch.from_numpy(ts.ts_tree_mask_from_parents(parent).view(np.int64)).cuda()


def _close(out, lse, ro, rl, what):
    o = out.float().cpu().double().numpy().reshape(ro.shape)
    err = np.abs(o - ro).max()
    rel = np.linalg.norm(o - ro) / np.linalg.norm(ro)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max abs {err:.3e} rel {rel:.3e}"
    assert np.abs(lse.cpu().double().numpy().reshape(rl.shape) - rl).max() <= LSE_ABS, what


@pytest.mark.parametrize("Hq,Hkv,N0", [(40, 8, 4094), (32, 32, 1022)])
def test_spec_loop_verify_accept_commit_refresh_draft(Hq, Hkv, N0):
    d, budget, Td, steps, V, Wn = 128, 1024, 4, 4, 4096, 128
    parent = W.verify_parents()
    T = len(parent)
    draft_parent = [-1, 0, 1, 2]
    scale = 1 / math.sqrt(d)
    cap = N0 + steps * (T + 8)
    gen = torch.Generator(device="cuda").manual_seed(N0)
    rint = lambda shape: torch.randint(-4, 5, shape, generator=gen, device="cuda").to(torch.bfloat16)
    rnorm = lambda shape: torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.zeros((Hkv, cap, d), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    k[:, :N0] = rint((Hkv, N0, d))
    v[:, :N0] = rnorm((Hkv, N0, d))
    mask, dmask = _mask(parent), _mask(draft_parent)
    kk = budget // 64
    B = kk * 64
    kp = torch.zeros((Hkv, B + Td, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    sel = torch.empty((Hkv, kk), dtype=torch.int32, device="cuda")
    plen = torch.empty((Hkv,), dtype=torch.int32, device="cuda")
    ws = torch.empty(max(ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, cap),
                         ts.ts_tree_attn_workspace_bytes(Td, Hq, Hkv, d, B), 16), dtype=torch.uint8, device="cuda")

    # initial partial cache: scores of a first query over the prefix
    q_prev = rint((Hq, d))
    sc = torch.empty((Hkv, (N0 + 63) // 64), dtype=torch.float32, device="cuda")
    ts.ts_score_chunks(q_prev, k, N0, sc)
    ts.ts_select_gather(sc, N0, budget, k, v, sel, kp, vp, part_len=plen)
    N = N0
    crossed = False
    lengths = []
    for step in range(steps):
        # ---- the draft batch's own K/V rows after the gathered tokens, then drafting
        qd = rint((Td, Hq, d))
        kp[:, B:] = rint((Hkv, Td, d))
        vp[:, B:] = rnorm((Hkv, Td, d))
        od = torch.empty((Td, Hq, d), dtype=torch.bfloat16, device="cuda")
        ld = torch.empty((Td, Hq), dtype=torch.float32, device="cuda")
        ts.ts_tree_attn_partial(qd, kp, vp, B, dmask, plen, od, lse=ld, workspace=ws, scale=scale)
        torch.cuda.synchronize()
        kp_h, vp_h, plen_h = kp.cpu(), vp.cpu(), plen.cpu().numpy()
        ro, rl = oracle.tree_attn(qd.cpu(), kp_h, vp_h, B, draft_parent, scale, prefix_len=plen_h)
        _close(od, ld, ro, rl, f"step {step} draft")

        # ---- verify: the batch's K/V rows at [N, N+T), fused chunk scores of row 0
        q = rint((T, Hq, d))
        k[:, N:N + T] = rint((Hkv, T, d))
        v[:, N:N + T] = rnorm((Hkv, T, d))
        out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        sc = torch.full((Hkv, (N + 63) // 64), float("nan"), dtype=torch.float32, device="cuda")
        ts.ts_tree_attn(q, k, v, N, mask, out, lse=lse, chunk_scores=sc, score_row=0, workspace=ws, scale=scale)
        # ---- vocab stage: targets, acceptance
        vi = W.make_vocab_inputs(parent, V, Wn, seed=100 * N0 + step, device="cuda", flip_rows=0.25)
        target = torch.empty((T,), dtype=torch.int32, device="cuda")
        kept = torch.empty_like(target)
        result = torch.empty((4,), dtype=torch.int32, device="cuda")
        path = torch.empty_like(target)
        ts.ts_penalty_minp_verify(vi.logits, vi.history, 1.2, 0.1, 1.0, vi.draft, vi.parent, vi.anchor, target,
                                  kept, result, path)
        torch.cuda.synchronize()
        k_before, v_before = k.cpu(), v.cpu()
        rows = np.unique(np.concatenate([np.arange(Hq), (T - 1) * Hq + np.arange(Hq),
                                         np.random.default_rng(step).integers(0, T * Hq, 16)])).astype(np.int32)
        ro, rl = oracle.tree_attn(q.cpu(), k_before, v_before, N, parent, scale, rows=rows)
        _close(out.reshape(-1, d)[rows], lse.reshape(-1)[rows], ro, rl, f"step {step} verify")
        rs = oracle.score_chunks(q[0].cpu(), k_before, N).astype(np.float32)
        np.testing.assert_array_equal(sc.cpu().numpy(), rs, err_msg=f"step {step} scores")
        rt, rk = oracle.penalty_minp(vi.logits.cpu().numpy(), vi.history.cpu().numpy(), 1.2, 0.1, 1.0)
        np.testing.assert_array_equal(target.cpu().numpy(), rt)
        rres, rpath = oracle.accept(vi.draft.cpu().numpy(), parent, rt, vi.anchor)
        np.testing.assert_array_equal(result.cpu().numpy(), rres)
        np.testing.assert_array_equal(path.cpu().numpy(), rpath)

        # ---- commit the accepted path, N grows by L
        ts.ts_commit_path(k, v, N, result, path)
        L = int(result[0].item())
        lengths.append(L)
        rk_c, rv_c, st = oracle.commit_path(k_before, v_before, N, rres, rpath)
        torch.cuda.synchronize()
        assert st == 0
        assert torch.equal(k.cpu(), rk_c) and torch.equal(v.cpu(), rv_c), f"step {step} commit"
        N_new = N + L
        crossed |= (N_new + 63) // 64 > (N + 63) // 64

        # ---- refresh: re-score the touched chunks with the verify pass's scoring query, re-select, re-gather
        sc_new = torch.full((Hkv, (N_new + 63) // 64), float("nan"), dtype=torch.float32, device="cuda")
        ts.ts_rescore_tail(sc, N, q[0], k, N_new, sc_new)
        ts.ts_select_gather(sc_new, N_new, budget, k, v, sel, kp, vp, part_len=plen)
        torch.cuda.synchronize()
        k_now = k.cpu()
        rs_new = oracle.score_chunks(q[0].cpu(), k_now, N_new).astype(np.float32)
        np.testing.assert_array_equal(sc_new.cpu().numpy(), rs_new, err_msg=f"step {step} rescore")
        rsel = oracle.select(rs_new, kk)
        np.testing.assert_array_equal(sel.cpu().numpy(), rsel, err_msg=f"step {step} sel")
        rkp, rlen = oracle.gather(rsel, k_now, N_new, 64, B + Td, fill=kp_h, return_len=True)
        np.testing.assert_array_equal(plen.cpu().numpy(), rlen)
        assert torch.equal(kp.cpu()[:, :B], rkp[:, :B]), f"step {step} k_part"
        rvp = oracle.gather(rsel, v.cpu(), N_new, 64, B + Td, fill=vp_h)
        assert torch.equal(vp.cpu()[:, :B], rvp[:, :B]), f"step {step} v_part"
        N = N_new
    assert sum(lengths) > 0, lengths          # the planted drafts are accepted at some steps
    assert N0 % 64 != 0 and crossed           # a short last chunk, and the chunk count grew
    assert ts.ts_device_error(True) == ts.TS_OK
