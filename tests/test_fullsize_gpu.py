"""Full-size parity in the launch configuration the benchmark times.

The whole spec step (every layer: verify attention with fused chunk scores,
top-k select + gather, draft attention; then the vocabulary stage) runs once
through the C ABI; afterwards every layer is checked against the fp64 oracle:
chunk scores, selections and gathered caches bit for bit, attention outputs on
sampled rows (the oracle computes rows one by one), and the vocab stage
exactly."""
import numpy as np
import pytest
import torch

import oracle
from long_context_attention_tree_b300 import workloads as W
from long_context_attention_tree_b300.step import SpecStep

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 2e-2, 1e-2, 1e-3


def _check_rows(out, lse, ref_o, ref_l, rows, what):
    o = out.reshape(-1, out.shape[-1])[rows].float().cpu().double().numpy()
    l = lse.reshape(-1)[rows].cpu().double().numpy()
    err = np.abs(o - ref_o).max()
    rel = np.linalg.norm(o - ref_o) / np.linalg.norm(ref_o)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max abs {err:.3e}, rel L2 {rel:.3e}"
    assert np.abs(l - ref_l).max() <= LSE_ABS, what


def _check_step(step: SpecStep, layers, rows_per_layer=6):
    cfg = step.cfg
    rng = np.random.default_rng(cfg.cid)
    for i in layers:
        Lb = step.layers[i]
        q, k, v = Lb.q.cpu(), Lb.k.cpu(), Lb.v.cpu()
        # chunk scores (fused into the verify pass) and selection: bit-exact
        rs = oracle.score_chunks(q[0], k, cfg.N).astype(np.float32)
        np.testing.assert_array_equal(Lb.scores.cpu().numpy(), rs, err_msg=f"layer {i} scores")
        rsel = oracle.select(rs, cfg.k_sel)
        np.testing.assert_array_equal(Lb.sel.cpu().numpy(), rsel, err_msg=f"layer {i} sel")
        kp, vp = Lb.k_part.cpu(), Lb.v_part.cpu()
        rkp, rlen = oracle.gather(rsel, k, cfg.N, 64, kp.shape[1], fill=kp, return_len=True)
        assert torch.equal(kp, rkp), f"layer {i} k_part"
        np.testing.assert_array_equal(Lb.part_len.cpu().numpy(), rlen, err_msg=f"layer {i} part_len")
        assert torch.equal(vp, oracle.gather(rsel, v, cfg.N, 64, vp.shape[1], fill=vp)), f"layer {i} v_part"
        # verify attention on sampled rows: always the scoring row's heads, a tree leaf, a chain end
        rows = np.unique(np.concatenate([
            np.arange(cfg.Hq), [39 * cfg.Hq + 1, (step.T - 1) * cfg.Hq + cfg.Hq - 1],
            rng.integers(0, step.T * cfg.Hq, size=rows_per_layer)])).astype(np.int32)
        ro, rl = oracle.tree_attn(q, k, v, cfg.N, step.parents, cfg.scale, rows=rows)
        _check_rows(Lb.out, Lb.lse, ro, rl, rows, f"layer {i} verify")
        # draft attention over the partial cache: every row
        ro, rl = oracle.tree_attn(Lb.q_draft.cpu(), kp, vp, step.B, step.draft_parents, cfg.scale, prefix_len=rlen)
        _check_rows(Lb.out_draft, Lb.lse_draft, ro.reshape(-1, cfg.d), rl.reshape(-1),
                    np.arange(step.Td * cfg.Hq), f"layer {i} draft")


def test_qwen14b_full_step_all_layers():
    cfg = W.WORKLOADS["qwen14b-100k"]
    step = SpecStep(cfg)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)
    s.synchronize()
    _check_step(step, range(step.n_layers), rows_per_layer=4)
    vi = step.vocab_inputs
    rt, rk = oracle.penalty_minp(vi.logits.cpu().numpy(), vi.history.cpu().numpy(), cfg.theta, cfg.min_p,
                                 cfg.temperature)
    np.testing.assert_array_equal(step.target.cpu().numpy(), rt)
    np.testing.assert_array_equal(step.kept.cpu().numpy(), rk)
    rr, rp = oracle.accept(vi.draft.cpu().numpy(), step.parents, rt, vi.anchor)
    np.testing.assert_array_equal(step.result.cpu().numpy(), rr)
    np.testing.assert_array_equal(step.path.cpu().numpy(), rp)
    assert rr[0] >= 1  # the planted drafts give a non-trivial accepted length


def test_step_graph_replay_matches_eager():
    cfg = W.WORKLOADS["qwen14b-100k"]
    step = SpecStep(cfg, layers=3)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)
    s.synchronize()
    eager = [(L.out.clone(), L.lse.clone(), L.scores.clone(), L.sel.clone(), L.out_draft.clone())
             for L in step.layers]
    res = step.result.clone()
    for L in step.layers:
        L.out.zero_(); L.scores.zero_(); L.sel.zero_(); L.out_draft.zero_()
    step.result.zero_()
    g = step.capture(s)
    g.replay()
    s.synchronize()
    for L, e in zip(step.layers, eager):
        assert torch.equal(L.out, e[0]) and torch.equal(L.lse, e[1]) and torch.equal(L.scores, e[2])
        assert torch.equal(L.sel, e[3]) and torch.equal(L.out_draft, e[4])
    assert torch.equal(step.result, res)


@pytest.mark.parametrize("N", [20480, 40960, 61440, 81920, 102400])
def test_llama8b_sweep_layers(N):
    cfg = W.WORKLOADS["llama8b-sweep"].with_N(N)
    step = SpecStep(cfg, layers=2)
    step.run()
    torch.cuda.synchronize()
    _check_step(step, range(2))


def test_qwen14b_layers_with_a_separate_gather():
    """The step with the gather as its own call (selection + gather, then the
    drafting attention over the compact cache) instead of fused with the
    drafting pass."""
    cfg = W.WORKLOADS["qwen14b-100k"]
    step = SpecStep(cfg, layers=2, fuse_gather=False)
    step.run()
    torch.cuda.synchronize()
    _check_step(step, range(2))


def test_qwen14b_layers_with_the_selection_as_its_own_call():
    """The step with the selection as its own call before the gather-and-draft
    call (instead of inside the drafting kernel)."""
    cfg = W.WORKLOADS["qwen14b-100k"]
    step = SpecStep(cfg, layers=2, fuse_select=False)
    step.run()
    torch.cuda.synchronize()
    _check_step(step, range(2))


def test_llama2_7b_mha_layer():
    cfg = W.WORKLOADS["llama2-7b-100k"]
    step = SpecStep(cfg)
    step.run()
    torch.cuda.synchronize()
    _check_step(step, [0], rows_per_layer=24)
