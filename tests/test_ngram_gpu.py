"""The device n-gram table and its top-k 4-gram retrieval against the oracle,
bit for bit: hand-worked cases, long random sequences (a small vocabulary for
heavy repetition and the Qwen2.5 vocabulary size), incremental updates equal to
one build, ties, a full table reported as a data error, and the chains fed
straight into the verify batch's draft tokens."""
import os

import numpy as np
import pytest
import torch

import long_context_attention_tree_b300 as ts
import oracle
from long_context_attention_tree_b300 import workloads as W

pytestmark = pytest.mark.gpu


def _table(capacity):
    t = torch.empty(ts.ts_ngram_table_bytes(capacity), dtype=torch.uint8, device="cuda")
    ts.ts_ngram_reset(t, capacity)
    return t


def _topk(table, capacity, seq, anchor, k):
    a = torch.tensor([anchor], dtype=torch.int32, device="cuda")
    chains = torch.full((k, 4), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    found = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ts.ts_ngram_topk(table, capacity, seq, seq.numel(), a, k, chains, counts, found)
    torch.cuda.synchronize()
    m = int(found.item())
    c, n = chains.cpu().numpy(), counts.cpu().numpy()
    assert (c[m:] == -1).all() and (n[m:] == 0).all()
    return c[:m], n[:m]


def _build(seq, capacity, steps=None):
    s = torch.tensor(seq, dtype=torch.int32, device="cuda")
    t = _table(capacity)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bounds = [0, len(seq)] if steps is None else steps
    for a, b in zip(bounds[:-1], bounds[1:]):
        ts.ts_ngram_update(t, capacity, s, a, b, status)
    torch.cuda.synchronize()
    return t, s, int(status.item())


def test_ngram_hand_examples(golden_dir):
    for line in open(os.path.join(golden_dir, "ngram_hand.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, seq, anchor, k, want = [x.strip() for x in line.split("|")]
        seq = [int(x) for x in seq.split()]
        t, sd, st = _build(seq, 64)
        assert st == 0
        chains, counts = _topk(t, 64, sd, int(anchor), int(k))
        got = "-" if len(chains) == 0 else " ; ".join(
            " ".join(str(int(x)) for x in c) + f" : {int(n)}" for c, n in zip(chains, counts))
        assert got == want, name


@pytest.mark.parametrize("vocab,n,capacity", [(50, 100000, 1 << 18), (152064, 100000, 1 << 18), (7, 3000, 1 << 13),
                                              (3, 500, 256)])
def test_ngram_topk_matches_oracle_long_sequences(vocab, n, capacity):
    rng = np.random.default_rng(vocab + n)
    seq = rng.integers(0, vocab, n).astype(np.int32)
    if vocab > 1000:  # plant repeats of a few phrases so that counts tie and differ
        for _ in range(400):
            p = int(rng.integers(0, n - 8))
            seq[p:p + 5] = [11, 12, 13, 14 + int(rng.integers(0, 3)), 15]
    t, sd, st = _build(seq.tolist(), capacity)
    assert st == 0
    anchors = list(rng.choice(seq, 12)) + [11, vocab + 5, 0]
    for a in anchors:
        for k in (1, 20, 64):
            chains, counts = _topk(t, capacity, sd, int(a), k)
            rc, rn = oracle.ngram_topk(seq, int(a), k)
            np.testing.assert_array_equal(chains, rc, err_msg=f"anchor {a} k {k}")
            np.testing.assert_array_equal(counts, rn, err_msg=f"anchor {a} k {k}")


def test_incremental_updates_equal_one_build():
    """Adding the sequence in steps of 1-5 tokens (as commits append them)
    gives the same table contents as one build."""
    rng = np.random.default_rng(5)
    seq = rng.integers(0, 20, 4000).astype(np.int32)
    steps = [0, 100]
    while steps[-1] < len(seq):
        steps.append(min(len(seq), steps[-1] + int(rng.integers(1, 6))))
    t1, sd, s1 = _build(seq.tolist(), 1 << 14)
    t2, _, s2 = _build(seq.tolist(), 1 << 14, steps)
    assert s1 == 0 and s2 == 0
    for a in range(21):
        c1, n1 = _topk(t1, 1 << 14, sd, a, 1024)
        c2, n2 = _topk(t2, 1 << 14, sd, a, 1024)
        rc, rn = oracle.ngram_topk(seq, a, 1024)
        np.testing.assert_array_equal(c1, rc)
        np.testing.assert_array_equal(c2, rc)
        np.testing.assert_array_equal(n1, rn)
        np.testing.assert_array_equal(n2, rn)
    # every window counted once: the counts of all anchors add up to n - 3
    assert sum(int(_topk(t2, 1 << 14, sd, a, 1024)[1].sum()) for a in range(20)) == len(seq) - 3


def test_anchor_with_more_candidates_than_shared_memory_holds():
    """An anchor followed by ~6000 distinct 4-grams: the candidates are cut to
    k in rounds and the result still equals the oracle's."""
    rng = np.random.default_rng(8)
    n = 60000
    seq = rng.integers(1, 5000, n).astype(np.int32)
    seq[::10] = 0  # anchor 0 every 10 tokens
    t, sd, st = _build(seq.tolist(), 1 << 17)
    assert st == 0
    for k in (20, 1024):
        chains, counts = _topk(t, 1 << 17, sd, 0, k)
        rc, rn = oracle.ngram_topk(seq, 0, k)
        np.testing.assert_array_equal(chains, rc)
        np.testing.assert_array_equal(counts, rn)


def test_full_table_and_bad_ids_are_data_errors():
    seq = list(range(200))  # 197 distinct 4-grams, 64 slots
    _, _, st = _build(seq, 64)
    assert st == ts.TS_ERR_DATA
    _, _, st = _build([1, 2, -3, 4, 5], 64)
    assert st == ts.TS_ERR_DATA
    assert ts.ts_device_error(True) == ts.TS_OK


def test_chains_feed_the_verify_batch_on_device():
    """The anchor comes from the vocab stage's bonus token (device memory) and
    the chains land in the draft tokens of the verify batch's chain rows."""
    parent = W.verify_parents()
    T = len(parent)
    vi = W.make_vocab_inputs(parent, 4096, 64, seed=3, device="cuda")
    rng = np.random.default_rng(3)
    seq = rng.integers(0, 30, 20000).astype(np.int32)
    t, sd, _ = _build(seq.tolist(), 1 << 15)
    result = torch.tensor([0, -1, 7, 0], dtype=torch.int32, device="cuda")  # bonus token 7
    draft = vi.draft.clone()
    counts = torch.empty(20, dtype=torch.int32, device="cuda")
    found = torch.empty(1, dtype=torch.int32, device="cuda")
    ts.ts_ngram_topk(t, 1 << 15, sd, sd.numel(), result[2:], 20, draft[40:], counts, found)
    torch.cuda.synchronize()
    rc, rn = oracle.ngram_topk(seq, 7, 20)
    np.testing.assert_array_equal(draft[40:40 + 4 * len(rc)].cpu().numpy().reshape(-1, 4), rc)
    np.testing.assert_array_equal(draft[:40].cpu().numpy(), vi.draft[:40].cpu().numpy())
