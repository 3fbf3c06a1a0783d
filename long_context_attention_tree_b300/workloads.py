"""Seeded synthetic inputs for the TokenSwift attention-side hot path.

This module only draws numbers and lays out shapes. It holds none of the
method's arithmetic (no attention, no scoring, no penalty, no acceptance), so
that the CUDA path and the fp64 oracle can both be fed from it.

Shapes follow the workloads the TokenSwift pages evaluate (LLaMA3.1-8B GQA,
LLaMA2-7B-128k MHA, Qwen2.5-14B; 20K-100K context; "Key results" of the ICML
2025 summary page) and the inference flags of the TokenSwift model card
("Example using TokenSwift command line": retrieval budget 4096, gamma 4,
min_p 0.1, temperature 1.0, ngram_topk 20, penalty 1.2, penalty_length 1024).
The draft tree is [1,3,3,3] (ablation table of the summary page).

Value recipe (stated once, used everywhere):
  * Q and K are integers drawn uniformly from [-4, 4] and stored as bf16, so
    every q.k product and every chunk sum is an exact small integer.
  * V is N(0, 1) rounded to bf16.
  * seed = 1000 * config_id + layer; draw order per layer: Q, K (N+T rows),
    V (N+T rows), draft Q (4 rows), draft tail K, draft tail V.
  * Vocab stage: logits N(0, 3) fp32; a window of W uniform history ids;
    per-row designed target tokens (see ``make_vocab_inputs``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

CHUNK = 64


# --------------------------------------------------------------------------
# tree / chain structure (parent arrays; topological order, parent[i] < i)
# --------------------------------------------------------------------------
def tree_parents(branching: Sequence[int]) -> List[int]:
    """Parent array of a BFS-numbered draft tree.

    ``branching[0]`` roots, then every node of level k has ``branching[k]``
    children.  [1,3,3,3] gives 1+3+9+27 = 40 nodes (the tree of the
    TokenSwift ablation table)."""
    parents: List[int] = []
    prev_start, prev_count = -1, 0
    for level, b in enumerate(branching):
        start = len(parents)
        if level == 0:
            parents.extend([-1] * b)
            count = b
        else:
            count = prev_count * b
            for i in range(count):
                parents.append(prev_start + i // b)
        prev_start, prev_count = start, count
    return parents


def chain_parents(n_chains: int, length: int, offset: int = 0) -> List[int]:
    """Parent array of ``n_chains`` independent chains of ``length`` rows,
    numbered from ``offset`` (each chain head is a root, parent -1)."""
    out: List[int] = []
    for c in range(n_chains):
        for j in range(length):
            row = offset + c * length + j
            out.append(-1 if j == 0 else row - 1)
    return out


def verify_parents(branching: Sequence[int] = (1, 3, 3, 3), n_chains: int = 20,
                   chain_len: int = 4) -> List[int]:
    """Verify batch: the draft tree followed by the candidate n-gram chains."""
    p = tree_parents(branching)
    return p + chain_parents(n_chains, chain_len, offset=len(p))


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    cid: int
    name: str
    Hq: int
    Hkv: int
    d: int
    N: int                     # prefix (cache) tokens, excluding the T tail rows
    branching: tuple = (1, 3, 3, 3)
    n_chains: int = 20
    chain_len: int = 4
    budget: int = 4096         # partial-cache budget in tokens
    chunk: int = CHUNK
    layers: int = 1
    draft_rows: int = 4        # gamma
    vocab: int = 0             # 0: no vocab stage
    window: int = 1024
    theta: float = 1.2
    min_p: float = 0.1
    temperature: float = 1.0

    @property
    def parents(self) -> List[int]:
        return verify_parents(self.branching, self.n_chains, self.chain_len)

    @property
    def T(self) -> int:
        return len(self.parents)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_chunks(self) -> int:
        return (self.N + self.chunk - 1) // self.chunk

    @property
    def k_sel(self) -> int:
        return min(self.budget // self.chunk, self.n_chunks)

    @property
    def scale(self) -> float:
        # fp32 value of 1/sqrt(d)
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def with_N(self, N: int) -> "Config":
        return dataclasses.replace(self, N=N)

    def kv_bytes_per_layer(self) -> int:
        """Prefix K+V bytes one verify pass reads (bf16)."""
        return 2 * self.Hkv * self.N * self.d * 2


WORKLOADS = {
    "tiny": Config(1, "tiny-1layer", Hq=4, Hkv=1, d=64, N=4096, n_chains=0, budget=1024),
    "llama8b-20k": Config(2, "llama3.1-8b-20k-1layer", Hq=32, Hkv=8, d=128, N=20480),
    "llama8b-sweep": Config(3, "llama3.1-8b-sweep-32layer", Hq=32, Hkv=8, d=128, N=102400, layers=32),
    "llama2-7b-100k": Config(4, "llama2-7b-mha-100k-1layer", Hq=32, Hkv=32, d=128, N=102400),
    "qwen14b-100k": Config(5, "qwen2.5-14b-100k-48layer-step", Hq=40, Hkv=8, d=128, N=102400, layers=48,
                           vocab=152064),
}
SWEEP_N = (20480, 40960, 61440, 81920, 102400)


# --------------------------------------------------------------------------
# per-layer tensors
# --------------------------------------------------------------------------
@dataclasses.dataclass
class LayerInputs:
    q: torch.Tensor        # bf16 [T][Hq][d]
    k: torch.Tensor        # bf16 [Hkv][N+T][d]  (prefix rows then tail rows)
    v: torch.Tensor        # bf16 [Hkv][N+T][d]
    q_draft: torch.Tensor  # bf16 [Td][Hq][d]
    k_draft_tail: torch.Tensor  # bf16 [Hkv][Td][d]
    v_draft_tail: torch.Tensor  # bf16 [Hkv][Td][d]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _int_bf16(shape, g, device) -> torch.Tensor:
    return torch.randint(-4, 5, shape, generator=g, device=device, dtype=torch.int32).to(torch.bfloat16)


def _normal_bf16(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_layer_inputs(cfg: Config, layer: int = 0, device="cpu", seed: Optional[int] = None,
                      T: Optional[int] = None, value_kind: str = "int") -> LayerInputs:
    """Draw one layer's tensors.  ``value_kind='int'`` is the recipe above;
    ``'normal'`` draws Q and K from N(0,1) as well (non-integer stress case)."""
    if seed is None:
        seed = 1000 * cfg.cid + layer
    T = cfg.T if T is None else T
    g = _gen(seed, device)
    draw_qk = _int_bf16 if value_kind == "int" else _normal_bf16
    q = draw_qk((T, cfg.Hq, cfg.d), g, device)
    k = draw_qk((cfg.Hkv, cfg.N + T, cfg.d), g, device)
    v = _normal_bf16((cfg.Hkv, cfg.N + T, cfg.d), g, device)
    Td = cfg.draft_rows
    qd = draw_qk((Td, cfg.Hq, cfg.d), g, device)
    kd = draw_qk((cfg.Hkv, Td, cfg.d), g, device)
    vd = _normal_bf16((cfg.Hkv, Td, cfg.d), g, device)
    return LayerInputs(q, k, v, qd, kd, vd)


def make_qkv(T: int, Hq: int, Hkv: int, d: int, N: int, seed: int, device="cpu",
             value_kind: str = "int", ld_extra: int = 0):
    """Free-shape Q/K/V for parity sweeps.  K/V have N+T+ld_extra rows."""
    g = _gen(seed, device)
    draw_qk = _int_bf16 if value_kind == "int" else _normal_bf16
    q = draw_qk((T, Hq, d), g, device)
    k = draw_qk((Hkv, N + T + ld_extra, d), g, device)
    v = _normal_bf16((Hkv, N + T + ld_extra, d), g, device)
    return q, k, v


# --------------------------------------------------------------------------
# vocab stage
# --------------------------------------------------------------------------
@dataclasses.dataclass
class VocabInputs:
    logits: torch.Tensor    # fp32 [T][V]
    history: torch.Tensor   # int32 [W]
    draft: torch.Tensor     # int32 [T]
    parent: torch.Tensor    # int32 [T]
    anchor: int
    designed_target: torch.Tensor  # int32 [T]: the token each row was built to prefer


def make_vocab_inputs(T_parents: Sequence[int], V: int, W: int, seed: int, device="cpu",
                      flip_rows: float = 0.0, p_match: float = 0.85) -> VocabInputs:
    """Logits N(0,3), a uniform history window, and drafts planted along the tree.

    Each row i gets a designed token t_i outside the history window whose logit
    is raised to (row max) + U(0.05, 1.5); it is then the row's greedy choice
    whatever the windowed penalty does to the history tokens.  With
    ``flip_rows`` > 0, that fraction of rows also gets a history token a_i with
    logit (row max) + 1.0 and t_i at (row max) + 0.5: a_i wins only when the
    penalty is NOT applied, so drafts planted on t_i test the penalty for real.

    Drafts: walking the rows in order, every node (and the virtual anchor for
    the roots) picks at most one child, with probability ``p_match``, whose
    draft equals the node's designed token; other children draw a different
    uniform id.  Acceptance rates of 0.83-0.90 are what the TokenSwift
    ablation reports across temperatures; 0.85 sits in that range.
    """
    T = len(T_parents)
    g = _gen(seed, "cpu")  # small host-side draws; moved to device at the end
    logits = torch.randn((T, V), generator=g, dtype=torch.float32) * 3.0
    history = torch.randint(0, V, (W,), generator=g, dtype=torch.int64)
    in_hist = torch.zeros(V, dtype=torch.bool)
    if W > 0:
        in_hist[history] = True
    non_hist = torch.nonzero(~in_hist).flatten()

    def pick_non_hist() -> int:
        return int(non_hist[torch.randint(0, non_hist.numel(), (1,), generator=g)])

    target = torch.empty(T, dtype=torch.int64)
    u = torch.rand(T, generator=g)
    flips = torch.rand(T, generator=g) < flip_rows
    hist_list = history.tolist()
    for i in range(T):
        row_max = float(logits[i].max())
        t = pick_non_hist()
        if bool(flips[i]) and W > 0 and row_max > 2.0:
            a = hist_list[int(torch.randint(0, W, (1,), generator=g))]
            if a != t:
                logits[i, a] = row_max + 1.0
                logits[i, t] = row_max + 0.5
            else:
                logits[i, t] = row_max + 0.05 + 1.45 * float(u[i])
        else:
            logits[i, t] = row_max + 0.05 + 1.45 * float(u[i])
        target[i] = t

    anchor = pick_non_hist()
    draft = torch.randint(0, V, (T,), generator=g, dtype=torch.int64)
    children = {}
    for i, p in enumerate(T_parents):
        children.setdefault(p, []).append(i)
    # roots: the tree root and each chain head are independent roots
    for node, kids in children.items():
        expected = anchor if node < 0 else int(target[node])
        if node < 0:
            # every root independently matches the anchor with p_match
            chosen = [c for c in kids if float(torch.rand(1, generator=g)) < p_match]
        else:
            chosen = [kids[int(torch.randint(0, len(kids), (1,), generator=g))]] \
                if float(torch.rand(1, generator=g)) < p_match else []
        for c in kids:
            if c in chosen:
                draft[c] = expected
            else:
                x = int(torch.randint(0, V, (1,), generator=g))
                draft[c] = x if x != expected else (x + 1) % V
    return VocabInputs(
        logits=logits.to(device),
        history=history.to(torch.int32).to(device),
        draft=draft.to(torch.int32).to(device),
        parent=torch.tensor(list(T_parents), dtype=torch.int32, device=device),
        anchor=int(anchor),
        designed_target=target.to(torch.int32).to(device),
    )
