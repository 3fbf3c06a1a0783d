"""One TokenSwift speculative step over all layers, on device-resident buffers.

Per layer (the order of "How it works" on the TokenSwift tool listing, with the
partial cache refreshed every step as the ICML 2025 summary's ablation
favours, dynamic over one-time):
  1. verify attention: the T-row batch (draft tree + n-gram chains) against
     the full KV cache, producing the chunk importance of the scoring row in
     the same pass;
  2. top-k chunk selection up to the retrieval budget;
  3. gather of the chosen chunks into the compact partial cache and the draft
     attention of the 4-row self-drafting batch over it, in one pass over the
     chosen K/V (fuse_gather; otherwise a separate gather call before the
     drafting attention over the compact cache).  By default (fuse_select)
     steps 2 and 3 are one kernel: every CTA of the drafting kernel selects its
     KV head's chunks itself.
Then, once per step, the vocabulary stage (penalty, min-p, greedy target,
acceptance).

Every step is one C-ABI call into libts.so; this module only owns device
memory (allocated once, through torch) and orders the calls on a stream
(the merge of a layer's verify partials on a side stream beside the
selection and drafting pass, joined before the next layer).  The step can be
captured into a CUDA graph.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from . import (ts_gather_tree_attn, ts_penalty_minp_verify, ts_select_chunks, ts_select_gather,
               ts_select_gather_tree_attn, ts_tree_attn, ts_tree_attn_merge, ts_tree_attn_partial,
               ts_tree_attn_unmerged, ts_tree_attn_workspace_bytes, ts_tree_mask_from_parents)
from . import workloads as W


@dataclasses.dataclass
class LayerBuffers:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    q_draft: torch.Tensor
    k_part: torch.Tensor
    v_part: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor
    scores: torch.Tensor
    sel: torch.Tensor
    part_len: torch.Tensor
    out_draft: torch.Tensor
    lse_draft: torch.Tensor


class SpecStep:
    def __init__(self, cfg: W.Config, device="cuda", layers: Optional[int] = None, vocab: Optional[bool] = None,
                 value_kind: str = "int", fill_draft_tail: bool = True, want_lse: bool = True,
                 fuse_gather: bool = True, overlap_select: bool = True, fuse_select: bool = True):
        self.cfg = cfg
        self.fuse_gather = fuse_gather
        # the selection inside the drafting kernel (every CTA selects its head's
        # chunks), so the refresh call has nothing left to do
        self.fuse_select = fuse_gather and fuse_select
        # with a stream given, the merge of a layer's verify partials runs on a
        # side stream beside the selection and the drafting pass (the
        # selection needs only the chunk scores of the verify kernel)
        self.overlap_select = overlap_select
        # the log-sum-exp outputs (the method itself consumes only O; the
        # kernels skip the exact normaliser sum when it is not asked for)
        self.want_lse = want_lse
        self.device = torch.device(device)
        self.n_layers = cfg.layers if layers is None else layers
        self.T = cfg.T
        self.Td = cfg.draft_rows
        self.k_sel = cfg.k_sel
        self.B = self.k_sel * cfg.chunk
        parents = cfg.parents
        self.parents = parents
        self.draft_parents = [-1] + list(range(self.Td - 1))
        self.mask = torch.from_numpy(ts_tree_mask_from_parents(parents).view(np.int64)).to(self.device)
        self.mask_draft = torch.from_numpy(ts_tree_mask_from_parents(self.draft_parents).view(np.int64)).to(self.device)
        ws = ts_tree_attn_workspace_bytes(self.T, cfg.Hq, cfg.Hkv, cfg.d, cfg.N)
        ws_d = ts_tree_attn_workspace_bytes(self.Td, cfg.Hq, cfg.Hkv, cfg.d, self.B)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=self.device)
        self.workspace_draft = torch.empty(max(ws_d, 16), dtype=torch.uint8, device=self.device)
        self.layers: List[LayerBuffers] = []
        nc = cfg.n_chunks
        for layer in range(self.n_layers):
            x = W.make_layer_inputs(cfg, layer, device=self.device, value_kind=value_kind)
            kp = torch.zeros((cfg.Hkv, self.B + self.Td, cfg.d), dtype=torch.bfloat16, device=self.device)
            vp = torch.zeros_like(kp)
            if fill_draft_tail:
                kp[:, self.B:] = x.k_draft_tail
                vp[:, self.B:] = x.v_draft_tail
            self.layers.append(LayerBuffers(
                q=x.q, k=x.k, v=x.v, q_draft=x.q_draft, k_part=kp, v_part=vp,
                out=torch.empty((self.T, cfg.Hq, cfg.d), dtype=torch.bfloat16, device=self.device),
                lse=torch.empty((self.T, cfg.Hq), dtype=torch.float32, device=self.device),
                scores=torch.empty((cfg.Hkv, nc), dtype=torch.float32, device=self.device),
                sel=torch.empty((cfg.Hkv, self.k_sel), dtype=torch.int32, device=self.device),
                part_len=torch.empty((cfg.Hkv,), dtype=torch.int32, device=self.device),
                out_draft=torch.empty((self.Td, cfg.Hq, cfg.d), dtype=torch.bfloat16, device=self.device),
                lse_draft=torch.empty((self.Td, cfg.Hq), dtype=torch.float32, device=self.device),
            ))
        self.vocab = (cfg.vocab > 0) if vocab is None else vocab
        if self.vocab:
            vi = W.make_vocab_inputs(parents, cfg.vocab, cfg.window, seed=1000 * cfg.cid + 999,
                                     device=self.device, flip_rows=0.25)
            self.vocab_inputs = vi
            self.target = torch.empty(self.T, dtype=torch.int32, device=self.device)
            self.kept = torch.empty(self.T, dtype=torch.int32, device=self.device)
            self.result = torch.empty(4, dtype=torch.int32, device=self.device)
            self.path = torch.empty(self.T, dtype=torch.int32, device=self.device)

    # ------------------------------------------------------------------
    def run_verify(self, i: int, stream=None) -> None:
        cfg, L = self.cfg, self.layers[i]
        ts_tree_attn(L.q, L.k, L.v, cfg.N, self.mask, L.out, lse=L.lse if self.want_lse else None,
                     chunk_scores=L.scores, score_row=0,
                     workspace=self.workspace, scale=cfg.scale, stream=stream)

    def run_refresh(self, i: int, stream=None) -> None:
        cfg, L = self.cfg, self.layers[i]
        if self.fuse_select:
            return  # done by the drafting kernel
        if self.fuse_gather:
            ts_select_chunks(L.scores, cfg.N, cfg.budget, L.sel, chunk=cfg.chunk, part_len=L.part_len, stream=stream)
        else:
            ts_select_gather(L.scores, cfg.N, cfg.budget, L.k, L.v, L.sel, L.k_part, L.v_part, chunk=cfg.chunk,
                             part_len=L.part_len, stream=stream)

    def run_draft(self, i: int, stream=None) -> None:
        cfg, L = self.cfg, self.layers[i]
        lse = L.lse_draft if self.want_lse else None
        if self.fuse_select:
            ts_select_gather_tree_attn(L.scores, L.q_draft, L.k, L.v, cfg.N, cfg.budget, L.sel, L.k_part, L.v_part,
                                       self.mask_draft, L.out_draft, part_len=L.part_len, lse=lse,
                                       workspace=self.workspace_draft, chunk=cfg.chunk, scale=cfg.scale,
                                       stream=stream)
        elif self.fuse_gather:
            ts_gather_tree_attn(L.q_draft, L.k, L.v, cfg.N, L.sel, L.k_part, L.v_part, self.mask_draft, L.out_draft,
                                lse=lse, workspace=self.workspace_draft, scale=cfg.scale, stream=stream)
        else:
            ts_tree_attn_partial(L.q_draft, L.k_part, L.v_part, self.B, self.mask_draft, L.part_len, L.out_draft,
                                 lse=lse, workspace=self.workspace_draft, scale=cfg.scale, stream=stream)

    def run_layer(self, i: int, stream=None) -> None:
        if not (self.overlap_select and stream is not None):
            self.run_verify(i, stream)
            self.run_refresh(i, stream)
            self.run_draft(i, stream)
            return
        cfg, L = self.cfg, self.layers[i]
        if not hasattr(self, "_side"):
            self._side = torch.cuda.Stream(device=self.device)
            self._ev_scores = [torch.cuda.Event() for _ in range(self.n_layers)]
            self._ev_draft = [torch.cuda.Event() for _ in range(self.n_layers)]
        # verify kernel; its chunk scores feed the selection and drafting pass
        # right behind it on this stream (each a programmatic dependent of the
        # kernel before it), while the merge of its split partials runs on the
        # side stream
        lse = L.lse if self.want_lse else None
        ts_tree_attn_unmerged(L.q, L.k, L.v, cfg.N, self.mask, L.out, lse=lse, chunk_scores=L.scores, score_row=0,
                              workspace=self.workspace, scale=cfg.scale, stream=stream)
        self._ev_scores[i].record(stream)
        self._side.wait_event(self._ev_scores[i])
        ts_tree_attn_merge(L.out, cfg.Hkv, cfg.N, lse=lse, workspace=self.workspace, stream=self._side)
        self._ev_draft[i].record(self._side)
        self.run_refresh(i, stream)
        self.run_draft(i, stream)
        stream.wait_event(self._ev_draft[i])  # the merge is done before the workspace is used again

    def run_vocab(self, stream=None) -> None:
        cfg, vi = self.cfg, self.vocab_inputs
        ts_penalty_minp_verify(vi.logits, vi.history, cfg.theta, cfg.min_p, cfg.temperature, vi.draft, vi.parent,
                               vi.anchor, self.target, self.kept, self.result, self.path, stream=stream)

    def run(self, stream=None) -> None:
        for i in range(self.n_layers):
            self.run_layer(i, stream)
        if self.vocab:
            self.run_vocab(stream)

    # ------------------------------------------------------------------
    def capture(self, stream: torch.cuda.Stream) -> torch.cuda.CUDAGraph:
        """Capture one whole step into a CUDA graph (launch gaps removed)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.run(stream)  # warm-up outside capture (sets kernel attributes)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            self.run(stream)
        return g

    def kv_bytes_per_step(self) -> int:
        return self.n_layers * self.cfg.kv_bytes_per_layer()
