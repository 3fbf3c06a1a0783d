"""B300-native (sm_103a) attention-side hot path of TokenSwift speculative decoding.

The compute lives in the C-ABI library ``libts.so`` (hand-written CUDA, see
``include/ts.h``); this package is a thin ctypes binding with the same names.
It marshals torch tensors into raw pointers and the current CUDA stream, and
raises :class:`TSError` on any non-OK status.  There is no fallback: if the
library is missing, every call raises.

``workloads`` (seeded synthetic inputs) imports nothing from here.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libts.so")

TS_NOALLOC_SCRATCH_BYTES = 64 << 20
TS_OK, TS_ERR_INVALID_ARG, TS_ERR_UNSUPPORTED, TS_ERR_CUDA, TS_ERR_TIMEOUT, TS_ERR_DATA = range(6)
TS_VOCAB_SAMPLE, TS_VOCAB_PATH_WINDOW = 1, 2
_STATUS = {0: "TS_OK", 1: "TS_ERR_INVALID_ARG", 2: "TS_ERR_UNSUPPORTED", 3: "TS_ERR_CUDA",
           4: "TS_ERR_TIMEOUT", 5: "TS_ERR_DATA"}

__all__ = ["TSError", "lib", "ts_version", "ts_tree_mask_from_parents", "ts_tree_attn_workspace_bytes",
           "ts_launch_count", "ts_tree_attn_uses_tensor_cores", "ts_device_error", "ts_selftest_bounded_wait",
           "ts_selftest_fail_launches", "ts_tree_attn",
           "ts_tree_attn_unmerged", "ts_tree_attn_merge", "ts_tree_attn_partial", "ts_tree_attn_noalloc", "ts_score_chunks", "ts_rescore_tail",
           "ts_select_gather", "ts_select_chunks", "ts_gather_tree_attn",
           "ts_select_gather_tree_attn", "ts_penalty_minp_verify", "ts_penalty_minp_sample_verify", "ts_commit_path",
           "ts_ngram_table_bytes", "ts_ngram_reset", "ts_ngram_update", "ts_ngram_topk", "ts_vocab_verify"]


class TSError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libts.so (built in-tree by ``python -m long_context_attention_tree_b300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m long_context_attention_tree_b300.build` (no fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        L.ts_last_error.restype = ctypes.c_char_p
        L.ts_version.restype = ctypes.c_char_p
        L.ts_launch_count.restype = ctypes.c_uint64
        L.ts_tree_mask_from_parents.argtypes = [P, i32, P]
        L.ts_tree_mask_words.argtypes = [i32]
        L.ts_tree_mask_words.restype = i32
        L.ts_tree_attn_workspace_bytes.argtypes = [i32, i32, i32, i32, i64]
        L.ts_tree_attn_workspace_bytes.restype = sz
        L.ts_tree_attn_uses_tensor_cores.argtypes = [i32, i32, i32, i32, i64]
        L.ts_tree_attn_uses_tensor_cores.restype = i32
        L.ts_device_error.argtypes = [i32]
        L.ts_device_error.restype = i32
        L.ts_selftest_bounded_wait.argtypes = [ctypes.c_uint64, P]
        L.ts_selftest_bounded_wait.restype = i32
        L.ts_selftest_fail_launches.argtypes = [i32]
        L.ts_selftest_fail_launches.restype = None
        L.ts_tree_attn.argtypes = [P, P, P, i64, i64, i32, i32, i32, i32, f32, P, P, P, P, i32, P, sz, P]
        L.ts_tree_attn_partial.argtypes = [P, P, P, i64, i64, i32, i32, i32, i32, f32, P, P, P, P, P, sz, P]
        L.ts_tree_attn_unmerged.argtypes = [P, P, P, i64, i64, i32, i32, i32, i32, f32, P, P, P, P, i32, P, sz, P]
        L.ts_tree_attn_merge.argtypes = [i64, i32, i32, i32, i32, P, P, P, sz, P]
        L.ts_tree_attn_noalloc.argtypes = [P, P, P, i64, i64, i32, i32, i32, i32, f32, P, P, P, P, i32, P]
        L.ts_score_chunks.argtypes = [P, P, i64, i64, i32, i32, i32, i32, P, P]
        L.ts_rescore_tail.argtypes = [P, i64, P, P, i64, i64, i32, i32, i32, i32, P, P]
        L.ts_select_gather.argtypes = [P, i32, i64, i32, i32, i32, i32, P, P, i64, i32, P, P, P, P, i64, P]
        L.ts_select_chunks.argtypes = [P, i32, i64, i32, i32, i32, i32, P, P, P]
        L.ts_gather_tree_attn.argtypes = [P, P, P, i64, i64, P, i32, P, P, i64, i32, i32, i32, i32, f32, P, P, P,
                                          P, sz, P]
        L.ts_select_gather_tree_attn.argtypes = [P, i64, i32, i32, i32, i32, P, P, P, P, P, i64, P, P, i64, i32, i32,
                                                 i32, i32, f32, P, P, P, P, sz, P]
        L.ts_vocab_verify.argtypes = [P, i32, i32, P, i32, f32, f32, f32, ctypes.c_uint, ctypes.c_uint64,
                                      ctypes.c_uint64, P, P, ctypes.c_int32, P, P, P, P, P]
        L.ts_penalty_minp_verify.argtypes = [P, i32, i32, P, i32, f32, f32, f32, P, P, ctypes.c_int32,
                                             P, P, P, P, P, sz, P]
        L.ts_commit_path.argtypes = [P, P, i64, i64, i32, i32, i32, P, P, P]
        L.ts_ngram_table_bytes.argtypes = [i64]
        L.ts_ngram_table_bytes.restype = sz
        L.ts_ngram_reset.argtypes = [P, i64, P]
        L.ts_ngram_update.argtypes = [P, i64, P, i64, i64, P, P]
        L.ts_ngram_topk.argtypes = [P, i64, P, i64, P, i32, P, P, P, P]
        u64 = ctypes.c_uint64
        L.ts_penalty_minp_sample_verify.argtypes = [P, i32, i32, P, i32, f32, f32, f32, u64, u64, P, P,
                                                    ctypes.c_int32, P, P, P, P, P]
        for name in ("ts_tree_mask_from_parents", "ts_tree_attn", "ts_tree_attn_unmerged", "ts_tree_attn_merge",
                     "ts_tree_attn_partial", "ts_tree_attn_noalloc",
                     "ts_score_chunks", "ts_rescore_tail", "ts_select_gather", "ts_select_chunks",
                     "ts_gather_tree_attn", "ts_select_gather_tree_attn", "ts_penalty_minp_verify",
                     "ts_commit_path", "ts_penalty_minp_sample_verify", "ts_ngram_reset", "ts_ngram_update",
                     "ts_ngram_topk", "ts_vocab_verify"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != TS_OK:
        raise TSError(status, lib().ts_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def ts_version() -> str:
    return lib().ts_version().decode()


def ts_launch_count() -> int:
    """Kernels the library has launched so far in this process."""
    return int(lib().ts_launch_count())


def ts_tree_mask_from_parents(parent) -> np.ndarray:
    """uint64 [T][max(2, ceil(T/64))] ancestor-or-self mask (host)."""
    p = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    T = p.size
    mask = np.zeros((max(T, 1), int(lib().ts_tree_mask_words(T))), dtype=np.uint64)
    _check(lib().ts_tree_mask_from_parents(p.ctypes.data_as(ctypes.c_void_p), T,
                                           mask.ctypes.data_as(ctypes.c_void_p)))
    return mask[:T]


def ts_tree_attn_workspace_bytes(T: int, Hq: int, Hkv: int, d: int, N: int) -> int:
    return int(lib().ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N))


def ts_tree_attn_uses_tensor_cores(T: int, Hq: int, Hkv: int, d: int, N: int) -> bool:
    """True when these sizes run on the tcgen05 tensor-core kernel."""
    return bool(lib().ts_tree_attn_uses_tensor_cores(T, Hq, Hkv, d, N))


def ts_device_error(clear: bool = True) -> int:
    """Sticky device status (0 = OK, TS_ERR_TIMEOUT if a bounded wait gave up).
    Waits for the device."""
    st = lib().ts_device_error(1 if clear else 0)
    return int(st)


def ts_selftest_bounded_wait(budget_ns: int, stream=None) -> None:
    """One warp whose bounded wait on an mbarrier nobody arrives at gives up
    after budget_ns and records TS_ERR_TIMEOUT (read it with ts_device_error)."""
    _check(lib().ts_selftest_bounded_wait(int(budget_ns), _stream(stream)))


def ts_selftest_fail_launches(n: int) -> None:
    """Make the next n kernel launches fail on the host (TS_ERR_CUDA); 0 = off."""
    lib().ts_selftest_fail_launches(int(n))


def ts_tree_attn(q, k, v, N: int, mask, out, lse=None, chunk_scores=None, score_row: int = 0,
                 workspace=None, scale: Optional[float] = None, stream=None) -> None:
    """Tree-masked GQA attention.  q [T][Hq][d], k/v [Hkv][ld][d] (bf16, CUDA),
    mask uint64 [T][2] (CUDA), out bf16 [T][Hq][d]; lse fp32 [T][Hq] optional;
    chunk_scores fp32 [Hkv][ceil(N/64)] optional; workspace uint8 CUDA tensor."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ts_tree_attn(_ptr(q), _ptr(k), _ptr(v), ld, N, T, Hq, Hkv, d, scale, _ptr(mask), _ptr(out),
                              _ptr(lse), _ptr(chunk_scores), score_row, _ptr(workspace), ws_bytes,
                              _stream(stream)))


def ts_tree_attn_unmerged(q, k, v, N: int, mask, out, lse=None, chunk_scores=None, score_row: int = 0,
                          workspace=None, scale: Optional[float] = None, stream=None) -> None:
    """The attention kernel of ts_tree_attn without the merge of its split
    partials; ts_tree_attn_merge completes out / lse."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ts_tree_attn_unmerged(_ptr(q), _ptr(k), _ptr(v), ld, N, T, Hq, Hkv, d, scale, _ptr(mask), _ptr(out),
                                       _ptr(lse), _ptr(chunk_scores), score_row, _ptr(workspace), ws_bytes,
                                       _stream(stream)))


def ts_tree_attn_merge(out, Hkv: int, N: int, lse=None, workspace=None, stream=None) -> None:
    """The log-sum-exp merge that completes ts_tree_attn_unmerged (same out,
    lse, workspace and shapes)."""
    T, Hq, d = out.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ts_tree_attn_merge(N, T, Hq, Hkv, d, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                    _stream(stream)))


def ts_tree_attn_partial(q, k_part, v_part, B: int, mask, part_len, out, lse=None, workspace=None,
                         scale: Optional[float] = None, stream=None) -> None:
    """Drafting attention over the compact partial cache: KV head g sees the
    gathered rows [0, part_len[g]) and the batch rows [B, B+T) by the mask."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k_part.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ts_tree_attn_partial(_ptr(q), _ptr(k_part), _ptr(v_part), ld, B, T, Hq, Hkv, d, scale, _ptr(mask),
                                      _ptr(part_len), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                      _stream(stream)))


def ts_tree_attn_noalloc(q, k, v, N: int, mask, out, lse=None, chunk_scores=None, score_row: int = 0,
                         scale: Optional[float] = None, stream=None) -> None:
    """ts_tree_attn without a caller workspace, for callers that cannot
    allocate device memory: the split partials go to the library's own
    file-scope device array (TS_NOALLOC_SCRATCH_BYTES, held by every GPU
    that loads the library).  Calls that overlap on the GPU race on it."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    _check(lib().ts_tree_attn_noalloc(_ptr(q), _ptr(k), _ptr(v), ld, N, T, Hq, Hkv, d, scale, _ptr(mask),
                                      _ptr(out), _ptr(lse), _ptr(chunk_scores), score_row, _stream(stream)))


def ts_score_chunks(q_row, k, N: int, scores, chunk: int = 64, stream=None) -> None:
    Hq, d = q_row.shape
    Hkv, ld, _ = k.shape
    _check(lib().ts_score_chunks(_ptr(q_row), _ptr(k), ld, N, Hq, Hkv, d, chunk, _ptr(scores), _stream(stream)))


def ts_rescore_tail(scores_old, N_old: int, q_row, k, N_new: int, scores_new, chunk: int = 64,
                    stream=None) -> None:
    """Chunk scores at N_new from the scores at N_old: only the chunks from
    floor(N_old/64) on are scored again."""
    Hq, d = q_row.shape
    Hkv, ld, _ = k.shape
    _check(lib().ts_rescore_tail(_ptr(scores_old), N_old, _ptr(q_row), _ptr(k), ld, N_new, Hq, Hkv, d, chunk,
                                 _ptr(scores_new), _stream(stream)))


def ts_select_gather(scores, N: int, budget_tokens: int, k, v, sel, k_part, v_part, chunk: int = 64,
                     part_len=None, sink_chunks: int = 0, recent_chunks: int = 0, stream=None) -> None:
    Hkv, ld, d = k.shape
    ld_part = k_part.shape[1]
    _check(lib().ts_select_gather(_ptr(scores), Hkv, N, budget_tokens, chunk, int(sink_chunks), int(recent_chunks),
                                  _ptr(k), _ptr(v), ld, d, _ptr(sel), _ptr(part_len), _ptr(k_part), _ptr(v_part),
                                  ld_part, _stream(stream)))


def ts_select_chunks(scores, N: int, budget_tokens: int, sel, chunk: int = 64, part_len=None, sink_chunks: int = 0,
                     recent_chunks: int = 0, stream=None) -> None:
    """The selection of ts_select_gather alone (sel, part_len)."""
    Hkv = scores.shape[0]
    _check(lib().ts_select_chunks(_ptr(scores), Hkv, N, budget_tokens, chunk, int(sink_chunks), int(recent_chunks),
                                  _ptr(sel), _ptr(part_len), _stream(stream)))


def ts_gather_tree_attn(q, k, v, N: int, sel, k_part, v_part, mask, out, lse=None, workspace=None,
                        scale: Optional[float] = None, stream=None) -> None:
    """The gather of the selected chunks (sel [Hkv][k_sel]) into k_part/v_part
    fused with the drafting attention over them (batch rows at [64 k_sel, +T))."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    k_sel = sel.shape[1]
    ld_part = k_part.shape[1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ts_gather_tree_attn(_ptr(q), _ptr(k), _ptr(v), ld, N, _ptr(sel), k_sel, _ptr(k_part), _ptr(v_part),
                                     ld_part, T, Hq, Hkv, d, scale, _ptr(mask), _ptr(out), _ptr(lse),
                                     _ptr(workspace), ws_bytes, _stream(stream)))


def ts_select_gather_tree_attn(scores, q, k, v, N: int, budget_tokens: int, sel, k_part, v_part, mask, out,
                               part_len=None, lse=None, workspace=None, chunk: int = 64, sink_chunks: int = 0,
                               recent_chunks: int = 0, scale: Optional[float] = None, stream=None) -> None:
    """ts_select_chunks and ts_gather_tree_attn in one pass (every CTA selects
    its head's chunks itself): sel, part_len, the compact cache, out, lse."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    ld_part = k_part.shape[1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ts_select_gather_tree_attn(_ptr(scores), N, budget_tokens, chunk, int(sink_chunks),
                                            int(recent_chunks), _ptr(sel), _ptr(part_len), _ptr(q), _ptr(k), _ptr(v),
                                            ld, _ptr(k_part), _ptr(v_part), ld_part, T, Hq, Hkv, d, scale, _ptr(mask),
                                            _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))


def ts_penalty_minp_verify(logits, history, theta: float, min_p: float, temperature: float, draft, parent,
                           anchor: int, target, kept, result, path, stream=None) -> None:
    T, V = logits.shape
    W = 0 if history is None else history.numel()
    _check(lib().ts_penalty_minp_verify(_ptr(logits), T, V, _ptr(history) if W else None, W, theta, min_p,
                                        temperature, _ptr(draft), _ptr(parent), int(anchor), _ptr(target),
                                        _ptr(kept), _ptr(result), _ptr(path), None, 0, _stream(stream)))


def ts_commit_path(k, v, N: int, result, path, stream=None) -> None:
    """Move the accepted rows N + path[i] to N + i (i < result[0]) in place."""
    Hkv, ld, d = k.shape
    T = path.numel()
    _check(lib().ts_commit_path(_ptr(k), _ptr(v), ld, N, T, Hkv, d, _ptr(result), _ptr(path), _stream(stream)))


def ts_penalty_minp_sample_verify(logits, history, theta: float, min_p: float, temperature: float, seed: int,
                                  offset: int, draft, parent, anchor: int, target, kept, result, path,
                                  stream=None) -> None:
    """ts_penalty_minp_verify with min-p sampled targets (Gumbel-max, Philox4x64-10)."""
    T, V = logits.shape
    W = 0 if history is None else history.numel()
    _check(lib().ts_penalty_minp_sample_verify(_ptr(logits), T, V, _ptr(history) if W else None, W, theta, min_p,
                                               temperature, int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                               _ptr(draft), _ptr(parent), int(anchor), _ptr(target), _ptr(kept),
                                               _ptr(result), _ptr(path), _stream(stream)))


def ts_ngram_table_bytes(capacity: int) -> int:
    """Bytes of an n-gram table of `capacity` slots (0 if capacity is invalid)."""
    return int(lib().ts_ngram_table_bytes(int(capacity)))


def ts_ngram_reset(table, capacity: int, stream=None) -> None:
    _check(lib().ts_ngram_reset(_ptr(table), int(capacity), _stream(stream)))


def ts_ngram_update(table, capacity: int, seq, n_old: int, n_new: int, status, stream=None) -> None:
    """Add the 4-grams ending at positions [max(3, n_old), n_new) of seq (int32, CUDA)."""
    _check(lib().ts_ngram_update(_ptr(table), int(capacity), _ptr(seq), int(n_old), int(n_new), _ptr(status),
                                 _stream(stream)))


def ts_ngram_topk(table, capacity: int, seq, n: int, anchor, k: int, chains, counts, found, stream=None) -> None:
    """Top-k 4-grams of seq[0, n) starting with the device int32 anchor:
    chains [k][4], counts [k], found [1] (the table holds the windows of seq[0, n))."""
    _check(lib().ts_ngram_topk(_ptr(table), int(capacity), _ptr(seq), int(n), _ptr(anchor), int(k), _ptr(chains),
                               _ptr(counts), _ptr(found), _stream(stream)))


def ts_vocab_verify(logits, history, theta: float, min_p: float, temperature: float, flags: int, seed: int,
                    offset: int, draft, parent, anchor: int, target, kept, result, path, stream=None) -> None:
    """The vocab stage with options: TS_VOCAB_SAMPLE, TS_VOCAB_PATH_WINDOW."""
    T, V = logits.shape
    W = 0 if history is None else history.numel()
    _check(lib().ts_vocab_verify(_ptr(logits), T, V, _ptr(history) if W else None, W, theta, min_p, temperature,
                                 int(flags), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(draft),
                                 _ptr(parent), int(anchor), _ptr(target), _ptr(kept), _ptr(result), _ptr(path),
                                 _stream(stream)))
