"""fp64 CPU oracle of the TokenSwift attention-side hot path (test infrastructure).

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg use
this package; the product library never imports it, and it imports nothing
from the product.  The arithmetic lives in ``oracle.c`` (plain C, fp64,
OpenMP over output rows); this module marshals numpy/torch CPU arrays into it.

Functions, each following the definition stated in ``oracle.c``:
  visible            -- ancestor-or-self visibility of the speculative batch
  tree_attn          -- tree-masked attention (all rows or a sample of rows)
  score_chunks       -- chunk importance max_h q_h . sum(K_chunk)
  select             -- top-k chunks, ties to the lower index, ascending
  gather             -- compact partial cache
  penalty_minp       -- windowed penalty, temperature, min-p count, greedy target
  accept             -- exact-match acceptance, longest path
  commit_path        -- the accepted path's K/V rows moved to the end of the sequence
  philox4x64, ln_f32 -- Philox4x64-10 and the fp32 logarithm the sampler uses
  sample             -- min-p sampling (Gumbel-max over the kept set)
  ngram_topk         -- top-k 4-grams of the generated text that start with the anchor
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, dbl, flt = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
        lib.oracle_visible.argtypes = [P, i32, P]
        lib.oracle_tree_attn_rows.argtypes = [P, P, P, i64, i64, i32, i32, i32, i32, dbl, P, P, P, i32, P, P]
        lib.oracle_score_chunks.argtypes = [P, P, i64, i64, i32, i32, i32, i32, P]
        lib.oracle_select.argtypes = [P, i32, i32, i32, P]
        lib.oracle_gather.argtypes = [P, i32, i32, i32, i64, P, i64, i32, P, i64, P]
        lib.oracle_penalty_minp.argtypes = [P, i32, i32, P, i32, flt, flt, dbl, P, P, P]
        lib.oracle_penalty_minp_path.argtypes = [P, i32, i32, P, i32, P, P, flt, flt, dbl, P, P, P]
        lib.oracle_select_kept.argtypes = [P, i32, i32, i32, i32, i32, P]
        lib.oracle_accept.argtypes = [P, P, P, i32, i32, P, P]
        lib.oracle_accept_ex.argtypes = [P, P, P, i32, i32, i32, ctypes.c_uint64, ctypes.c_uint64, P, P]
        lib.oracle_commit.argtypes = [P, i64, i64, i32, i32, i32, P, P, P]
        lib.oracle_philox4x64.argtypes = [P, P, P]
        lib.oracle_ln_f32.argtypes = [flt]
        lib.oracle_ln_f32.restype = flt
        lib.oracle_sample.argtypes = [P, i32, i32, dbl, ctypes.c_uint64, ctypes.c_uint64, P]
        lib.oracle_ngram_topk.argtypes = [P, i64, i32, i32, P, P, P]
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_num_threads.restype = i32
        _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    import torch
    assert isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def visible(parent) -> np.ndarray:
    """bool [T][T]: row i sees batch row j (ancestor-or-self)."""
    p = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    T = p.size
    vis = np.zeros((T, T), dtype=np.uint8)
    rc = _load().oracle_visible(_ptr(p), T, _ptr(vis))
    if rc:
        raise ValueError("parent array must satisfy -1 <= parent[i] < i")
    return vis.astype(bool)


def tree_attn(q, k, v, N: int, parent, scale: float, rows=None, prefix_len=None):
    """Tree-masked attention in fp64.

    q: bf16 [T][Hq][d]; k, v: bf16 [Hkv][ld][d] (prefix [0,N), batch rows [N,N+T)).
    rows: None for every (t, h), else an int array of row ids t*Hq + h.
    prefix_len: None, or int [Hkv]: KV head g sees prefix rows [0, prefix_len[g]) only.
    Returns (out float64 [n_rows][d] or [T][Hq][d] when rows is None, lse float64)."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    p = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    pl = None if prefix_len is None else np.ascontiguousarray(np.asarray(prefix_len, dtype=np.int32))
    rid = np.arange(T * Hq, dtype=np.int32) if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    out = np.zeros((rid.size, d), dtype=np.float64)
    lse = np.zeros(rid.size, dtype=np.float64)
    rc = _load().oracle_tree_attn_rows(_ptr(qb), _ptr(kb), _ptr(vb), ld, N, T, Hq, Hkv, d,
                                       float(scale), _ptr(p), _ptr(pl) if pl is not None else None,
                                       _ptr(rid), rid.size, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_tree_attn_rows failed ({rc})")
    if rows is None:
        return out.reshape(T, Hq, d), lse.reshape(T, Hq)
    return out, lse


def score_chunks(q_row, k, N: int, chunk: int = 64) -> np.ndarray:
    """float64 [Hkv][ceil(N/chunk)]: max over the group of q_h . sum(K_chunk)."""
    Hq, d = q_row.shape
    Hkv, ld, _ = k.shape
    qb, kb = _bf16_bits(q_row), _bf16_bits(k)
    nc = (N + chunk - 1) // chunk
    out = np.zeros((Hkv, nc), dtype=np.float64)
    rc = _load().oracle_score_chunks(_ptr(qb), _ptr(kb), ld, N, Hq, Hkv, d, chunk, _ptr(out))
    if rc:
        raise ValueError(f"oracle_score_chunks failed ({rc})")
    return out


def select(scores_f32, k: int, sink: int = 0, recent: int = 0) -> np.ndarray:
    """int32 [Hkv][min(k, nc)]: top-k by (score desc, index asc), returned ascending.
    The decision is taken on fp32 scores (the kernel's precision).  The first
    `sink` and last `recent` chunks are always kept (sink + recent <= k)."""
    s = np.ascontiguousarray(np.asarray(scores_f32, dtype=np.float32))
    Hkv, nc = s.shape
    kk = min(k, nc)
    sel = np.zeros((Hkv, kk), dtype=np.int32)
    rc = _load().oracle_select_kept(_ptr(s), Hkv, nc, k, int(sink), int(recent), _ptr(sel))
    if rc:
        raise ValueError(f"oracle_select failed ({rc})")
    return sel


def gather(sel, src, N: int, chunk: int, ld_dst: int, fill=None, return_len=False):
    """bf16 [Hkv][ld_dst][d] compact cache holding the selected chunks (rows past
    k*chunk, and rows of a partial last chunk past N, keep ``fill`` (zeros)).
    With return_len, also the int32 [Hkv] count of tokens gathered per head."""
    import torch
    Hkv, ld_src, d = src.shape
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    kk = s.shape[1]
    srcb = _bf16_bits(src)
    dst = np.zeros((Hkv, ld_dst, d), dtype=np.uint16) if fill is None else _bf16_bits(fill).copy()
    plen = np.zeros(Hkv, dtype=np.int32)
    rc = _load().oracle_gather(_ptr(s), Hkv, kk, chunk, N, _ptr(srcb), ld_src, d, _ptr(dst), ld_dst, _ptr(plen))
    if rc:
        raise ValueError(f"oracle_gather failed ({rc})")
    out = torch.from_numpy(dst.view(np.int16)).view(torch.bfloat16)
    return (out, plen) if return_len else out


def log_min_p(min_p: float) -> float:
    """Natural log of min_p as a double (the min-p threshold offset in logit space)."""
    mp = float(np.float32(min_p))
    return -math.inf if mp <= 0.0 else math.log(mp)


def penalty_minp(logits, history, theta: float, min_p: float, temperature: float, return_logits=False,
                 path_parent=None, path_draft=None):
    """(target int32 [T], kept int32 [T][, final fp32 logits]) for fp32 logits [T][V].
    With path_parent / path_draft, each row's window is the last W tokens of
    history followed by the drafts on its path (root .. the row)."""
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.float32))
    T, V = lg.shape
    h = np.ascontiguousarray(np.asarray(history, dtype=np.int32))
    target = np.zeros(T, dtype=np.int32)
    kept = np.zeros(T, dtype=np.int32)
    pen = np.zeros((T, V), dtype=np.float32) if return_logits else None
    pp = None if path_parent is None else np.ascontiguousarray(np.asarray(path_parent, dtype=np.int32))
    pd = None if path_draft is None else np.ascontiguousarray(np.asarray(path_draft, dtype=np.int32))
    rc = _load().oracle_penalty_minp_path(_ptr(lg), T, V, _ptr(h), h.size, _ptr(pp) if pp is not None else None,
                                          _ptr(pd) if pd is not None else None, float(theta), float(temperature),
                                          log_min_p(min_p), _ptr(target), _ptr(kept),
                                          _ptr(pen) if pen is not None else None)
    if rc:
        raise ValueError(f"oracle_penalty_minp failed ({rc})")
    return (target, kept, pen) if return_logits else (target, kept)


def accept(draft, parent, target, anchor: int, seed=None, offset: int = 0):
    """(result int32[4] = {L, best, bonus, status}, path int32[T]).
    seed None keeps the lowest of the longest accepted rows; a seed draws it
    uniformly (Philox4x64-10 at counter (0, 0, offset, 1), key (seed, 0))."""
    dr = np.ascontiguousarray(np.asarray(draft, dtype=np.int32))
    p = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    tg = np.ascontiguousarray(np.asarray(target, dtype=np.int32))
    T = dr.size
    res = np.zeros(4, dtype=np.int32)
    path = np.zeros(max(T, 1), dtype=np.int32)
    _load().oracle_accept_ex(_ptr(dr), _ptr(p), _ptr(tg), T, int(anchor), 0 if seed is None else 1,
                             0 if seed is None else int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                             _ptr(res), _ptr(path))
    return res, path[:T]


def commit_path(k, v, N: int, result, path):
    """(k', v', status): bf16 caches after moving the accepted rows
    N + path[i] to N + i (i < result[0]); status 5 (and no move) on a bad path."""
    import torch
    res = np.ascontiguousarray(np.asarray(result, dtype=np.int32))
    pth = np.ascontiguousarray(np.asarray(path, dtype=np.int32))
    T = pth.size
    out = []
    status = 0
    for x in (k, v):
        Hkv, ld, d = x.shape
        xb = _bf16_bits(x).copy()
        st = np.zeros(1, dtype=np.int32)
        rc = _load().oracle_commit(_ptr(xb), ld, N, T, Hkv, d, _ptr(res), _ptr(pth), _ptr(st))
        if rc:
            raise ValueError(f"oracle_commit failed ({rc})")
        status = int(st[0])
        out.append(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16))
    return out[0], out[1], status


def philox4x64(counter, key) -> np.ndarray:
    """uint64[4]: Philox4x64-10 of a 4-word counter under a 2-word key."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_philox4x64(_ptr(c), _ptr(k), _ptr(out))
    return out


def ln_f32(x: float) -> float:
    """The sampler's fp32 natural logarithm (normal positive inputs)."""
    return float(_load().oracle_ln_f32(float(np.float32(x))))


def sample(pen_logits, min_p: float, seed: int, offset: int = 0) -> np.ndarray:
    """int32 [T]: min-p sampled targets from final fp32 logits [T][V] (Gumbel-max
    over the kept set, Philox4x64-10 uniforms keyed by (seed, 0) at counter
    (v / 4, row, offset, 0))."""
    lg = np.ascontiguousarray(np.asarray(pen_logits, dtype=np.float32))
    T, V = lg.shape
    out = np.zeros(T, dtype=np.int32)
    rc = _load().oracle_sample(_ptr(lg), T, V, log_min_p(min_p), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                               _ptr(out))
    if rc:
        raise ValueError(f"oracle_sample failed ({rc})")
    return out


def ngram_topk(seq, anchor: int, k: int):
    """(chains int32 [m][4], counts int32 [m]), m <= k: the 4-grams of seq that
    start with anchor, most frequent first, then by their last three tokens."""
    sq = np.ascontiguousarray(np.asarray(seq, dtype=np.int32))
    chains = np.zeros((max(k, 1), 4), dtype=np.int32)
    counts = np.zeros(max(k, 1), dtype=np.int32)
    found = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_ngram_topk(_ptr(sq), sq.size, int(anchor), int(k), _ptr(chains), _ptr(counts), _ptr(found))
    if rc:
        raise ValueError(f"oracle_ngram_topk failed ({rc})")
    m = int(found[0])
    return chains[:m], counts[:m]
