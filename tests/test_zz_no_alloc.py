"""The allocation-free attention entry point, for callers that cannot
allocate device memory (code inside another runtime's execution callback, or
a C caller without an allocator, where cudaMalloc is forbidden or would
synchronize the device).  It must give the same results as ts_tree_attn with
a caller workspace.  Collected last on purpose: a failure here leaves every
other test already run."""
import ctypes
import math

import numpy as np
import pytest
import torch

import long_context_attention_tree_b300 as ts
from long_context_attention_tree_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 2e-2, 1e-2, 1e-3


def _mask(parent):
    return torch.from_numpy(ts.ts_tree_mask_from_parents(parent).view(np.int64)).cuda()


def _outputs(T, Hq, d):
    return (torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda"),
            torch.empty((T, Hq), dtype=torch.float32, device="cuda"))


def _call_noalloc_cabi(q, k, v, N, mask, out, lse, scores, scale):
    """Direct C-ABI call (raw pointers, current stream)."""
    T, Hq, d = q.shape
    Hkv, ld, _ = k.shape
    L = ts.lib()
    st = L.ts_tree_attn_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                ctypes.c_void_p(v.data_ptr()), ld, N, T, Hq, Hkv, d, scale,
                                ctypes.c_void_p(mask.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(lse.data_ptr()),
                                ctypes.c_void_p(scores.data_ptr()) if scores is not None else None, 0,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ts.TS_OK, L.ts_last_error().decode()


def _close(a, b, what):
    x = a.float().cpu().double().numpy()
    y = b.float().cpu().double().numpy()
    assert np.abs(x - y).max() <= MAX_ABS, what
    assert np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30) <= REL_L2, what


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    from long_context_attention_tree_b300 import build
    build.build()
    cases = [
        # verify pass over a 20K cache with fused chunk scores, then a 4-row draft pass
        (W.verify_parents(), 32, 8, 128, 20480, 11, True),
        ([-1, 0, 1, 2], 40, 8, 128, 4096, 12, False),
    ]
    runs = []
    for parent, Hq, Hkv, d, N, seed, with_scores in cases:
        T = len(parent)
        q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=seed, device="cuda")
        assert ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N) > 0   # the split path really uses scratch
        runs.append((q, k, v, N, _mask(parent), Hq, d, with_scores, Hkv))
    # two no-alloc calls in a row on one stream
    got = []
    for q, k, v, N, mask, Hq, d, with_scores, Hkv in runs:
        out, lse = _outputs(q.shape[0], Hq, d)
        sc = torch.empty((Hkv, (N + 63) // 64), dtype=torch.float32, device="cuda") if with_scores else None
        _call_noalloc_cabi(q, k, v, N, mask, out, lse, sc, 1.0 / math.sqrt(d))
        got.append((out, lse, sc))
    torch.cuda.synchronize()
    for (q, k, v, N, mask, Hq, d, with_scores, Hkv), (out2, lse2, sc2) in zip(runs, got):
        out1, lse1 = _outputs(q.shape[0], Hq, d)
        sc1 = torch.empty_like(sc2) if sc2 is not None else None
        ws = torch.empty(ts.ts_tree_attn_workspace_bytes(q.shape[0], Hq, Hkv, d, N), dtype=torch.uint8,
                         device="cuda")
        ts.ts_tree_attn(q, k, v, N, mask, out1, lse=lse1, chunk_scores=sc1, workspace=ws)
        torch.cuda.synchronize()
        _close(out2, out1, "out")
        assert (lse2 - lse1).abs().max().item() <= LSE_ABS
        if sc2 is not None:
            assert torch.equal(sc2, sc1)


def test_noalloc_rejects_sizes_above_its_scratch():
    """Sizes whose split partials need more than the fixed array are refused
    before any pointer is read or any kernel is launched, and the message names
    the maximum.  A 4-row drafting batch over 400000 tokens splits into 1563
    ranges of 256 tokens: 1563 x 4 x 40 x 130 x 4 bytes, above 64 MiB."""
    from long_context_attention_tree_b300 import build
    build.build()
    T, Hq, Hkv, d, N = 4, 40, 8, 128, 400000
    need = ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N)
    assert need > ts.TS_NOALLOC_SCRATCH_BYTES
    L = ts.lib()
    P = ctypes.c_void_p(0x10000)
    st = L.ts_tree_attn_noalloc(P, P, P, N + T, N, T, Hq, Hkv, d, 0.088, P, P, None, None, 0, None)
    assert st == ts.TS_ERR_UNSUPPORTED
    assert str(ts.TS_NOALLOC_SCRATCH_BYTES).encode() in L.ts_last_error()
