"""Failure paths, exercised without faulting, trapping or hanging the GPU.

* A bounded device-side wait that gives up: one warp waits on an mbarrier that
  no thread arrives at, its wait runs out after a few microseconds, the sticky
  status reads TS_ERR_TIMEOUT, clears, and the next attention call is correct.
* A failing kernel launch, injected on the host: the library's launch reports
  cudaErrorInvalidValue without launching, the call returns TS_ERR_CUDA with
  the CUDA error named, and nothing else is left behind.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import long_context_attention_tree_b300 as ts
from long_context_attention_tree_b300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_attention_tree_b300 import build
    build.build()
    yield
    ts.ts_selftest_fail_launches(0)


def test_injected_launch_failure_is_reported_on_the_host():
    """No GPU needed: the injected failure is taken before any launch (a batch
    for the CUDA-core kernel that needs no tensor map)."""
    L = ts.lib()
    P = ctypes.c_void_p(0x10000)
    ts.ts_selftest_fail_launches(1)
    st = L.ts_tree_attn(P, P, P, 4100, 4000, 30, 40, 8, 128, 0.088, P, P, None, None, 0, P, 1 << 30, None)
    assert st == ts.TS_ERR_CUDA
    assert b"cudaErrorInvalidValue" in L.ts_last_error() and b"launch" in L.ts_last_error()
    ts.ts_selftest_fail_launches(0)


def test_bounded_wait_rejects_bad_budget():
    L = ts.lib()
    assert L.ts_selftest_bounded_wait(0, None) == ts.TS_ERR_INVALID_ARG
    assert L.ts_selftest_bounded_wait(2_000_000_000, None) == ts.TS_ERR_INVALID_ARG


def _attn_case():
    import oracle
    T, Hq, Hkv, d, N = 120, 40, 8, 128, 3000
    q, k, v = W.make_qkv(T, Hq, Hkv, d, N, seed=99, device="cuda")
    parent = W.verify_parents()
    mask = torch.from_numpy(ts.ts_tree_mask_from_parents(parent).view(np.int64)).cuda()
    out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N)), dtype=torch.uint8, device="cuda")
    ro, _ = oracle.tree_attn(q.cpu(), k.cpu(), v.cpu(), N, parent, 1 / math.sqrt(d))
    return q, k, v, N, mask, out, ws, ro


def _assert_close(out, ro):
    o = out.float().cpu().double().numpy()
    assert np.abs(o - ro).max() <= 2e-2
    assert np.linalg.norm(o - ro) / np.linalg.norm(ro) <= 1e-2


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_the_context_stays_usable():
    assert ts.ts_device_error(True) == ts.TS_OK
    ts.ts_selftest_bounded_wait(20_000)   # 20 us
    torch.cuda.synchronize()
    assert ts.ts_device_error(False) == ts.TS_ERR_TIMEOUT   # sticky until cleared
    assert ts.ts_device_error(True) == ts.TS_ERR_TIMEOUT
    assert ts.ts_device_error(True) == ts.TS_OK
    q, k, v, N, mask, out, ws, ro = _attn_case()
    ts.ts_tree_attn(q, k, v, N, mask, out, workspace=ws)
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK
    _assert_close(out, ro)


@pytest.mark.gpu
def test_injected_launch_failure_then_a_clean_call():
    q, k, v, N, mask, out, ws, ro = _attn_case()
    out.fill_(0)
    n0 = ts.ts_launch_count()
    ts.ts_selftest_fail_launches(1)
    with pytest.raises(ts.TSError) as e:
        ts.ts_tree_attn(q, k, v, N, mask, out, workspace=ws)
    assert e.value.status == ts.TS_ERR_CUDA and "cudaErrorInvalidValue" in str(e.value)
    torch.cuda.synchronize()
    assert ts.ts_launch_count() == n0 and bool((out == 0).all())   # nothing ran
    ts.ts_tree_attn(q, k, v, N, mask, out, workspace=ws)           # the next call launches
    torch.cuda.synchronize()
    assert ts.ts_device_error(True) == ts.TS_OK
    _assert_close(out, ro)
