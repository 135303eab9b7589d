"""The allocation-free selection entry point (ts_partial_kv_select_gather_noalloc)
gives exactly the results of the workspace entry point.

It serves callers that may not allocate device memory (a plugin inside a host
runtime that owns every allocation, a serving loop that forbids allocation once
running): its scratch is a fixed device array inside the library, shared by
every call on a device.  Two calls in a row with different inputs check that
what one call leaves in that shared array does not leak into the next.  The
calls go straight through the C ABI.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import ts_synth as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import self_speculative_ultra_gb300 as ts
    ts.build()
    return ts


def _inputs(Hkv, L, d, seed, grid=None):
    imp = syn.importance_scores(Hkv, L, seed, grid=grid)
    rng = np.random.default_rng(seed)
    kb = rng.integers(0, 2 ** 16, size=(Hkv, L + 8, d), dtype=np.uint16)
    vb = rng.integers(0, 2 ** 16, size=(Hkv, L + 8, d), dtype=np.uint16)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    bf = lambda a: dev(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    return dev(imp), bf(kb), bf(vb)


def _noalloc_call(ts, imp, k, v, L, B, S, R):
    Hkv, L_cap, d = k.shape
    N = min(L, S + B + R)
    idx = torch.full((Hkv, N), -7, dtype=torch.int32, device="cuda")
    kd = torch.zeros((Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros((Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_out = ctypes.c_int64(0)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = ts.lib().ts_partial_kv_select_gather_noalloc(
        p(imp), p(k), p(v), L, L_cap, Hkv, d, B, S, R, p(idx), p(kd), p(vd), ctypes.byref(n_out),
        p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, n_out.value, idx, kd, vd, status


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(ts):
    cases = [(8, 102400, 4096, 4, 64, 11, None), (3, 20000, 3000, 4, 64, 12, 1.0)]
    for Hkv, L, B, S, R, seed, grid in cases:
        imp, k, v = _inputs(Hkv, L, 128, seed, grid)
        rc, n, idx, kd, vd, status = _noalloc_call(ts, imp, k, v, L, B, S, R)
        torch.cuda.synchronize()
        assert rc == 0, ts.ts_last_error()
        assert n == min(L, S + B + R) and int(status.item()) == 0
        i1, k1, v1 = ts.ts_partial_kv_select_gather(imp, k, v, L, B, S, R)
        torch.cuda.synchronize()
        assert torch.equal(idx, i1)
        assert torch.equal(kd.view(torch.int16), k1.view(torch.int16))
        assert torch.equal(vd.view(torch.int16), v1.view(torch.int16))


def test_noalloc_rejects_shapes_beyond_its_scratch(ts):
    imp, k, v = _inputs(16, 102400, 64, 13)
    rc, _, _, _, _, _ = _noalloc_call(ts, imp, k, v, 102400, 4096, 4, 64)
    assert rc == 2
    assert "fixed array" in ts.ts_last_error()
