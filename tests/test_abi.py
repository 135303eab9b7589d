"""The C-ABI library builds, loads and exports every symbol its header
declares; host-side argument checks reject bad calls before any CUDA work
(CPU only: no call here reaches the GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tokenswift_gb300.h")


@pytest.fixture(scope="module")
def ts():
    import self_speculative_ultra_gb300 as ts
    ts.build()
    return ts


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(ts):
    names = _declared()
    assert "ts_verify_attention" in names and "ts_kv_commit" in names
    h = ctypes.CDLL(ts.LIB_PATH)
    for n in names:
        assert hasattr(h, n), n


def test_status_strings_and_version(ts):
    assert ts.ts_status_string(0) == "ok"
    assert "workspace" in ts.ts_status_string(5)
    assert ts.ts_version() >= 100


def test_workspace_queries(ts):
    assert ts.ts_verify_workspace_bytes(64, 32, 8, 128, 102400) > 0
    assert ts.ts_verify_workspace_bytes(65, 32, 8, 128, 102400) == 0
    assert ts.ts_select_workspace_bytes(8, 102400) > 0
    assert ts.ts_sample_workspace_bytes(64, 128256) >= 64 * 128256 * 4


def _c(ts):
    return ts.lib()


def test_verify_rejects_bad_shapes(ts):
    f = _c(ts).ts_verify_attention
    p = ctypes.c_void_p(16)
    # T = 0
    assert f(p, p, p, 10, 100, p, 0, 4, 1, 64, 0, p, None, None, None, 0, None, None) == 1
    # T > 64
    assert f(p, p, p, 10, 100, p, 65, 4, 1, 64, 0, p, None, None, None, 0, None, None) == 2
    # Hq not a multiple of Hkv
    assert f(p, p, p, 10, 100, p, 4, 5, 2, 64, 0, p, None, None, None, 0, None, None) == 1
    # head dim 96 unsupported
    assert f(p, p, p, 10, 100, p, 4, 4, 1, 96, 0, p, None, None, None, 0, None, None) == 2
    # L + T > L_cap
    assert f(p, p, p, 98, 100, p, 4, 4, 1, 64, 0, p, None, None, None, 0, None, None) == 1
    # missing workspace
    assert f(p, p, p, 10, 100, p, 4, 4, 1, 64, 0, p, None, None, None, 0, None, None) == 5
    assert "workspace" in ts.ts_last_error()
    # misaligned workspace
    assert f(p, p, p, 10, 100, p, 4, 4, 1, 64, 0, p, None, None, ctypes.c_void_p(8), 1 << 30,
             None, None) == 5


def test_select_and_sample_reject_bad_args(ts):
    p = ctypes.c_void_p(16)
    g = _c(ts).ts_partial_kv_select_gather
    n = ctypes.c_int64(-1)
    assert g(p, p, p, 10, 5, 1, 128, 4, 4, 64, p, p, p, ctypes.byref(n), None, 0, None, None) == 1
    assert g(p, p, p, 0, 5, 1, 128, 4, 4, 64, p, p, p, ctypes.byref(n), None, 0, None, None) == 0
    assert n.value == 0
    s = _c(ts).ts_penalized_sample_accept
    args = [p, p, p, 4, p, 10, 10, 100, 1.2, 1.0, 0.9, 0.05, p, p, p, p, p, None, 0, None, None]
    bad = list(args); bad[9] = 0.0          # temperature 0
    assert s(*bad) == 1
    bad = list(args); bad[7] = 300000       # V too large
    assert s(*bad) == 2
    bad = list(args); bad[10] = 0.0         # top_p 0
    assert s(*bad) == 1
    assert s(*args) == 5                    # no workspace
    c = _c(ts).ts_kv_commit
    assert c(p, p, 10, 12, 1, 128, 4, p, p, None, None) == 1


def test_importance_softmax_rejects_bad_args(ts):
    f = _c(ts).ts_importance_softmax
    p = ctypes.c_void_p(16)
    # NULL lse (with a non-empty cache)
    assert f(p, p, None, 10, 100, 4, 4, 1, 64, 0, p, None, None) == 1
    # an empty cache needs no buffers
    assert f(p, p, None, 0, 100, 4, 4, 1, 64, 0, None, None, None) == 0
    # L > L_cap
    assert f(p, p, p, 101, 100, 4, 4, 1, 64, 0, p, None, None) == 1
    # n_imp > T
    assert f(p, p, p, 10, 100, 4, 4, 1, 64, 5, p, None, None) == 1
    # head dim 96
    assert f(p, p, p, 10, 100, 4, 4, 1, 96, 0, p, None, None) == 2
    # 64 nodes x 8 heads per group = 512 query rows do not fit one SM at d = 128
    assert f(p, p, p, 10, 100, 64, 8, 1, 128, 0, p, None, None) == 2
    assert "shared memory" in ts.ts_last_error()
    # 448 rows fit: the call passes the checks; L = 0 launches nothing
    assert f(p, p, p, 0, 100, 56, 8, 1, 128, 0, p, None, None) == 0


def test_sample_flags_reject_unknown_bits(ts):
    p = ctypes.c_void_p(16)
    f = _c(ts).ts_penalized_sample_accept_flags
    assert f(p, p, p, 4, p, 8, 8, 100, 1.2, 1.0, 0.9, 0.05, p, p, p, p, p, p, 1 << 30, 4,
             None, None) == 1
    assert "flags" in ts.ts_last_error()


def test_verify_and_append_flags_reject_unknown_bits(ts):
    """The fp16-V flag variants reject flag bits they do not define, on the
    host, before anything is enqueued."""
    p = ctypes.c_void_p(16)
    lib = _c(ts)
    f = lib.ts_verify_attention_flags
    assert f(p, p, p, 100, 200, p, 4, 8, 2, 128, 0, p, p, p, p, 1 << 20, 1 << 7, None,
             None) == 1
    assert "flags" in ts.ts_last_error()
    g = lib.ts_kv_append_batched_flags
    assert g(1, p, p, p, p, 100, 200, 2, 128, 4, 1 << 3, None, None) == 1
    assert "flags" in ts.ts_last_error()


def test_binding_signatures_match_the_header(ts):
    """Every function the header declares has a ctypes signature in the
    binding with the same number of parameters."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = dict(re.findall(r"\b(ts_[a-z_]+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S))
    assert decls, "no declarations parsed"
    for name, params in decls.items():
        assert name in ts._SIGNATURES, f"{name} has no ctypes signature"
        p = params.strip()
        n = 0 if p in ("", "void") else p.count(",") + 1
        assert len(ts._SIGNATURES[name][1]) == n, (name, n, len(ts._SIGNATURES[name][1]))


def test_rejection_call_rejects_bad_args(ts):
    p = ctypes.c_void_p(16)
    f = _c(ts).ts_rejection_sample_accept
    # more than 64 tree nodes
    assert f(p, p, p, p, 65, p, 8, 8, 1000, 1.2, 1.0, 0.9, 0.05, p, p, p, p, p, p, 1 << 30, 0,
             None, None) == 2
    # a top-p cut without min-p over a large vocabulary passes the argument
    # checks; the misaligned workspace (address 16) is then rejected
    assert f(p, p, p, p, 4, p, 8, 8, 100000, 1.2, 1.0, 0.9, 0.0, p, p, p, p, p, p, 1 << 30, 0,
             None, None) == 5
    # unknown flag bits
    assert f(p, p, p, p, 4, p, 8, 8, 1000, 1.2, 1.0, 0.9, 0.05, p, p, p, p, p, p, 1 << 30, 8,
             None, None) == 1
    assert ts.ts_reject_workspace_bytes(128256) >= 128256 * 4
