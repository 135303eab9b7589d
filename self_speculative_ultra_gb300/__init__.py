"""GB300 (sm_103a) decode hot path of TokenSwift-style ultra-long generation.

Thin Python binding over the C-ABI library libtokenswift_gb300.so (see
include/tokenswift_gb300.h).  The functions carry the C names and only
marshal arguments: torch tensors supply device memory and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB_PATH, build  # noqa: F401

__all__ = [
    "TsError", "lib", "build", "ts_status_string", "ts_last_error", "ts_version",
    "ts_set_wait_limit",
    "ts_verify_workspace_bytes", "ts_verify_attention", "ts_importance_softmax",
    "ts_select_workspace_bytes", "ts_partial_kv_select_gather", "ts_partial_kv_select_gather_noalloc",
    "ts_select_batched_workspace_bytes", "ts_partial_kv_select_gather_batched", "layer_pointer_table",
    "ts_refresh_workspace_bytes", "ts_partial_kv_refresh_incremental",
    "ts_partial_kv_refresh_incremental_batched",
    "ts_sample_workspace_bytes", "ts_penalized_sample_accept", "ts_kv_commit",
    "ts_kv_commit_batched", "commit_pointer_table", "ts_kv_append_batched",
    "ts_reject_workspace_bytes", "ts_rejection_sample_accept",
]

TS_OK, TS_ERR_INVALID_ARG, TS_ERR_UNSUPPORTED, TS_ERR_CUDA, TS_ERR_TIMEOUT, TS_ERR_WORKSPACE = range(6)
TS_VERIFY_V_FP16 = 1     # ts_verify_attention_flags: the V cache holds fp16
TS_KV_V_FP16 = 1         # ts_kv_append_batched_flags: write V rows into fp16 caches

_c_void_p, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float

_SIGNATURES = {
    "ts_status_string": (ctypes.c_char_p, [_i32]),
    "ts_last_error": (ctypes.c_char_p, []),
    "ts_version": (_i32, []),
    "ts_set_wait_limit": (_i32, [_i64]),
    "ts_verify_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i64]),
    "ts_verify_attention": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _c_void_p,
                                   _i32, _i32, _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p,
                                   _c_void_p, _sz, _c_void_p, _c_void_p]),
    "ts_verify_attention_flags": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _c_void_p,
                                         _i32, _i32, _i32, _i32, _i32, _c_void_p, _c_void_p,
                                         _c_void_p, _c_void_p, _sz, _i32, _c_void_p, _c_void_p]),
    "ts_select_workspace_bytes": (_sz, [_i32, _i64]),
    "ts_importance_softmax": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i32, _i32, _i32,
                                     _i32, _i32, _c_void_p, _c_void_p, _c_void_p]),
    "ts_partial_kv_select_gather": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i32, _i32,
                                           _i32, _i32, _i32, _c_void_p, _c_void_p, _c_void_p,
                                           ctypes.POINTER(_i64), _c_void_p, _sz, _c_void_p,
                                           _c_void_p]),
    "ts_partial_kv_select_gather_noalloc": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64,
                                                   _i32, _i32, _i32, _i32, _i32, _c_void_p,
                                                   _c_void_p, _c_void_p, ctypes.POINTER(_i64),
                                                   _c_void_p, _c_void_p]),
    "ts_select_batched_workspace_bytes": (_sz, [_i32, _i32, _i64]),
    "ts_partial_kv_select_gather_batched": (_i32, [_i32, _c_void_p, _c_void_p, _c_void_p, _i64, _i64,
                                                   _i32, _i32, _i32, _i32, _i32, _c_void_p,
                                                   _c_void_p, _c_void_p, ctypes.POINTER(_i64),
                                                   _c_void_p, _sz, _c_void_p, _c_void_p]),
    "ts_sample_workspace_bytes": (_sz, [_i32, _i32]),
    "ts_refresh_workspace_bytes": (_sz, [_i32, _i32, _i64, _i64]),
    "ts_partial_kv_refresh_incremental": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i32,
                                                 _i32, _i32, _i32, _i32, _c_void_p, _c_void_p,
                                                 _c_void_p, _i64, _i64, ctypes.POINTER(_i64),
                                                 _c_void_p, _c_void_p, _sz, _c_void_p, _c_void_p]),
    "ts_partial_kv_refresh_incremental_batched": (_i32, [_i32, _c_void_p, _c_void_p, _c_void_p,
                                                         _i64, _i64, _i32, _i32, _i32, _i32, _i32,
                                                         _c_void_p, _c_void_p, _c_void_p, _i64,
                                                         _i64, ctypes.POINTER(_i64), _c_void_p,
                                                         _c_void_p, _sz, _c_void_p, _c_void_p]),
    "ts_penalized_sample_accept": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i32,
                                          _i32, _i32, _f32, _f32, _f32, _f32, _c_void_p,
                                          _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                          _c_void_p, _sz, _c_void_p, _c_void_p]),
    "ts_penalized_sample_accept_flags": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p,
                                                _i32, _i32, _i32, _f32, _f32, _f32, _f32,
                                                _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                                _c_void_p, _c_void_p, _sz, _i32, _c_void_p,
                                                _c_void_p]),
    "ts_penalized_sample_accept_eta": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p,
                                              _i32, _i32, _i32, _f32, _f32, _f32, _f32,
                                              _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                              _c_void_p, _c_void_p, _sz, _c_void_p, _c_void_p]),
    "ts_kv_commit": (_i32, [_c_void_p, _c_void_p, _i64, _i64, _i32, _i32, _i32, _c_void_p,
                            _c_void_p, _c_void_p, _c_void_p]),
    "ts_ngram_table_bytes": (_sz, [_i32, _i32]),
    "ts_kv_commit_batched": (_i32, [_i32, _c_void_p, _c_void_p, _i64, _i64, _i32, _i32, _i32,
                                    _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "ts_kv_append_batched": (_i32, [_i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64, _i64,
                                    _i32, _i32, _i32, _c_void_p]),
    "ts_kv_append_batched_flags": (_i32, [_i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64,
                                          _i64, _i32, _i32, _i32, _i32, _c_void_p, _c_void_p]),
    "ts_reject_workspace_bytes": (_sz, [_i32]),
    "ts_rejection_sample_accept": (_i32, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32,
                                          _c_void_p, _i32, _i32, _i32, _f32, _f32, _f32, _f32,
                                          _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                          _c_void_p, _sz, _i32, _c_void_p, _c_void_p]),
    "ts_ngram_insert": (_i32, [_c_void_p, _i32, _i32, _c_void_p, _i32, _i32, _c_void_p,
                               _c_void_p]),
    "ts_ngram_build_tree": (_i32, [_c_void_p, _i32, _i32, _c_void_p, _c_void_p, _i32, _i32, _i32,
                                   _c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                   _c_void_p]),
}

_LIB = None


class TsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built: call "
                               "self_speculative_ultra_gb300.build() first")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = h
    return _LIB


def ts_status_string(code: int) -> str:
    return lib().ts_status_string(code).decode()


def ts_last_error() -> str:
    return lib().ts_last_error().decode()


def ts_version() -> int:
    return lib().ts_version()


def ts_set_wait_limit(cycles: int) -> None:
    """Limit of one bounded device wait (SM clocks) for later launches;
    cycles <= 0 restores the default (~1 s)."""
    _check(lib().ts_set_wait_limit(int(cycles)))


def _check(rc: int):
    if rc != TS_OK:
        raise TsError(rc, f"{ts_status_string(rc)}: {ts_last_error()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# a V cache holds bf16 or fp16 values (fp16: the precision of the P.V product)
_V_DTYPES = (torch.bfloat16, torch.float16)


def _dev(t, dtype, name, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: {nbytes} bytes needed")
    return workspace, workspace.numel() * workspace.element_size()


def ts_verify_workspace_bytes(T, Hq, Hkv, d, L) -> int:
    return lib().ts_verify_workspace_bytes(T, Hq, Hkv, d, L)


def ts_verify_attention(q, k, v, L, parents, n_imp=0, o=None, lse=None, imp=None,
                        want_lse=True, want_imp=True, workspace=None, status=None, stream=None):
    """Tree verification attention + importance.  q [T,Hq,d] bf16, k
    [Hkv,L_cap,d] bf16, v [Hkv,L_cap,d] bf16 or fp16 (an fp16 V cache skips the
    kernel's per-tile conversion), parents [T] int32.  Returns (o, lse, imp)."""
    T, Hq, d = q.shape
    Hkv, L_cap = k.shape[0], k.shape[1]
    _dev(q, torch.bfloat16, "q")
    _dev(k, torch.bfloat16, "k", (Hkv, L_cap, d))
    _dev(v, _V_DTYPES, "v", (Hkv, L_cap, d))
    _dev(parents, torch.int32, "parents", (T,))
    dev = q.device
    if o is None:
        o = torch.empty((T, Hq, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    if imp is None and want_imp:
        imp = torch.empty((Hkv, L), dtype=torch.float32, device=dev)
    ws, nb = _workspace(ts_verify_workspace_bytes(T, Hq, Hkv, d, L), dev, workspace)
    flags = TS_VERIFY_V_FP16 if v.dtype == torch.float16 else 0
    rc = lib().ts_verify_attention_flags(_ptr(q), _ptr(k), _ptr(v), L, L_cap, _ptr(parents), T, Hq,
                                         Hkv, d, n_imp, _ptr(o), _ptr(lse), _ptr(imp), _ptr(ws), nb,
                                         flags, _ptr(status), _stream(stream))
    _check(rc)
    return o, lse, imp


def ts_importance_softmax(q, k, L, lse, n_imp=0, imp=None, status=None, stream=None):
    """Softmax-weighted importance of cache positions [0, L): for each KV head
    the attention probability its positions receive from the group's last
    n_imp tree queries.  q [T,Hq,d] bf16, k [Hkv,L_cap,d] bf16, lse [T,Hq]
    fp32 (from ts_verify_attention).  Returns imp [Hkv, L] fp32."""
    T, Hq, d = q.shape
    Hkv, L_cap = k.shape[0], k.shape[1]
    _dev(q, torch.bfloat16, "q")
    _dev(k, torch.bfloat16, "k", (Hkv, L_cap, d))
    _dev(lse, torch.float32, "lse", (T, Hq))
    if imp is None:
        imp = torch.empty((Hkv, L), dtype=torch.float32, device=q.device)
    rc = lib().ts_importance_softmax(_ptr(q), _ptr(k), _ptr(lse), L, L_cap, T, Hq, Hkv, d, n_imp,
                                     _ptr(imp), _ptr(status), _stream(stream))
    _check(rc)
    return imp


def ts_select_workspace_bytes(Hkv, L) -> int:
    return lib().ts_select_workspace_bytes(Hkv, L)


def ts_partial_kv_select_gather(imp, k, v, L, B, S, R, idx=None, kd=None, vd=None,
                                workspace=None, status=None, stream=None):
    """Top-B + sinks + recent selection and gather.  Returns (idx, kd, vd)."""
    Hkv, L_cap, d = k.shape
    _dev(imp, torch.float32, "imp", (Hkv, L))
    _dev(k, torch.bfloat16, "k")
    _dev(v, _V_DTYPES, "v", (Hkv, L_cap, d))
    N = min(L, S + B + R)
    dev = k.device
    if idx is None:
        idx = torch.empty((Hkv, N), dtype=torch.int32, device=dev)
    if kd is None:
        kd = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=dev)
    if vd is None:
        vd = torch.empty((Hkv, N, d), dtype=v.dtype, device=dev)
    ws, nb = _workspace(ts_select_workspace_bytes(Hkv, L), dev, workspace)
    n_out = _i64(0)
    rc = lib().ts_partial_kv_select_gather(_ptr(imp), _ptr(k), _ptr(v), L, L_cap, Hkv, d, B, S, R,
                                           _ptr(idx), _ptr(kd), _ptr(vd), ctypes.byref(n_out),
                                           _ptr(ws), nb, _ptr(status), _stream(stream))
    _check(rc)
    assert n_out.value == N
    return idx, kd, vd


def ts_partial_kv_select_gather_noalloc(imp, k, v, L, B, S, R, idx, kd, vd, status=None,
                                        stream=None):
    """Selection + gather without a workspace, for callers that may not
    allocate device memory: the library keeps its scratch in a fixed device
    array (see the C header for the size limit and the sharing rules).  The
    outputs idx [Hkv,N] int32, kd/vd [Hkv,N,d] bf16 are the caller's."""
    Hkv, L_cap, d = k.shape
    _dev(imp, torch.float32, "imp", (Hkv, L))
    _dev(k, torch.bfloat16, "k")
    _dev(v, _V_DTYPES, "v", (Hkv, L_cap, d))
    N = min(L, S + B + R)
    _dev(idx, torch.int32, "idx", (Hkv, N))
    _dev(kd, torch.bfloat16, "kd", (Hkv, N, d))
    _dev(vd, v.dtype, "vd", (Hkv, N, d))
    n_out = _i64(0)
    rc = lib().ts_partial_kv_select_gather_noalloc(_ptr(imp), _ptr(k), _ptr(v), L, L_cap, Hkv, d,
                                                   B, S, R, _ptr(idx), _ptr(kd), _ptr(vd),
                                                   ctypes.byref(n_out), _ptr(status),
                                                   _stream(stream))
    _check(rc)
    return idx, kd, vd


def ts_select_batched_workspace_bytes(n_layers, Hkv, L) -> int:
    return lib().ts_select_batched_workspace_bytes(n_layers, Hkv, L)


def layer_pointer_table(imps, ks, vs, idxs, kds, vds):
    """Device table [6, n_layers] of the per-layer tensor addresses the batched
    selection reads (build it once and reuse it while the tensors live)."""
    rows = [imps, ks, vs, idxs, kds, vds]
    n = len(imps)
    if any(len(r) != n for r in rows):
        raise ValueError("every per-layer list must have n_layers entries")
    host = torch.tensor([[t.data_ptr() for t in r] for r in rows], dtype=torch.int64)
    return host.to(imps[0].device)


def ts_partial_kv_select_gather_batched(imps, ks, vs, L, B, S, R, idxs, kds, vds, table=None,
                                        workspace=None, status=None, stream=None):
    """Selection + gather for several layers in one pipeline of launches.
    Lists of per-layer tensors with the single-layer shapes."""
    n = len(imps)
    Hkv, L_cap, d = ks[0].shape
    for i in range(n):
        _dev(imps[i], torch.float32, "imp", (Hkv, L))
        _dev(ks[i], torch.bfloat16, "k", (Hkv, L_cap, d))
        _dev(vs[i], _V_DTYPES, "v", (Hkv, L_cap, d))
    if table is None:
        table = layer_pointer_table(imps, ks, vs, idxs, kds, vds)
    ws, nb = _workspace(ts_select_batched_workspace_bytes(n, Hkv, L), ks[0].device, workspace)
    n_out = _i64(0)
    row = lambda r: ctypes.c_void_p(table[r].data_ptr())  # noqa: E731
    rc = lib().ts_partial_kv_select_gather_batched(n, row(0), row(1), row(2), L, L_cap, Hkv, d, B,
                                                   S, R, row(3), row(4), row(5), ctypes.byref(n_out),
                                                   _ptr(ws), nb, _ptr(status), _stream(stream))
    _check(rc)
    return idxs, kds, vds


def ts_refresh_workspace_bytes(n_layers, Hkv, L, N_cap) -> int:
    return lib().ts_refresh_workspace_bytes(n_layers, Hkv, L, N_cap)


def ts_partial_kv_refresh_incremental(imp, k, v, L, B, S, R, idx, kd, vd, N_prev, n_written=None,
                                      workspace=None, status=None, stream=None):
    """Update one layer's compact cache in place: slots whose position stays
    selected keep their row, newly selected positions fill the freed slots
    (then the new ones while the cache grows).  idx [Hkv, N_cap] int32,
    kd/vd [Hkv, N_cap, d] bf16 hold the previous state in slots [0, N_prev).
    Returns N_new (the slots now valid)."""
    Hkv, L_cap, d = k.shape
    _dev(imp, torch.float32, "imp", (Hkv, L))
    _dev(k, torch.bfloat16, "k")
    _dev(v, _V_DTYPES, "v", (Hkv, L_cap, d))
    N_cap = idx.shape[1]
    _dev(idx, torch.int32, "idx", (Hkv, N_cap))
    _dev(kd, torch.bfloat16, "kd", (Hkv, N_cap, d))
    _dev(vd, v.dtype, "vd", (Hkv, N_cap, d))
    ws, nb = _workspace(ts_refresh_workspace_bytes(1, Hkv, L, N_cap), k.device, workspace)
    n_out = _i64(0)
    rc = lib().ts_partial_kv_refresh_incremental(_ptr(imp), _ptr(k), _ptr(v), L, L_cap, Hkv, d, B,
                                                 S, R, _ptr(idx), _ptr(kd), _ptr(vd), N_cap,
                                                 N_prev, ctypes.byref(n_out), _ptr(n_written),
                                                 _ptr(ws), nb, _ptr(status), _stream(stream))
    _check(rc)
    return n_out.value


def ts_partial_kv_refresh_incremental_batched(imps, ks, vs, L, B, S, R, idxs, kds, vds, N_prev,
                                              table=None, n_written=None, workspace=None,
                                              status=None, stream=None):
    """The incremental refresh of several layers in one pipeline of launches
    (per-layer lists with the single-layer shapes).  Returns N_new."""
    n = len(imps)
    Hkv, L_cap, d = ks[0].shape
    N_cap = idxs[0].shape[1]
    for i in range(n):
        _dev(imps[i], torch.float32, "imp", (Hkv, L))
        _dev(ks[i], torch.bfloat16, "k", (Hkv, L_cap, d))
        _dev(vs[i], _V_DTYPES, "v", (Hkv, L_cap, d))
        _dev(idxs[i], torch.int32, "idx", (Hkv, N_cap))
        _dev(kds[i], torch.bfloat16, "kd", (Hkv, N_cap, d))
        _dev(vds[i], vs[i].dtype, "vd", (Hkv, N_cap, d))
    if table is None:
        table = layer_pointer_table(imps, ks, vs, idxs, kds, vds)
    ws, nb = _workspace(ts_refresh_workspace_bytes(n, Hkv, L, N_cap), ks[0].device, workspace)
    n_out = _i64(0)
    row = lambda r: ctypes.c_void_p(table[r].data_ptr())  # noqa: E731
    rc = lib().ts_partial_kv_refresh_incremental_batched(
        n, row(0), row(1), row(2), L, L_cap, Hkv, d, B, S, R, row(3), row(4), row(5), N_cap, N_prev,
        ctypes.byref(n_out), _ptr(n_written), _ptr(ws), nb, _ptr(status), _stream(stream))
    _check(rc)
    return n_out.value


def ts_sample_workspace_bytes(T, V) -> int:
    return lib().ts_sample_workspace_bytes(T, V)


TS_PENALTY_CTRL_LITERAL = 1


def ts_penalized_sample_accept(logits, tree_tokens, parents, prior, W, penalty, temperature,
                               top_p, min_p, uniforms, sampled=None, path=None, n_path=None,
                               bonus=None, workspace=None, status=None, stream=None,
                               literal=False):
    """Penalised top-p/min-p draw at every node + exact-match acceptance
    (literal=True: the literal CTRL penalty, every windowed logit divided).
    Returns (sampled [T], path [T], n_path [1], bonus [1]) device int32."""
    T, V = logits.shape
    _dev(logits, torch.float32, "logits")
    _dev(tree_tokens, torch.int32, "tree_tokens", (T,))
    _dev(parents, torch.int32, "parents", (T,))
    _dev(prior, torch.int32, "prior")
    _dev(uniforms, torch.float32, "uniforms", (T,))
    dev = logits.device
    mk = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    sampled = mk(T) if sampled is None else sampled
    path = mk(T) if path is None else path
    n_path = mk(1) if n_path is None else n_path
    bonus = mk(1) if bonus is None else bonus
    ws, nb = _workspace(ts_sample_workspace_bytes(T, V), dev, workspace)
    rc = lib().ts_penalized_sample_accept_flags(
        _ptr(logits), _ptr(tree_tokens), _ptr(parents), T, _ptr(prior), prior.numel(), W, V,
        penalty, temperature, top_p, min_p, _ptr(uniforms), _ptr(sampled), _ptr(path),
        _ptr(n_path), _ptr(bonus), _ptr(ws), nb, TS_PENALTY_CTRL_LITERAL if literal else 0,
        _ptr(status), _stream(stream))
    _check(rc)
    return sampled, path, n_path, bonus


def ts_penalized_sample_accept_eta(logits, tree_tokens, parents, prior, W, penalty, temperature,
                                   eta_epsilon, eta_alpha, uniforms, sampled=None, path=None,
                                   n_path=None, bonus=None, workspace=None, status=None,
                                   stream=None):
    """Penalised eta-sampling draw at every node + exact-match acceptance.
    Returns (sampled [T], path [T], n_path [1], bonus [1]) device int32."""
    T, V = logits.shape
    _dev(logits, torch.float32, "logits")
    _dev(tree_tokens, torch.int32, "tree_tokens", (T,))
    _dev(parents, torch.int32, "parents", (T,))
    _dev(prior, torch.int32, "prior")
    _dev(uniforms, torch.float32, "uniforms", (T,))
    dev = logits.device
    mk = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    sampled = mk(T) if sampled is None else sampled
    path = mk(T) if path is None else path
    n_path = mk(1) if n_path is None else n_path
    bonus = mk(1) if bonus is None else bonus
    ws, nb = _workspace(ts_sample_workspace_bytes(T, V), dev, workspace)
    rc = lib().ts_penalized_sample_accept_eta(_ptr(logits), _ptr(tree_tokens), _ptr(parents), T,
                                              _ptr(prior), prior.numel(), W, V, penalty,
                                              temperature, eta_epsilon, eta_alpha, _ptr(uniforms),
                                              _ptr(sampled), _ptr(path), _ptr(n_path), _ptr(bonus),
                                              _ptr(ws), nb, _ptr(status), _stream(stream))
    _check(rc)
    return sampled, path, n_path, bonus


def ts_kv_commit(k, v, L, T, path, n_path, status=None, stream=None):
    """Move the accepted tree rows L+path[t] to L+t (in place)."""
    Hkv, L_cap, d = k.shape
    _dev(k, torch.bfloat16, "k")
    _dev(v, _V_DTYPES, "v", (Hkv, L_cap, d))
    rc = lib().ts_kv_commit(_ptr(k), _ptr(v), L, L_cap, Hkv, d, T, _ptr(path), _ptr(n_path),
                            _ptr(status), _stream(stream))
    _check(rc)


def commit_pointer_table(ks, vs):
    """Device table [2, n_layers] of the per-layer K and V cache addresses the
    batched commit reads (build it once and reuse it while the caches live)."""
    if len(ks) != len(vs):
        raise ValueError("ks and vs must have one entry per layer")
    host = torch.tensor([[t.data_ptr() for t in ks], [t.data_ptr() for t in vs]],
                        dtype=torch.int64)
    return host.to(ks[0].device)


def ts_kv_commit_batched(ks, vs, L, T, path, n_path, table=None, status=None, stream=None):
    """ts_kv_commit for every layer in one launch (lists of per-layer caches
    [Hkv, L_cap, d] bf16)."""
    Hkv, L_cap, d = ks[0].shape
    for x, y in zip(ks, vs):
        _dev(x, torch.bfloat16, "k", (Hkv, L_cap, d))
        _dev(y, _V_DTYPES, "v", (Hkv, L_cap, d))
    if table is None:
        table = commit_pointer_table(ks, vs)
    rc = lib().ts_kv_commit_batched(len(ks), ctypes.c_void_p(table[0].data_ptr()),
                                    ctypes.c_void_p(table[1].data_ptr()), L, L_cap, Hkv, d, T,
                                    _ptr(path), _ptr(n_path), _ptr(status), _stream(stream))
    _check(rc)


def ts_kv_append_batched(ks, vs, k_rows, v_rows, L, table=None, status=None, stream=None):
    """Write the tree's K/V rows [L, L+T) into every layer's cache in one
    launch.  k_rows, v_rows [n_layers, Hkv, T, d] bf16 (contiguous); fp16 V
    caches receive the V rows rounded to fp16."""
    Hkv, L_cap, d = ks[0].shape
    n, T = len(ks), k_rows.shape[2]
    _dev(k_rows, torch.bfloat16, "k_rows", (n, Hkv, T, d))
    _dev(v_rows, torch.bfloat16, "v_rows", (n, Hkv, T, d))
    for x, y in zip(ks, vs):
        _dev(x, torch.bfloat16, "k", (Hkv, L_cap, d))
        _dev(y, _V_DTYPES, "v", (Hkv, L_cap, d))
    if table is None:
        table = commit_pointer_table(ks, vs)
    if len({y.dtype for y in vs}) != 1:
        raise TypeError("every layer's V cache must have the same dtype")
    flags = TS_KV_V_FP16 if vs[0].dtype == torch.float16 else 0
    rc = lib().ts_kv_append_batched_flags(n, ctypes.c_void_p(table[0].data_ptr()),
                                          ctypes.c_void_p(table[1].data_ptr()), _ptr(k_rows),
                                          _ptr(v_rows), L, L_cap, Hkv, d, T, flags, _ptr(status),
                                          _stream(stream))
    _check(rc)


def ts_reject_workspace_bytes(V) -> int:
    return lib().ts_reject_workspace_bytes(V)


def ts_rejection_sample_accept(logits, q, tree_tokens, parents, prior, W, penalty, temperature,
                               top_p, min_p, u_accept, u_draw, path=None, n_path=None, bonus=None,
                               workspace=None, status=None, stream=None, literal=False):
    """Speculative-sampling acceptance over the draft tree: children tried in
    index order against the draft distributions q [T, V].  Returns
    (path [T], n_path [1], bonus [1]) device int32."""
    T, V = logits.shape
    _dev(logits, torch.float32, "logits")
    _dev(q, torch.float32, "q", (T, V))
    _dev(tree_tokens, torch.int32, "tree_tokens", (T,))
    _dev(parents, torch.int32, "parents", (T,))
    _dev(prior, torch.int32, "prior")
    _dev(u_accept, torch.float32, "u_accept", (T,))
    _dev(u_draw, torch.float32, "u_draw", (T,))
    dev = logits.device
    mk = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    path = mk(T) if path is None else path
    n_path = mk(1) if n_path is None else n_path
    bonus = mk(1) if bonus is None else bonus
    ws, nb = _workspace(ts_reject_workspace_bytes(V), dev, workspace)
    rc = lib().ts_rejection_sample_accept(
        _ptr(logits), _ptr(q), _ptr(tree_tokens), _ptr(parents), T, _ptr(prior), prior.numel(), W,
        V, penalty, temperature, top_p, min_p, _ptr(u_accept), _ptr(u_draw), _ptr(path),
        _ptr(n_path), _ptr(bonus), _ptr(ws), nb, TS_PENALTY_CTRL_LITERAL if literal else 0,
        _ptr(status), _stream(stream))
    _check(rc)
    return path, n_path, bonus


def ts_ngram_table_bytes(V, cap) -> int:
    return lib().ts_ngram_table_bytes(V, cap)


def ngram_table(V, cap, device="cuda"):
    """A zeroed (empty) 4-gram table: int32 device buffer."""
    nb = ts_ngram_table_bytes(V, cap)
    if nb == 0:
        raise ValueError(f"unsupported table shape V={V}, cap={cap}")
    return torch.zeros(nb // 4, dtype=torch.int32, device=device)


def ts_ngram_insert(table, V, cap, tokens, start, n_tokens=None, status=None, stream=None):
    """Insert the 4-grams ending at positions start .. n_tokens-1 of tokens."""
    _dev(table, torch.int32, "table")
    _dev(tokens, torch.int32, "tokens")
    n = tokens.numel() if n_tokens is None else n_tokens
    _check(lib().ts_ngram_insert(_ptr(table), V, cap, _ptr(tokens), n, start, _ptr(status),
                                 _stream(stream)))


def ts_ngram_build_tree(table, V, cap, root_token, head_topk, k, rand_keys, T_max,
                        parents=None, tokens=None, n_nodes=None, status=None, stream=None):
    """Draft tree from the heads' candidates [n_heads, head_k] and the root's
    retrieved continuations.  Returns (parents [T_max], tokens [T_max],
    n_nodes [1]) device int32; entries past n_nodes are untouched."""
    _dev(table, torch.int32, "table")
    _dev(root_token, torch.int32, "root_token", (1,))
    _dev(head_topk, torch.int32, "head_topk")
    _dev(rand_keys, torch.int32, "rand_keys", (cap,))
    n_heads, head_k = head_topk.shape
    dev = table.device
    if parents is None:
        parents = torch.full((T_max,), -2, dtype=torch.int32, device=dev)
    if tokens is None:
        tokens = torch.full((T_max,), -2, dtype=torch.int32, device=dev)
    if n_nodes is None:
        n_nodes = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().ts_ngram_build_tree(_ptr(table), V, cap, _ptr(root_token), _ptr(head_topk),
                                     n_heads, head_k, k, _ptr(rand_keys), T_max, _ptr(parents),
                                     _ptr(tokens), _ptr(n_nodes), _ptr(status), _stream(stream)))
    return parents, tokens, n_nodes
