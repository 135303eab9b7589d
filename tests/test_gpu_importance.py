"""GPU parity: softmax-weighted importance (ts_importance_softmax) against the
oracle.

Two comparisons per case:
  * same normaliser: the oracle evaluates the definition with the lse values
    the library's verification returned (fp32, carried as float64), so only
    the importance pass itself is compared.  Bound: every term
    exp(s - lse) is positive, so the sum's relative error is at most the
    worst term's: the fp32 score error (at most d * 2^-24 * |q| |k| / sqrt(d)
    for a d-term dot product; |q|, |k| <= ~sqrt(2 d) here, ~1.5e-4 at
    d = 128 in the worst case, far less in practice) plus the exponent's
    rounding (~1e-6).  IMP_RTOL = 2e-4.
  * end to end: against the oracle's own fp64 LSE.  The library's lse is
    within 2e-3 of it (the attention tolerance), which moves every term by a
    factor within exp(+-2e-3): rtol 2.5e-3.
"""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu

IMP_RTOL = 2e-4
E2E_RTOL = 2.5e-3


def _check(got, ref, rtol, what):
    err = np.abs(got.astype(np.float64) - ref)
    bad = err > rtol * ref + 1e-30
    assert not bad.any(), (f"{what}: {int(bad.sum())} positions off, worst rel "
                           f"{float((err / np.maximum(ref, 1e-30)).max()):.3e}")
    return float((err / np.maximum(ref, 1e-30)).max())


def _run(w, L=None, n_imp=None, layer=0, tree=None, n_sample=None):
    import self_speculative_ultra_gb300 as ts
    inp = syn.attention_inputs(w, layer=layer, L=L, tree=tree)
    L = inp["L"]
    n_imp = w.n_imp if n_imp is None else n_imp
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    parents = pu.to_dev(inp["parents"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, lse, _ = ts.ts_verify_attention(q, k, v, L, parents, n_imp=n_imp, want_imp=False,
                                       status=status)
    imp = ts.ts_importance_softmax(q, k, L, lse, n_imp=n_imp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    imp = imp.cpu().numpy()
    q64 = orc.bf16_to_f64(inp["q"])
    lse_lib = lse.cpu().numpy().astype(np.float64)
    if n_sample is None:
        k64 = orc.bf16_to_f64(inp["k"])
        ref = orc.importance_softmax(q64, k64, L, lse_lib, n_imp)
        worst = _check(imp, ref, IMP_RTOL, "same normaliser")
        v64 = orc.bf16_to_f64(inp["v"])
        _, LSE, _ = orc.verify_attention(q64, k64, v64, L, inp["parents"], n_imp)
        _check(imp, orc.importance_softmax(q64, k64, L, LSE, n_imp), E2E_RTOL, "end to end")
        return worst
    # full-size cache: the definition is per position, so the oracle runs on a
    # sample of positions (every planted heavy hitter, the first and last
    # tiles, random positions); the result must also carry the mass property
    rng = np.random.default_rng(11)
    worst = 0.0
    for kv in range(w.Hkv):
        pos = np.unique(np.concatenate([inp["planted"][kv], np.arange(0, 200),
                                        np.arange(L - 200, L),
                                        rng.integers(0, L, size=n_sample)]))
        k_sub = orc.bf16_to_f64(inp["k"][kv:kv + 1, pos])
        q_sub = q64[:, kv * w.G:(kv + 1) * w.G]
        ref = orc.importance_softmax(q_sub, k_sub, len(pos), lse_lib[:, kv * w.G:(kv + 1) * w.G],
                                     n_imp)[0]
        worst = max(worst, _check(imp[kv, pos], ref, IMP_RTOL, f"head {kv}"))
        # each importance row's weights sum to at most 1 over the cache
        assert imp[kv].sum() <= n_imp * w.G * (1 + 1e-4)
    return worst


def test_tiny_full():
    _run(syn.WORKLOADS["tiny"])


@pytest.mark.parametrize("name", ["qwen2.5-1.5b", "llama3.1-8b", "mha-7b", "qwen2.5-14b"])
@pytest.mark.parametrize("L", [1000, 4133])
def test_configs_small_cache(name, L):
    """Every model shape (256, 320 and 384 importance rows: one and two row
    chunks), caches spanning several tiles and splits with a ragged tail."""
    _run(syn.WORKLOADS[name], L=L)


@pytest.mark.parametrize("L", [1, 127, 128, 129, 300])
def test_edge_cache_lengths(L):
    _run(syn.scaled(syn.WORKLOADS["tiny"], planted=0), L=L)


def test_empty_cache_launches_nothing():
    import self_speculative_ultra_gb300 as ts
    q = torch.zeros((16, 4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 16, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((16, 4), dtype=torch.float32, device="cuda")
    imp = ts.ts_importance_softmax(q, k, 0, lse)
    assert imp.shape == (1, 0)


@pytest.mark.parametrize("n_imp", [1, 5, 33])
def test_partial_importance_queries(n_imp):
    _run(syn.WORKLOADS["llama3.1-8b"], L=2500, n_imp=n_imp)


def test_single_node_tree():
    _run(syn.scaled(syn.WORKLOADS["tiny"], T=1, n_imp=1), L=777)


@pytest.mark.parametrize("name", ["llama3.1-8b", "qwen2.5-14b"])
def test_full_size_one_layer(name):
    """Full 100K cache in the launch configuration the benchmark times,
    checked on sampled positions."""
    _run(syn.WORKLOADS[name], layer=2, n_sample=3000)
