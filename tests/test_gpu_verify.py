"""GPU parity: tree verification attention + importance (ts_verify_attention)
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _run(w, L=None, layer=0, n_imp=None, tree=None, kv_heads=None, v_fp16=False):
    """Run the library on all heads; compare the KV heads `kv_heads` (all by
    default) and their query heads element by element with the oracle.
    v_fp16: the V cache is handed over in fp16 (the same values: the
    synthetic bf16 values convert exactly, subnormals rounding to nearest)."""
    import self_speculative_ultra_gb300 as ts
    inp = syn.attention_inputs(w, layer=layer, L=L, tree=tree)
    L = inp["L"]
    n_imp = w.n_imp if n_imp is None else n_imp
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    if v_fp16:
        v = v.to(torch.float16)
    parents = pu.to_dev(inp["parents"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, imp = ts.ts_verify_attention(q, k, v, L, parents, n_imp=n_imp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o, lse, imp = o.cpu().numpy(), lse.cpu().numpy(), imp.cpu().numpy()
    del q, k, v
    kvs = list(range(w.Hkv)) if kv_heads is None else list(kv_heads)
    hq = [kv * w.G + g for kv in kvs for g in range(w.G)]
    q64 = orc.bf16_to_f64(inp["q"][:, hq])
    k64, v64 = (orc.bf16_to_f64(inp[n][kvs]) for n in ("k", "v"))
    O, LSE, IMP = orc.verify_attention(q64, k64, v64, L, inp["parents"], n_imp)
    rel = pu.check_attention(o[:, hq], lse[:, hq], O, LSE)
    pu.check_importance(imp[kvs], IMP, q64, k64, n_imp, w.G)
    return rel


def test_tiny_full():
    _run(syn.WORKLOADS["tiny"])


@pytest.mark.parametrize("name", ["qwen2.5-1.5b", "llama3.1-8b", "mha-7b", "qwen2.5-14b"])
@pytest.mark.parametrize("L", [1000, 4133])
def test_configs_small_cache(name, L):
    """Every model shape, caches spanning several tiles with a ragged tail."""
    _run(syn.WORKLOADS[name], L=L)


@pytest.mark.parametrize("L", [0, 1, 63, 64, 65])
def test_edge_cache_lengths(L):
    _run(syn.scaled(syn.WORKLOADS["tiny"], planted=0), L=L)


def test_single_node_tree():
    w = syn.scaled(syn.WORKLOADS["tiny"], T=1, n_imp=1)
    _run(w, L=777)


def test_chain_tree_and_partial_importance():
    w = syn.scaled(syn.WORKLOADS["llama3.1-8b"], T=64)
    parents = np.array([-1] + list(range(63)), dtype=np.int32)
    _run(w, L=3000, n_imp=5, tree=(parents, np.zeros(64, np.int32)))


@pytest.mark.parametrize("name,kv_heads,v_fp16", [("llama3.1-8b", None, False),
                                                  ("llama3.1-8b", None, True),
                                                  ("qwen2.5-14b", None, True),
                                                  ("qwen2.5-1.5b", None, True),
                                                  ("mha-7b", (0, 13, 31), True)])
def test_full_size_one_layer(name, kv_heads, v_fp16):
    """Every model shape at its full cache length (102,400 tokens; 32,768 for
    Qwen2.5-1.5B), the launch configuration the benchmark times (an fp16 V
    cache; LLaMA3.1-8B also with the bf16 one).  For the 32-head MHA shape
    three KV heads (first, middle, last) are compared in full against the
    oracle; the others are computed by the same launch."""
    _run(syn.WORKLOADS[name], layer=1, kv_heads=kv_heads, v_fp16=v_fp16)


@pytest.mark.parametrize("name", ["tiny", "qwen2.5-1.5b", "llama3.1-8b", "mha-7b", "qwen2.5-14b"])
def test_fp16_v_cache_is_bit_identical(name):
    """An fp16 V cache only moves the bf16 -> fp16 rounding of V from the
    kernel's shared memory to the cache: on the same values every output
    (O, LSE, importance) is bit for bit that of the bf16 call."""
    import self_speculative_ultra_gb300 as ts
    w = syn.WORKLOADS[name]
    inp = syn.attention_inputs(w, L=4133)
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    parents = pu.to_dev(inp["parents"])
    outs = []
    for vv in (v, v.to(torch.float16)):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(ts.ts_verify_attention(q, k, vv, 4133, parents, n_imp=w.n_imp, status=status))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name,T,L", [("llama3.1-8b", 4, 0), ("llama3.1-8b", 4, 65),
                                      ("llama3.1-8b", 8, 4133), ("qwen2.5-1.5b", 5, 3000),
                                      ("mha-7b", 8, 6000), ("tiny", 8, 777)])
def test_draft_sized_calls_match_oracle(name, T, L):
    """At most 32 packed rows per KV head over a short cache (the draft-side
    shape: a 128-row tile that is mostly padding): attention and importance
    against the oracle, random trees of T nodes, caches from empty to several
    splits, bf16 and fp16 V caches."""
    w = syn.scaled(syn.WORKLOADS[name], T=T, n_imp=T, planted=0 if L < 300 else None)
    if w.planted is None:
        w = syn.scaled(syn.WORKLOADS[name], T=T, n_imp=T)
    _run(w, L=L)
    _run(w, L=L, v_fp16=True)


def test_bad_parent_sets_status():
    import self_speculative_ultra_gb300 as ts
    w = syn.scaled(syn.WORKLOADS["tiny"], planted=0)
    inp = syn.attention_inputs(w, L=100)
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    par = inp["parents"].copy()
    par[5] = 9   # not an earlier node
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_verify_attention(q, k, v, 100, pu.to_dev(par), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1


def test_value_beyond_fp16_range_is_reported():
    """P.V runs in fp16: a V entry of 1e5 cannot be represented, and the call
    reports TS_ERR_UNSUPPORTED (2) in the status word instead of failing
    silently."""
    import self_speculative_ultra_gb300 as ts
    w = syn.scaled(syn.WORKLOADS["tiny"], planted=0)
    inp = syn.attention_inputs(w, L=300)
    vb = inp["v"].copy()
    vb[0, 17, 5] = syn.f32_to_bf16_bits(np.array([1e5], np.float32))[0]
    q, k, v = pu.to_dev_bf16(inp["q"]), pu.to_dev_bf16(inp["k"]), pu.to_dev_bf16(vb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_verify_attention(q, k, v, 300, pu.to_dev(inp["parents"]), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2
