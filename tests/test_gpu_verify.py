"""GPU parity: tree verification attention + importance (ts_verify_attention)
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _run(w, L=None, layer=0, n_imp=None, tree=None):
    import self_speculative_ultra_gb300 as ts
    inp = syn.attention_inputs(w, layer=layer, L=L, tree=tree)
    L = inp["L"]
    n_imp = w.n_imp if n_imp is None else n_imp
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    parents = pu.to_dev(inp["parents"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, imp = ts.ts_verify_attention(q, k, v, L, parents, n_imp=n_imp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    q64, k64, v64 = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    O, LSE, IMP = orc.verify_attention(q64, k64, v64, L, inp["parents"], n_imp)
    rel = pu.check_attention(o.cpu().numpy(), lse.cpu().numpy(), O, LSE)
    pu.check_importance(imp.cpu().numpy(), IMP, q64, k64, n_imp, w.G)
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


@pytest.mark.parametrize("name", ["llama3.1-8b", "qwen2.5-14b"])
def test_full_size_one_layer(name):
    """Full 100K cache, the launch configuration the benchmark times."""
    _run(syn.WORKLOADS[name], layer=1)


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


@pytest.mark.parametrize("L", [1000, 4133, 102400])
def test_cta_pair_kernel(L):
    """The opt-in CTA-pair (tcgen05 .cta_group::2) kernel for M = T*G = 256,
    d = 128 against the oracle, in a child process with TS_VERIFY_PAIR=1."""
    import os
    import subprocess
    import sys
    code = ("import sys; sys.path[:0] = ['tests', '.']\n"
            "import test_gpu_verify as t, ts_synth as syn\n"
            f"t._run(syn.WORKLOADS['llama3.1-8b'], L={L}, layer=1)\n"
            "print('ok')\n")
    env = dict(os.environ, TS_VERIFY_PAIR="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
