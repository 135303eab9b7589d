"""GPU parity for draft-side attention over the compact cache: the drafting
pass attends to the partial KV cache (sinks + top-B + recent rows) followed by
the draft tokens' own rows.  The library path is ts_partial_kv_select_gather
then ts_verify_attention with a short draft chain (T = 1..4) over the gathered
rows; the oracle runs its own selection, gather and attention on the same
seeded inputs."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _draft(name, L, T_d, seed=0, v_fp16=False):
    import self_speculative_ultra_gb300 as ts
    w = syn.WORKLOADS[name]
    inp = syn.attention_inputs(w, L=L)
    Hkv, d = inp["k"].shape[0], inp["k"].shape[2]
    imp = syn.importance_scores(Hkv, L, seed)
    chain = np.array([-1] + list(range(T_d - 1)), dtype=np.int32)
    # library: select + gather, then attention over [compact rows ; draft rows]
    k, v = pu.to_dev_bf16(inp["k"]), pu.to_dev_bf16(inp["v"])
    if v_fp16:
        v = v.to(torch.float16)   # the same values: the compact V rows and the call are fp16
    idx, kd, vd = ts.ts_partial_kv_select_gather(pu.to_dev(imp), k, v, L, w.B, w.S, w.R)
    N = idx.shape[1]
    k_ext = torch.cat([kd, k[:, L:L + T_d]], dim=1).contiguous()
    v_ext = torch.cat([vd, v[:, L:L + T_d]], dim=1).contiguous()
    q = pu.to_dev_bf16(inp["q"][:T_d])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, _ = ts.ts_verify_attention(q, k_ext, v_ext, N, pu.to_dev(chain), n_imp=T_d,
                                       want_imp=False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: its own selection and gather on the same inputs
    kc, vc = [], []
    for h in range(Hkv):
        ref = orc.select_partial(imp[h].astype(np.float64), L, w.B, w.S, w.R)
        np.testing.assert_array_equal(idx[h].cpu().numpy(), ref)
        kc.append(orc.gather_rows(inp["k"][h], ref))
        vc.append(orc.gather_rows(inp["v"][h], ref))
    k64 = orc.bf16_to_f64(np.concatenate([np.stack(kc), inp["k"][:, L:L + T_d]], axis=1))
    v64 = orc.bf16_to_f64(np.concatenate([np.stack(vc), inp["v"][:, L:L + T_d]], axis=1))
    q64 = orc.bf16_to_f64(inp["q"][:T_d])
    O, LSE, _ = orc.verify_attention(q64, k64, v64, N, chain, T_d)
    pu.check_attention(o.cpu().numpy(), lse.cpu().numpy(), O, LSE)
    return N


@pytest.mark.parametrize("name", ["llama3.1-8b", "qwen2.5-1.5b", "mha-7b"])
@pytest.mark.parametrize("T_d", [1, 4])
def test_draft_attention_over_compact_cache(name, T_d):
    N = _draft(name, 20000, T_d)
    w = syn.WORKLOADS[name]
    assert N == w.S + w.B + w.R


@pytest.mark.parametrize("name", ["llama3.1-8b", "qwen2.5-14b"])
def test_draft_attention_fp16_v_cache(name):
    """fp16 V caches through the gather and the draft attention."""
    w = syn.WORKLOADS[name]
    assert _draft(name, 20000, 4, v_fp16=True) == w.S + w.B + w.R


def test_draft_attention_cache_within_budget():
    """L <= S+B+R: the compact cache is the whole cache."""
    assert _draft("tiny", 900, 3) == 900
