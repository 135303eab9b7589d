"""GPU: a bounded device wait that runs out (failure detection without a
GPU fault).  With a wait limit of a few dozen clocks the verification kernel
gives up its first wait on another warp, writes TS_ERR_TIMEOUT (4) into the
status word, waits for its own copies and tensor-core work in flight, frees
its tensor memory and returns; the context stays usable and the next call,
with the default limit, matches the oracle."""
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _call(ts, w, inp, status):
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    out = ts.ts_verify_attention(q, k, v, inp["L"], pu.to_dev(inp["parents"]), n_imp=w.n_imp,
                                 status=status)
    torch.cuda.synchronize()
    return out


def test_expired_wait_reports_timeout_then_next_call_matches_oracle():
    import self_speculative_ultra_gb300 as ts
    w = syn.WORKLOADS["tiny"]
    inp = syn.attention_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_set_wait_limit(64)
    try:
        _call(ts, w, inp, status)
    finally:
        ts.ts_set_wait_limit(0)
    assert int(status.item()) == 4
    status.zero_()
    o, lse, imp = _call(ts, w, inp, status)
    assert int(status.item()) == 0
    q64, k64, v64 = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    O, LSE, IMP = orc.verify_attention(q64, k64, v64, inp["L"], inp["parents"], w.n_imp)
    pu.check_attention(o.cpu().numpy(), lse.cpu().numpy(), O, LSE)
    pu.check_importance(imp.cpu().numpy(), IMP, q64, k64, w.n_imp, w.G)
