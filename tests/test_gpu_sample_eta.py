"""GPU parity of the eta-sampling variant (ts_penalized_sample_accept_eta)
against the oracle: draws bit-exact except near-cut ties (counted), then
acceptance exact given the draws."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _run(w, eps, alpha, step=0, logits=None, temperature=None, W=None, uniforms=None):
    import self_speculative_ultra_gb300 as ts
    inp = syn.sampling_inputs(w, step=step)
    logits = inp["logits"] if logits is None else logits
    u = inp["uniforms"] if uniforms is None else uniforms
    temperature = w.temperature if temperature is None else temperature
    W = w.W if W is None else W
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sampled, path, n_path, bonus = ts.ts_penalized_sample_accept_eta(
        pu.to_dev(logits), pu.to_dev(inp["tokens"]), pu.to_dev(inp["parents"]),
        pu.to_dev(np.asarray(inp["prior"], np.int32)), W, w.penalty, temperature, eps, alpha,
        pu.to_dev(u), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sampled = sampled.cpu().numpy()
    ref, infos = orc.sample_all_nodes_eta(logits, inp["prior"], inp["parents"], inp["tokens"], W,
                                          w.penalty, temperature, eps, alpha, u, return_info=True)
    ties = pu.compare_draws(sampled, ref, infos, kind="eta draw")
    n = int(n_path.item())
    p_ref, b_ref = orc.accept_from_samples(inp["parents"], inp["tokens"], sampled)
    assert path.cpu().numpy()[:n].tolist() == p_ref and int(bonus.item()) == b_ref
    return ties


@pytest.mark.parametrize("name", ["tiny", "llama3.1-8b", "qwen2.5-14b"])
@pytest.mark.parametrize("eps", [0.0009, 0.02])
def test_configs(name, eps):
    _run(syn.WORKLOADS[name], eps, float(np.sqrt(eps)))


@pytest.mark.parametrize("eps,alpha,temp", [(0.0, 0.0, 1.0), (0.3, 1.0, 1.0), (0.0009, 0.03, 3.0),
                                            (0.05, 0.2, 0.5)])
def test_settings(eps, alpha, temp):
    """eps = 0 keeps every token (plain categorical over the whole vocabulary:
    the radix path); a large eps with alpha 1 keeps only the top tokens."""
    w = syn.scaled(syn.WORKLOADS["tiny"], V=50000)
    _run(w, eps, alpha, temperature=temp)


def test_flat_distribution():
    w = syn.scaled(syn.WORKLOADS["tiny"], V=4096)
    logits = np.zeros((w.T, w.V), dtype=np.float32)
    u = np.linspace(0.01, 0.99, w.T).astype(np.float32)
    _run(w, 0.0009, 0.03, logits=logits, W=0, uniforms=u)
