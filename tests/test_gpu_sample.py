"""GPU parity: contextual-penalty sampling, tree acceptance and KV commit
(ts_penalized_sample_accept, ts_kv_commit) against the oracle."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _run(w, step=0, logits=None, prior=None, top_p=None, min_p=None, temperature=None,
         penalty=None, W=None, tree=None, uniforms=None, literal=False):
    import self_speculative_ultra_gb300 as ts
    inp = syn.sampling_inputs(w, step=step, tree=tree)
    logits = inp["logits"] if logits is None else logits
    prior = inp["prior"] if prior is None else prior
    u = inp["uniforms"] if uniforms is None else uniforms
    top_p = w.top_p if top_p is None else top_p
    min_p = w.min_p if min_p is None else min_p
    temperature = w.temperature if temperature is None else temperature
    penalty = w.penalty if penalty is None else penalty
    W = w.W if W is None else W
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sampled, path, n_path, bonus = ts.ts_penalized_sample_accept(
        pu.to_dev(logits), pu.to_dev(inp["tokens"]), pu.to_dev(inp["parents"]),
        pu.to_dev(np.asarray(prior, np.int32)), W, penalty, temperature, top_p, min_p,
        pu.to_dev(u), status=status, literal=literal)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sampled = sampled.cpu().numpy()
    n = int(n_path.item())
    path = path.cpu().numpy()[:n].tolist()
    bonus = int(bonus.item())
    ref, infos = orc.sample_all_nodes(logits, prior, inp["parents"], inp["tokens"], W, penalty,
                                      temperature, top_p, min_p, u, return_info=True,
                                      literal=literal)
    ties = pu.compare_draws(sampled, ref, infos)
    # acceptance is exact given the GPU's own draws (integer work)
    p_ref, b_ref = orc.accept_from_samples(inp["parents"], inp["tokens"], sampled)
    assert path == p_ref and bonus == b_ref
    if ties == 0:
        assert (path, bonus) == orc.sample_accept_sequential(
            logits, prior, inp["parents"], inp["tokens"], W, penalty, temperature, top_p, min_p, u,
            literal=literal)
    return sampled, path, bonus, ties


@pytest.mark.parametrize("name", ["tiny", "qwen2.5-1.5b", "llama3.1-8b", "mha-7b", "qwen2.5-14b"])
def test_configs(name):
    _, path, _, ties = _run(syn.WORKLOADS[name])
    print(name, "path", path, "ties", ties)


@pytest.mark.parametrize("step", [1, 2, 3])
def test_more_steps_llama(step):
    _run(syn.WORKLOADS["llama3.1-8b"], step=step)


@pytest.mark.parametrize("top_p,min_p,temp", [(1.0, 0.0, 1.0), (0.9, 0.0, 1.0), (0.5, 0.0, 0.7),
                                              (1.0, 0.05, 1.0), (0.9, 0.05, 2.0),
                                              (0.9, 1.5, 1.0), (1e-6, 0.0, 1.0)])
def test_truncation_settings(top_p, min_p, temp):
    w = syn.scaled(syn.WORKLOADS["tiny"], V=50000)
    _run(w, top_p=top_p, min_p=min_p, temperature=temp)


def test_flat_distribution_ranks_by_id():
    w = syn.scaled(syn.WORKLOADS["tiny"], V=4096)
    logits = np.zeros((w.T, w.V), dtype=np.float32)
    u = np.linspace(0.01, 0.99, w.T).astype(np.float32)
    _run(w, logits=logits, W=0, top_p=0.5, min_p=0.0, uniforms=u)


@pytest.mark.parametrize("layout,n_pool", [("spread", 8000), ("front", 6000), ("spread", 20000)])
def test_large_min_p_sets(layout, n_pool):
    """min-p sets above the 4,096 that are sorted in shared memory: a pool of
    n_pool tokens near the top (the rest 7 below), spread over the vocabulary
    (no slice overflows: the draw's radix descent over the row, leaving out
    the tokens below the pool; 20,000: some slice overflows and the pool is
    too large to list) or at its front (one slice overflows: the descent over
    the pool compacted by the node's row scan)."""
    w = syn.scaled(syn.WORKLOADS["tiny"], V=60000)
    rng = np.random.default_rng(11)
    logits = (rng.standard_normal((w.T, w.V)) * 0.3 - 5.0).astype(np.float32)
    for i in range(w.T):
        pos = (rng.permutation(w.V)[:n_pool] if layout == "spread" else np.arange(n_pool))
        logits[i, pos] = (rng.standard_normal(n_pool) * 0.3 + 2.0).astype(np.float32)
    _run(w, logits=logits, top_p=0.9, min_p=0.01)


def test_heavily_tied_logits():
    w = syn.scaled(syn.WORKLOADS["tiny"], V=30000)
    rng = np.random.default_rng(5)
    logits = rng.integers(-3, 4, size=(w.T, w.V)).astype(np.float32)
    _run(w, logits=logits, top_p=0.3, min_p=0.0)


def test_no_window_and_short_prior():
    w = syn.scaled(syn.WORKLOADS["tiny"], V=10000)
    _run(w, W=0)
    inp = syn.sampling_inputs(w)
    _run(w, prior=np.asarray([inp["tokens"][0]], np.int32), W=1024)


def test_single_node_and_tiny_vocab():
    _run(syn.scaled(syn.WORKLOADS["tiny"], T=1, V=1))
    _run(syn.scaled(syn.WORKLOADS["tiny"], T=1, V=7))


def test_max_vocab():
    _run(syn.scaled(syn.WORKLOADS["tiny"], T=4, V=262144))


def test_kv_commit_matches_oracle():
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(9)
    Hkv, L, T, d = 3, 500, 16, 128
    kb = rng.integers(0, 2 ** 16, size=(Hkv, L + T, d), dtype=np.uint16)
    vb = rng.integers(0, 2 ** 16, size=(Hkv, L + T, d), dtype=np.uint16)
    path = [0, 2, 7, 11]
    k, v = pu.to_dev_bf16(kb), pu.to_dev_bf16(vb)
    pdev = pu.to_dev(np.array(path + [0] * (T - 4), np.int32))
    ndev = pu.to_dev(np.array([4], np.int32))
    ts.ts_kv_commit(k, v, L, T, pdev, ndev)
    torch.cuda.synchronize()
    assert pu.bf16_dev_to_bits(k).tobytes() == orc.kv_commit(kb, L, path).tobytes()
    assert pu.bf16_dev_to_bits(v).tobytes() == orc.kv_commit(vb, L, path).tobytes()


@pytest.mark.parametrize("d,path", [(128, [0, 2, 7, 11]), (64, [0, 1, 2, 3]), (128, [0])])
def test_kv_commit_batched_matches_oracle(d, path):
    """Every layer in one launch: each layer's caches move exactly as the
    oracle's commit moves them (overlapping moves, a one-node path)."""
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(10 + d)
    n_layers, Hkv, L, T = 5, 4, 700, 16
    kbs = [rng.integers(0, 2 ** 16, size=(Hkv, L + T, d), dtype=np.uint16) for _ in range(n_layers)]
    vbs = [rng.integers(0, 2 ** 16, size=(Hkv, L + T, d), dtype=np.uint16) for _ in range(n_layers)]
    ks, vs = [pu.to_dev_bf16(x) for x in kbs], [pu.to_dev_bf16(x) for x in vbs]
    pdev = pu.to_dev(np.array(path + [0] * (T - len(path)), np.int32))
    ndev = pu.to_dev(np.array([len(path)], np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_kv_commit_batched(ks, vs, L, T, pdev, ndev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(n_layers):
        assert pu.bf16_dev_to_bits(ks[i]).tobytes() == orc.kv_commit(kbs[i], L, path).tobytes()
        assert pu.bf16_dev_to_bits(vs[i]).tobytes() == orc.kv_commit(vbs[i], L, path).tobytes()


@pytest.mark.parametrize("name", ["tiny", "llama3.1-8b", "qwen2.5-14b"])
def test_literal_ctrl_penalty(name):
    """The literal CTRL penalty (flag TS_PENALTY_CTRL_LITERAL) against the
    oracle's literal form, with a strong penalty so that negative windowed
    logits move visibly."""
    _run(syn.WORKLOADS[name], step=3, penalty=3.0, literal=True)


@pytest.mark.parametrize("d", [128, 64])
def test_kv_append_batched_matches_oracle(d):
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(20 + d)
    n_layers, Hkv, L, T = 4, 8, 3000, 64
    kbs = [rng.integers(0, 2 ** 16, size=(Hkv, L + T + 5, d), dtype=np.uint16) for _ in range(n_layers)]
    vbs = [rng.integers(0, 2 ** 16, size=(Hkv, L + T + 5, d), dtype=np.uint16) for _ in range(n_layers)]
    kr = rng.integers(0, 2 ** 16, size=(n_layers, Hkv, T, d), dtype=np.uint16)
    vr = rng.integers(0, 2 ** 16, size=(n_layers, Hkv, T, d), dtype=np.uint16)
    ks, vs = [pu.to_dev_bf16(x) for x in kbs], [pu.to_dev_bf16(x) for x in vbs]
    ts.ts_kv_append_batched(ks, vs, pu.to_dev_bf16(kr), pu.to_dev_bf16(vr), L)
    torch.cuda.synchronize()
    for i in range(n_layers):
        assert pu.bf16_dev_to_bits(ks[i]).tobytes() == orc.kv_append(kbs[i], L, kr[i]).tobytes()
        assert pu.bf16_dev_to_bits(vs[i]).tobytes() == orc.kv_append(vbs[i], L, vr[i]).tobytes()


def _bf16_bits_to_f16(bits):
    """bf16 bit patterns -> fp16 values, rounded to nearest even (numpy's
    float32 -> float16 conversion; the inputs below stay in fp16 range)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float16)


@pytest.mark.parametrize("d", [128, 64])
def test_kv_append_batched_into_fp16_v_cache(d):
    """fp16 V caches: the V rows arrive rounded to the nearest fp16 (normal
    values exactly, tiny ones to fp16 subnormals), the K rows bit for bit."""
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(40 + d)
    n_layers, Hkv, L, T = 3, 4, 2000, 64
    kbs = [rng.integers(0, 2 ** 16, size=(Hkv, L + T + 3, d), dtype=np.uint16) for _ in range(n_layers)]
    vfs = [rng.standard_normal((Hkv, L + T + 3, d)).astype(np.float16) for _ in range(n_layers)]
    kr = rng.integers(0, 2 ** 16, size=(n_layers, Hkv, T, d), dtype=np.uint16)
    vals = rng.standard_normal((n_layers, Hkv, T, d)).astype(np.float32)
    vals[..., :5] *= 1e-6          # fp16 subnormal range
    vals[..., 5:9] = np.clip(vals[..., 5:9] * 3e4, -6e4, 6e4)   # large but representable
    vr = syn.f32_to_bf16_bits(vals.reshape(-1)).reshape(vals.shape)
    ks = [pu.to_dev_bf16(x) for x in kbs]
    vs = [torch.from_numpy(x).cuda() for x in vfs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_kv_append_batched(ks, vs, pu.to_dev_bf16(kr), pu.to_dev_bf16(vr), L, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(n_layers):
        assert pu.bf16_dev_to_bits(ks[i]).tobytes() == orc.kv_append(kbs[i], L, kr[i]).tobytes()
        want = orc.kv_append(vfs[i], L, _bf16_bits_to_f16(vr[i]))
        assert vs[i].cpu().numpy().tobytes() == want.tobytes()


def test_kv_append_fp16_v_saturates_and_reports():
    """A V value beyond the fp16 range saturates to +-65504 and the call
    writes TS_ERR_UNSUPPORTED (2) to the status word."""
    import self_speculative_ultra_gb300 as ts
    Hkv, L, T, d = 2, 100, 8, 64
    ks = [torch.zeros((Hkv, L + T, d), dtype=torch.bfloat16, device="cuda")]
    vs = [torch.zeros((Hkv, L + T, d), dtype=torch.float16, device="cuda")]
    vals = np.zeros((1, Hkv, T, d), np.float32)
    vals[0, 1, 3, 7], vals[0, 0, 2, 1] = 1e5, -2e5
    vr = syn.f32_to_bf16_bits(vals.reshape(-1)).reshape(vals.shape)
    kr = np.zeros_like(vr)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_kv_append_batched(ks, vs, pu.to_dev_bf16(kr), pu.to_dev_bf16(vr), L, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2
    got = vs[0].cpu().numpy()
    assert got[1, L + 3, 7] == np.float16(65504) and got[0, L + 2, 1] == np.float16(-65504)
