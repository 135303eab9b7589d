"""GPU parity of the decode loop as a whole: several consecutive steps of
verify -> partial-cache refresh (batched over layers) -> penalised sampling
and acceptance -> KV commit, with the cache length advanced by the accepted
length and the penalty window fed by the committed tokens, checked against
the oracle's composition of the same steps after every step.

Each step's fresh inputs (tree K/V rows, queries, logits, uniforms) are
seeded; the next tree's root token is the bonus token the step produced, so
the GPU's own accepted path decides the state the next step starts from and
the oracle follows that state (the decisions themselves are checked every
step: importance within its bound, selection exact given the importance
values, draws exact up to counted ties, acceptance and commit exact).
"""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _bf16_normal(rng, shape):
    return syn.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


@pytest.mark.parametrize("base,L0,n_steps,n_layers", [
    ("tiny", 1500, 6, 2),
    ("llama3.1-8b", 5000, 3, 2),
])
def test_decode_loop_matches_oracle(base, L0, n_steps, n_layers):
    import self_speculative_ultra_gb300 as ts
    w = syn.scaled(syn.WORKLOADS[base], L=L0, B=min(syn.WORKLOADS[base].B, 1024), V=8192, W=256)
    T, Hq, Hkv, d, V, W = w.T, w.Hq, w.Hkv, w.d, w.V, w.W
    G = Hq // Hkv
    rng = np.random.default_rng([w.seed, 4242])
    L_cap = L0 + n_steps * T + T
    # host copies of every layer's cache (bf16 bits), committed rows [0, L)
    kc = [_bf16_normal(rng, (Hkv, L_cap, d)) for _ in range(n_layers)]
    vc = [_bf16_normal(rng, (Hkv, L_cap, d)) for _ in range(n_layers)]
    kd_ = [pu.to_dev_bf16(x) for x in kc]
    vd_ = [pu.to_dev_bf16(x) for x in vc]
    history = rng.integers(0, V, size=W + 7).astype(np.int32).tolist()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L, total_ties, committed = L0, 0, 0
    for step in range(n_steps):
        parents, tokens = syn.make_tree(w, rng)
        parents = np.asarray(parents, np.int32)
        tokens = np.asarray(tokens, np.int32)
        tokens[0] = history[-1]
        # fresh tree rows, queries, logits (first child planted with p = 0.7), uniforms
        for layer in range(n_layers):
            kc[layer][:, L:L + T] = _bf16_normal(rng, (Hkv, T, d))
            vc[layer][:, L:L + T] = _bf16_normal(rng, (Hkv, T, d))
            kd_[layer][:, L:L + T].copy_(pu.to_dev_bf16(kc[layer][:, L:L + T]))
            vd_[layer][:, L:L + T].copy_(pu.to_dev_bf16(vc[layer][:, L:L + T]))
        qb = [_bf16_normal(rng, (T, Hq, d)) for _ in range(n_layers)]
        logits = (rng.standard_normal((T, V), dtype=np.float32) * np.float32(3.0))
        first_child = np.full(T, -1)
        for i in range(T - 1, 0, -1):
            first_child[parents[i]] = i
        for i in range(T):
            if first_child[i] >= 0 and rng.random() < 0.7:
                logits[i, tokens[first_child[i]]] += np.float32(30.0)
        u = rng.random(T, dtype=np.float32)
        prior = np.asarray(history[-W:], np.int32)
        dev_par, dev_tok = pu.to_dev(parents), pu.to_dev(tokens)

        # ---- library: every layer's verify, one batched refresh, sample, commit
        outs = []
        imps = [torch.empty((Hkv, L), dtype=torch.float32, device="cuda") for _ in range(n_layers)]
        for layer in range(n_layers):
            o, lse, _ = ts.ts_verify_attention(pu.to_dev_bf16(qb[layer]), kd_[layer], vd_[layer], L,
                                               dev_par, n_imp=w.n_imp, imp=imps[layer],
                                               status=status)
            outs.append((o, lse))
        N = min(L, w.S + w.B + w.R)
        idxs = [torch.empty((Hkv, N), dtype=torch.int32, device="cuda") for _ in range(n_layers)]
        kds = [torch.empty((Hkv, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(n_layers)]
        vds = [torch.empty((Hkv, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(n_layers)]
        ts.ts_partial_kv_select_gather_batched(imps, kd_, vd_, L, w.B, w.S, w.R, idxs, kds, vds,
                                               status=status)
        sampled, path, n_path, bonus = ts.ts_penalized_sample_accept(
            pu.to_dev(logits), dev_tok, dev_par, pu.to_dev(prior), W, w.penalty, w.temperature,
            w.top_p, w.min_p, pu.to_dev(u), status=status)
        for layer in range(n_layers):
            ts.ts_kv_commit(kd_[layer], vd_[layer], L, T, path, n_path, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"step {step}: device status {int(status.item())}"

        # ---- oracle, step by step on the same state
        for layer in range(n_layers):
            q64 = orc.bf16_to_f64(qb[layer])
            k64 = orc.bf16_to_f64(kc[layer][:, :L + T])
            v64 = orc.bf16_to_f64(vc[layer][:, :L + T])
            O, LSE, IMP = orc.verify_attention(q64, k64, v64, L, parents, n_imp=w.n_imp)
            o, lse = outs[layer]
            pu.check_attention(o.cpu().numpy(), lse.cpu().numpy(), O, LSE)
            imp_g = imps[layer].cpu().numpy()
            pu.check_importance(imp_g, IMP, q64, k64, w.n_imp, G)
            # the selection is exact given the importance values it ranked
            idx_g = idxs[layer].cpu().numpy()
            kbits = pu.bf16_dev_to_bits(kds[layer])
            vbits = pu.bf16_dev_to_bits(vds[layer])
            for h in range(Hkv):
                ref = orc.select_partial(imp_g[h].astype(np.float64), L, w.B, w.S, w.R)
                np.testing.assert_array_equal(idx_g[h], ref)
                assert kbits[h].tobytes() == kc[layer][h][ref].tobytes()
                assert vbits[h].tobytes() == vc[layer][h][ref].tobytes()
        ref_s, infos = orc.sample_all_nodes(logits, prior, parents, tokens, W, w.penalty,
                                            w.temperature, w.top_p, w.min_p, u, return_info=True)
        s_g = sampled.cpu().numpy()
        total_ties += pu.compare_draws(s_g, ref_s, infos, kind="loop draw")
        n = int(n_path.item())
        p_g = path.cpu().numpy()[:n].tolist()
        p_ref, b_ref = orc.accept_from_samples(parents, tokens, s_g)
        assert p_g == p_ref and int(bonus.item()) == b_ref
        for layer in range(n_layers):
            kc[layer] = orc.kv_commit(kc[layer], L, p_g)
            vc[layer] = orc.kv_commit(vc[layer], L, p_g)
            assert pu.bf16_dev_to_bits(kd_[layer]).tobytes() == kc[layer].tobytes()
            assert pu.bf16_dev_to_bits(vd_[layer]).tobytes() == vc[layer].tobytes()
        # advance: the accepted rows are committed, the bonus token is the next root
        history += [int(tokens[j]) for j in p_g[1:]] + [b_ref]
        L += n
        committed += n
    print(f"{base}: {n_steps} steps, {committed} rows committed, {total_ties} tied draws")
    assert committed >= n_steps
