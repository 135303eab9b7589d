"""GPU parity: partial-KV top-B selection + gather (ts_partial_kv_select_gather)
against the oracle, standalone (same fp32 scores on both sides: bit-exact)
and chained after verification (oracle scores: exact up to counted ties)."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _standalone(Hkv, L, B, S, R, d=128, seed=0, grid=None):
    import self_speculative_ultra_gb300 as ts
    imp = syn.importance_scores(Hkv, L, seed, grid=grid)
    rng = np.random.default_rng(seed)
    kbits = rng.integers(0, 2 ** 16, size=(Hkv, L + 8, d), dtype=np.uint16)
    vbits = rng.integers(0, 2 ** 16, size=(Hkv, L + 8, d), dtype=np.uint16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, kd, vd = ts.ts_partial_kv_select_gather(pu.to_dev(imp), pu.to_dev_bf16(kbits),
                                                 pu.to_dev_bf16(vbits), L, B, S, R, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    idx = idx.cpu().numpy()
    kd, vd = pu.bf16_dev_to_bits(kd), pu.bf16_dev_to_bits(vd)
    for h in range(Hkv):
        ref = orc.select_partial(imp[h].astype(np.float64), L, B, S, R)
        np.testing.assert_array_equal(idx[h], ref)
        assert kd[h].tobytes() == orc.gather_rows(kbits[h], ref).tobytes()
        assert vd[h].tobytes() == orc.gather_rows(vbits[h], ref).tobytes()


@pytest.mark.parametrize("Hkv,L,B", [(1, 4096, 1024), (2, 32768, 4096), (8, 102400, 4096),
                                     (3, 5000, 700), (1, 70000, 4096)])
def test_standalone_bit_exact(Hkv, L, B):
    _standalone(Hkv, L, B, 4, 64)


@pytest.mark.parametrize("grid", [1.0, 8.0, 64.0])
def test_standalone_exact_ties_break_to_lower_position(grid):
    _standalone(4, 20000, 3000, 4, 64, grid=grid)


def test_standalone_signed_zero_ties():
    """-0.0 and +0.0 are equal scores: ties between them go to the lower position."""
    import self_speculative_ultra_gb300 as ts
    L, B = 3000, 500
    imp = np.where(np.arange(L) % 2 == 0, np.float32(0.0), np.float32(-0.0)).astype(np.float32)[None]
    kb = np.zeros((1, L + 1, 64), np.uint16)
    idx, _, _ = ts.ts_partial_kv_select_gather(pu.to_dev(imp), pu.to_dev_bf16(kb), pu.to_dev_bf16(kb),
                                               L, B, 4, 64)
    np.testing.assert_array_equal(idx.cpu().numpy()[0], orc.select_partial(imp[0], L, B, 4, 64))


@pytest.mark.parametrize("L,B,S,R", [(1, 10, 4, 64), (60, 10, 4, 64), (78, 10, 4, 64),
                                     (79, 10, 4, 64), (2000, 0, 4, 64), (2000, 100, 0, 0),
                                     (3000, 2931, 4, 64)])
def test_standalone_edges(L, B, S, R):
    _standalone(2, L, B, S, R, d=64)


@pytest.mark.parametrize("name", ["tiny", "qwen2.5-1.5b", "llama3.1-8b"])
def test_chained_after_verification(name):
    """GPU verify -> GPU select, against oracle verify -> oracle select.
    Planted heavy hitters must all be kept; differing positions must be
    ties at the cut."""
    import self_speculative_ultra_gb300 as ts
    w = syn.WORKLOADS[name]
    L = min(w.L, 32768)
    inp = syn.attention_inputs(w, L=L)
    q, k, v = (pu.to_dev_bf16(inp[n]) for n in ("q", "k", "v"))
    parents = pu.to_dev(inp["parents"])
    _, _, imp = ts.ts_verify_attention(q, k, v, L, parents, n_imp=w.n_imp)
    idx, kd, vd = ts.ts_partial_kv_select_gather(imp, k, v, L, w.B, w.S, w.R)
    torch.cuda.synchronize()
    q64, k64, v64 = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    _, _, IMP = orc.verify_attention(q64, k64, v64, L, inp["parents"], w.n_imp)
    imp_rank = IMP.astype(np.float32).astype(np.float64)
    idx_ref = np.stack([orc.select_partial(imp_rank[h], L, w.B, w.S, w.R) for h in range(w.Hkv)])
    idx_g = idx.cpu().numpy()
    ties = pu.compare_selection(idx_g, idx_ref, imp_rank, L, w.B, w.S, w.R)
    print(f"{name}: {ties} tied positions differ")
    for h in range(w.Hkv):
        assert set(inp["planted"][h].tolist()) <= set(idx_g[h].tolist())
    kd_bits = pu.bf16_dev_to_bits(kd)
    for h in range(w.Hkv):
        assert kd_bits[h].tobytes() == inp["k"][h][idx_g[h]].tobytes()


@pytest.mark.parametrize("n_layers,Hkv,L,B", [(3, 2, 9000, 1000), (4, 8, 102400, 4096), (2, 1, 50, 10)])
def test_batched_equals_per_layer_and_oracle(n_layers, Hkv, L, B):
    """The batched call returns exactly what the single-layer call returns for
    each layer, and both match the oracle bit for bit."""
    import self_speculative_ultra_gb300 as ts
    S, R, d = 4, 64, 128
    N = min(L, S + B + R)
    imps, ks, vs, bits = [], [], [], []
    for layer in range(n_layers):
        imp = syn.importance_scores(Hkv, L, 10 + layer, grid=1.0 if layer == 1 else None)
        rng = np.random.default_rng(layer)
        kb = rng.integers(0, 2 ** 16, size=(Hkv, L + 8, d), dtype=np.uint16)
        vb = rng.integers(0, 2 ** 16, size=(Hkv, L + 8, d), dtype=np.uint16)
        bits.append((imp, kb, vb))
        imps.append(pu.to_dev(imp))
        ks.append(pu.to_dev_bf16(kb))
        vs.append(pu.to_dev_bf16(vb))
    mk = lambda shape, dt: [torch.empty(shape, dtype=dt, device="cuda") for _ in range(n_layers)]  # noqa: E731
    idxs, kds, vds = mk((Hkv, N), torch.int32), mk((Hkv, N, d), torch.bfloat16), mk((Hkv, N, d), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_partial_kv_select_gather_batched(imps, ks, vs, L, B, S, R, idxs, kds, vds, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for layer in range(n_layers):
        i1, k1, v1 = ts.ts_partial_kv_select_gather(imps[layer], ks[layer], vs[layer], L, B, S, R)
        torch.cuda.synchronize()
        assert torch.equal(i1, idxs[layer])
        assert torch.equal(k1.view(torch.int16), kds[layer].view(torch.int16))
        assert torch.equal(v1.view(torch.int16), vds[layer].view(torch.int16))
        imp, kb, vb = bits[layer]
        got = idxs[layer].cpu().numpy()
        for h in range(Hkv):
            np.testing.assert_array_equal(got[h], orc.select_partial(imp[h].astype(np.float64), L, B, S, R))
