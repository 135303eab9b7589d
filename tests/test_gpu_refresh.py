"""GPU parity: incremental partial-cache refresh
(ts_partial_kv_refresh_incremental[_batched]) against the oracle, bit for bit:
the slot -> position map, the compact K/V rows and the number of rows
written, over sequences of steps in which the cache grows past the budget and
the importance drifts (with exact ties in some cases)."""
import numpy as np
import pytest
import torch

from oracle import ts_oracle as orc
import parity_util as pu

pytestmark = pytest.mark.gpu


def _imp(rng, base, L, drift, grid):
    x = base[:, :L] + drift * rng.standard_normal((base.shape[0], L))
    if grid:
        x = np.round(x / grid) * grid
    return x.astype(np.float32)


def _sequence(Hkv, d, B, S, R, L0, steps, grid=None, n_layers=1, drift=0.3, seed=0,
              v_fp16=False):
    """v_fp16: the V caches hold fp16 (the same random 16-bit patterns; the
    refresh copies bytes, so the expected rows are the same bits)."""
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(seed)
    N_cap = S + B + R
    L_end = L0 + 4 * steps + 8
    caches = []
    for _ in range(n_layers):
        kb = rng.integers(0, 2 ** 16, size=(Hkv, L_end, d), dtype=np.uint16)
        vb = rng.integers(0, 2 ** 16, size=(Hkv, L_end, d), dtype=np.uint16)
        base = rng.standard_normal((Hkv, L_end)) * 4.0
        caches.append((kb, vb, base))
    ks = [pu.to_dev_bf16(c[0]) for c in caches]
    vs = [pu.to_dev_bf16(c[1]) for c in caches]
    if v_fp16:
        vs = [v.view(torch.float16) for v in vs]
    idxs = [torch.full((Hkv, N_cap), -7, dtype=torch.int32, device="cuda") for _ in range(n_layers)]
    kds = [torch.zeros((Hkv, N_cap, d), dtype=torch.bfloat16, device="cuda") for _ in range(n_layers)]
    vds = [torch.zeros((Hkv, N_cap, d), dtype=vs[0].dtype, device="cuda") for _ in range(n_layers)]
    # oracle state per (layer, head)
    slots = [[np.zeros(0, dtype=np.int64) for _ in range(Hkv)] for _ in range(n_layers)]
    kc = [[np.zeros((0, d), dtype=np.uint16) for _ in range(Hkv)] for _ in range(n_layers)]
    vc = [[np.zeros((0, d), dtype=np.uint16) for _ in range(Hkv)] for _ in range(n_layers)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    written = torch.zeros(n_layers * Hkv, dtype=torch.int32, device="cuda")
    L, N_prev, total_written, total_full = L0, 0, 0, 0
    for step in range(steps):
        imps_np = [_imp(rng, c[2], L, drift, grid) for c in caches]
        imps = [pu.to_dev(x) for x in imps_np]
        # the K/V caches are immutable below L; only the slots move
        if n_layers == 1:
            N_new = ts.ts_partial_kv_refresh_incremental(
                imps[0], ks[0], vs[0], L, B, S, R, idxs[0], kds[0], vds[0],
                N_prev, n_written=written, status=status)
        else:
            N_new = ts.ts_partial_kv_refresh_incremental_batched(
                imps, ks, vs, L, B, S, R, idxs, kds, vds, N_prev, n_written=written,
                status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"step {step}: status {int(status.item())}"
        assert N_new == min(L, S + B + R)
        wr = written.cpu().numpy()
        for layer in range(n_layers):
            kb, vb, _ = caches[layer]
            idx_g = idxs[layer].cpu().numpy()
            kd_g = pu.bf16_dev_to_bits(kds[layer])
            vd_g = pu.bf16_dev_to_bits(vds[layer].view(torch.bfloat16))
            for h in range(Hkv):
                kept = orc.select_partial(imps_np[layer][h].astype(np.float64), L, B, S, R)
                grown_k = np.zeros((N_new, d), dtype=np.uint16)
                grown_v = np.zeros((N_new, d), dtype=np.uint16)
                grown_k[:len(kc[layer][h])] = kc[layer][h]
                grown_v[:len(vc[layer][h])] = vc[layer][h]
                s_new, k_new, n = orc.refresh_incremental(slots[layer][h], kept, kb[h], grown_k)
                _, v_new, _ = orc.refresh_incremental(slots[layer][h], kept, vb[h], grown_v)
                np.testing.assert_array_equal(idx_g[h, :N_new], s_new,
                                              err_msg=f"step {step} layer {layer} head {h}")
                assert kd_g[h, :N_new].tobytes() == k_new.tobytes()
                assert vd_g[h, :N_new].tobytes() == v_new.tobytes()
                assert wr[layer * Hkv + h] == n
                slots[layer][h], kc[layer][h], vc[layer][h] = s_new, k_new, v_new
                total_written += n
                total_full += N_new
        N_prev = N_new
        L += int(rng.integers(1, 5))
    return total_written / max(total_full, 1)


@pytest.mark.parametrize("Hkv,d,B,L0", [(1, 64, 64, 20), (2, 128, 300, 340), (8, 128, 1024, 5000)])
def test_sequence_matches_oracle(Hkv, d, B, L0):
    """From an empty compact cache through the growth phase (L < S+B+R) and
    past the budget; only changed rows are written."""
    frac = _sequence(Hkv, d, B, 4, 64, L0, steps=12)
    print(f"Hkv={Hkv} d={d} B={B}: {frac:.3f} of the full gather's rows written")


def test_sequence_fp16_v_cache():
    """An fp16 V cache: the same slots and the same row bytes."""
    _sequence(2, 128, 300, 4, 64, 340, steps=6, n_layers=2, v_fp16=True)


def test_sequence_with_exact_ties():
    _sequence(2, 128, 256, 4, 64, 3000, steps=8, grid=2.0, seed=3)


def test_batched_layers_match_oracle():
    _sequence(4, 128, 512, 4, 64, 4000, steps=6, n_layers=3, seed=5)


def test_first_call_equals_the_full_gather():
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(9)
    Hkv, d, L, B, S, R = 4, 128, 9000, 1000, 4, 64
    kb = rng.integers(0, 2 ** 16, size=(Hkv, L + 16, d), dtype=np.uint16)
    vb = rng.integers(0, 2 ** 16, size=(Hkv, L + 16, d), dtype=np.uint16)
    imp = pu.to_dev((rng.standard_normal((Hkv, L)) * 3).astype(np.float32))
    k, v = pu.to_dev_bf16(kb), pu.to_dev_bf16(vb)
    i1, k1, v1 = ts.ts_partial_kv_select_gather(imp, k, v, L, B, S, R)
    N = S + B + R
    idx = torch.empty((Hkv, N), dtype=torch.int32, device="cuda")
    kd = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    assert ts.ts_partial_kv_refresh_incremental(imp, k, v, L, B, S, R, idx, kd, vd, 0) == N
    torch.cuda.synchronize()
    assert torch.equal(idx, i1)
    assert torch.equal(kd.view(torch.int16), k1.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), v1.view(torch.int16))


def test_full_size_two_steps():
    """The 100K-token cache of the 8B shape: a full first refresh, then one
    step later (3 more tokens, drifted importance) an incremental one."""
    _sequence(8, 128, 4096, 4, 64, 102400, steps=2, seed=11)


def test_invalid_previous_slot_is_reported():
    import self_speculative_ultra_gb300 as ts
    Hkv, d, L, B, S, R = 1, 64, 500, 50, 4, 16
    N = S + B + R
    k = torch.zeros((Hkv, L, d), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((Hkv, L, d), dtype=torch.bfloat16, device="cuda")
    imp = torch.randn((Hkv, L), device="cuda")
    idx = torch.arange(N, dtype=torch.int32, device="cuda").reshape(1, N).contiguous()
    idx[0, 5] = L + 100                      # a position outside the cache
    kd = torch.zeros((Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros((Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_partial_kv_refresh_incremental(imp, k, v, L, B, S, R, idx, kd, vd, N, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
