"""Pins for the oracle's verification attention and importance (CPU only).

Each check compares the oracle with something other than itself: a library
attention routine, closed forms, invariants, or a textbook special case.
"""
import numpy as np
import pytest
import scipy.special
import torch

from oracle import ts_oracle as orc
import ts_synth as syn


def _case(seed, T=7, Hq=6, Hkv=2, d=16, L=41):
    rng = np.random.default_rng(seed)
    parents, _ = syn.random_tree(rng, T, 100)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((Hkv, L + T, d))
    v = rng.standard_normal((Hkv, L + T, d))
    return q, k, v, L, parents


def _reach(parents):
    """Ancestor-or-self relation by transitive closure of the parent
    adjacency matrix (repeated boolean matrix products), built without the
    oracle's parent-chain walk."""
    T = len(parents)
    A = np.zeros((T, T), dtype=np.int64)
    for i in range(1, T):
        A[i, parents[i]] = 1
    R = np.eye(T, dtype=np.int64)
    P = np.eye(T, dtype=np.int64)
    for _ in range(T):
        P = (P @ A > 0).astype(np.int64)
        R = R | P
    return R.astype(bool)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_library_sdpa_with_independent_mask(seed):
    q, k, v, L, parents = _case(seed)
    T, Hq, d = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    O, LSE, _ = orc.verify_attention(q, k, v, L, parents)
    reach = _reach(parents)
    mask = np.ones((T, L + T), dtype=bool)
    mask[:, L:] = reach
    kt = torch.from_numpy(k[:, :L + T]).repeat_interleave(G, dim=0)   # [Hq, L+T, d]
    vt = torch.from_numpy(v[:, :L + T]).repeat_interleave(G, dim=0)
    qt = torch.from_numpy(q).permute(1, 0, 2)                           # [Hq, T, d]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask))
    np.testing.assert_allclose(O, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
    scores = (qt @ kt.transpose(1, 2)) / np.sqrt(d)
    scores = scores.masked_fill(~torch.from_numpy(mask), float("-inf"))
    lse_ref = torch.logsumexp(scores, dim=-1).permute(1, 0).numpy()
    np.testing.assert_allclose(LSE, lse_ref, rtol=1e-12, atol=1e-12)


def test_importance_closed_form_linearity():
    """imp[kv, j] = (sum of the group's last n_imp queries) . k_j / sqrt(d)."""
    q, k, v, L, parents = _case(5, T=9, Hq=8, Hkv=2, d=8, L=30)
    T, Hq, d = q.shape
    for n_imp in (1, 4, 9):
        _, _, imp = orc.verify_attention(q, k, v, L, parents, n_imp=n_imp)
        for kv in range(2):
            qs = q[T - n_imp:, kv * 4:(kv + 1) * 4, :].sum(axis=(0, 1))
            np.testing.assert_allclose(imp[kv], k[kv, :L] @ qs / np.sqrt(d), rtol=1e-12, atol=1e-12)


def test_non_ancestor_tree_rows_carry_zero_weight():
    q, k, v, L, parents = _case(3, T=12)
    O, _, _ = orc.verify_attention(q, k, v, L, parents)
    reach = _reach(parents)
    T = len(parents)
    for i in range(T):
        v2 = v.copy()
        outside = [a for a in range(T) if not reach[i, a]]
        v2[:, [L + a for a in outside]] += 1000.0
        O2, _, _ = orc.verify_attention(q, k, v2, L, parents)
        np.testing.assert_array_equal(O2[i], O[i])
        if i > 0:    # an ancestor row does change the output
            v3 = v.copy()
            v3[:, L + parents[i]] += 1000.0
            O3, _, _ = orc.verify_attention(q, k, v3, L, parents)
            assert np.abs(O3[i] - O[i]).max() > 1e-6


def test_constant_values_reproduce_weights_sum_to_one():
    q, k, v, L, parents = _case(4)
    v[:] = 3.25
    O, _, _ = orc.verify_attention(q, k, v, L, parents)
    np.testing.assert_allclose(O, 3.25, rtol=1e-13)


def test_planted_key_dominates():
    q, k, v, L, parents = _case(6, T=3, Hq=2, Hkv=1, d=16, L=50)
    j = 17
    k[0, j] = 80.0 * q[:, 0, :].mean(axis=0) / np.linalg.norm(q[:, 0, :].mean(axis=0))
    for i in range(3):
        q[i, 0] = k[0, j] / np.linalg.norm(k[0, j]) * 20.0
    O, _, _ = orc.verify_attention(q, k, v, L, parents)
    np.testing.assert_allclose(O[:, 0], np.broadcast_to(v[0, j], (3, 16)), atol=1e-9)


def test_gqa_contiguous_grouping_equals_replicated_mha():
    q, k, v, L, parents = _case(7, T=5, Hq=6, Hkv=3, d=8, L=20)
    O, LSE, _ = orc.verify_attention(q, k, v, L, parents)
    O_mha, LSE_mha, _ = orc.verify_attention(q, np.repeat(k, 2, axis=0),
                                             np.repeat(v, 2, axis=0), L, parents)
    np.testing.assert_allclose(O, O_mha, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(LSE, LSE_mha, rtol=1e-13)
    O_wrong, _, _ = orc.verify_attention(q, np.tile(k, (2, 1, 1)), np.tile(v, (2, 1, 1)), L, parents)
    assert np.abs(O_wrong - O).max() > 1e-3     # interleaved grouping differs


def test_single_node_is_textbook_decode_attention():
    rng = np.random.default_rng(11)
    d, L = 32, 100
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, L + 1, d))
    v = rng.standard_normal((1, L + 1, d))
    O, LSE, _ = orc.verify_attention(q, k, v, L, np.array([-1]))
    s = k[0] @ q[0, 0] / np.sqrt(d)          # the root sees the cache and itself
    w = scipy.special.softmax(s)
    np.testing.assert_allclose(O[0, 0], w @ v[0], rtol=1e-12)
    np.testing.assert_allclose(LSE[0, 0], scipy.special.logsumexp(s), rtol=1e-13)


def test_empty_cache_attends_to_tree_only():
    rng = np.random.default_rng(12)
    parents = np.array([-1, 0, 1, 0])
    q = rng.standard_normal((4, 2, 8))
    k = rng.standard_normal((1, 4, 8))
    v = rng.standard_normal((1, 4, 8))
    O, _, imp = orc.verify_attention(q, k, v, 0, parents)
    assert imp.shape == (1, 0)
    np.testing.assert_allclose(O[0, :], np.broadcast_to(v[0, 0], (2, 8)), rtol=1e-13)


def test_bf16_decode_is_exact():
    x = np.array([1.0, -2.5, 3.140625, 65280.0, 1e-3], dtype=np.float32)
    bits = syn.f32_to_bf16_bits(x)
    back = orc.bf16_to_f64(bits)
    assert back[0] == 1.0 and back[1] == -2.5 and back[2] == 3.140625 and back[3] == 65280.0
    assert abs(back[4] - 1e-3) / 1e-3 < 2 ** -8


# ---- softmax-weighted importance (the variant of the importance score)
@pytest.mark.parametrize("seed,n_imp", [(0, 0), (1, 3), (2, 1)])
def test_softmax_importance_equals_library_attention_weights(seed, n_imp):
    """The importance is the column sum, over the group's heads and the last
    n_imp nodes, of the masked attention weights that torch's softmax gives
    (mask from the independent transitive closure)."""
    q, k, v, L, parents = _case(seed)
    T, Hq, d = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    _, LSE, _ = orc.verify_attention(q, k, v, L, parents)
    imp = orc.importance_softmax(q, k, L, LSE, n_imp=n_imp)
    mask = np.ones((T, L + T), dtype=bool)
    mask[:, L:] = _reach(parents)
    kt = torch.from_numpy(k[:, :L + T]).repeat_interleave(G, dim=0)   # [Hq, L+T, d]
    qt = torch.from_numpy(q).permute(1, 0, 2)                           # [Hq, T, d]
    scores = (qt @ kt.transpose(1, 2)) / np.sqrt(d)
    w = torch.softmax(scores.masked_fill(~torch.from_numpy(mask), float("-inf")), dim=-1)
    rows = T if n_imp == 0 else n_imp
    ref = w[:, T - rows:, :L].sum(dim=1).reshape(Hkv, G, L).sum(dim=1).numpy()
    np.testing.assert_allclose(imp, ref, rtol=1e-12, atol=1e-15)


def test_softmax_importance_uniform_keys_closed_form():
    """All keys equal: every row spreads its weight evenly over the L cache
    rows and its root path, so imp[kv, j] = G * sum_i 1 / (L + depth_i + 1)
    over the importance nodes, whatever the queries."""
    rng = np.random.default_rng(5)
    T, Hq, Hkv, d, L = 9, 6, 3, 8, 30
    parents, _ = syn.random_tree(rng, T, 50)
    q = rng.standard_normal((T, Hq, d))
    k = np.broadcast_to(rng.standard_normal(d), (Hkv, L + T, d)).copy()
    v = rng.standard_normal((Hkv, L + T, d))
    _, LSE, _ = orc.verify_attention(q, k, v, L, parents)
    path_len = _reach(parents).sum(axis=1)            # ancestors-or-self of each node
    for n_imp in (1, 4, T):
        imp = orc.importance_softmax(q, k, L, LSE, n_imp=n_imp)
        want = (Hq // Hkv) * sum(1.0 / (L + path_len[i]) for i in range(T - n_imp, T))
        np.testing.assert_allclose(imp, np.full((Hkv, L), want), rtol=1e-12)


def test_softmax_importance_planted_key_takes_the_group_mass():
    """Queries of group 1's last n_imp nodes aligned with key j* of KV head 1
    put almost all their weight there: imp[1, j*] ~ n_imp * G; head 0 and
    the earlier nodes do not see it."""
    rng = np.random.default_rng(9)
    T, Hq, Hkv, d, L, n_imp, js = 6, 4, 2, 16, 50, 2, 17
    parents = np.array([-1, 0, 1, 1, 2, 4], dtype=np.int32)
    q = rng.standard_normal((T, Hq, d)) * 0.1
    k = rng.standard_normal((Hkv, L + T, d)) * 0.1
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    k[1, js] = 12.0 * u
    q[T - n_imp:, 2:4, :] += 12.0 * u                 # heads 2, 3 = group 1
    v = rng.standard_normal((Hkv, L + T, d))
    _, LSE, _ = orc.verify_attention(q, k, v, L, parents)
    imp = orc.importance_softmax(q, k, L, LSE, n_imp=n_imp)
    G = Hq // Hkv
    assert imp[1, js] == pytest.approx(n_imp * G, rel=1e-6)
    assert imp[0].sum() < n_imp * G and imp[0].max() < 0.2
