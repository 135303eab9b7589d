"""GPU parity of token reutilization (ts_ngram_insert, ts_ngram_build_tree)
against the oracle: the table is compared entry by entry after every batch
of insertions, the draft trees node by node (integer work: bit-exact)."""
import numpy as np
import pytest
import torch

import ts_synth as syn
from oracle import ts_oracle as orc

pytestmark = pytest.mark.gpu


def _table_as_dict(table, V, cap):
    t = table.cpu().numpy()
    meta = t[:2 * V].reshape(V, 2)
    cont = t[2 * V:].reshape(V, cap, 3)
    out = {}
    for a in np.nonzero(meta[:, 0])[0]:
        cnt, head = int(meta[a, 0]), int(meta[a, 1])
        out[int(a)] = [tuple(int(x) for x in cont[a, (head + i) % cap]) for i in range(cnt)]
    return out


@pytest.mark.parametrize("V,cap,vocab_used", [(128256, 64, 40), (32000, 8, 12), (50, 1, 5),
                                              (151936, 64, 3000)])
def test_insert_matches_oracle(V, cap, vocab_used):
    import self_speculative_ultra_gb300 as ts
    rng = np.random.default_rng(V + cap)
    toks = rng.integers(0, vocab_used, size=2400).astype(np.int32)
    dtoks = torch.from_numpy(toks).cuda()
    table = ts.ngram_table(V, cap)
    ref, prev = {}, 0
    # a long prefix, then decode-step sized increments (1..4 new tokens)
    ends = [2048] + list(range(2049, 2400, 3)) + [2400]
    for n in ends:
        ts.ts_ngram_insert(table, V, cap, dtoks, prev, n_tokens=n)
        ref = orc.ngram_insert(ref, toks[:n], prev, cap)
        prev = n
        if n in (2048, 2400) or n % 60 == 0:
            torch.cuda.synchronize()
            assert _table_as_dict(table, V, cap) == ref


def test_insert_reports_out_of_range_tokens():
    import self_speculative_ultra_gb300 as ts
    V, cap = 100, 4
    toks = torch.tensor([1, 2, 3, 4, 5, 100, 6, 7, 8, 9], dtype=torch.int32, device="cuda")
    table = ts.ngram_table(V, cap)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts.ts_ngram_insert(table, V, cap, toks, 0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    ref = orc.ngram_insert({}, [1, 2, 3, 4, 5], 0, cap)
    ref = orc.ngram_insert(ref, [6, 7, 8, 9], 0, cap)
    assert _table_as_dict(table, V, cap) == ref


@pytest.mark.parametrize("T_max", [64, 41, 40, 5, 1])
@pytest.mark.parametrize("k", [20, 5, 0])
def test_build_tree_matches_oracle(T_max, k):
    import self_speculative_ultra_gb300 as ts
    V, cap = 32000, 32
    rng = np.random.default_rng(T_max * 100 + k)
    toks = rng.integers(0, 30, size=3000).astype(np.int32)     # dense: roots with many n-grams
    table = ts.ngram_table(V, cap)
    ts.ts_ngram_insert(table, V, cap, torch.from_numpy(toks).cuda(), 0)
    ref = orc.ngram_insert({}, toks, 0, cap)
    for step, root in enumerate([int(toks[-1]), 7, 29, 31, 12345]):
        heads = rng.integers(0, V, size=(3, 3)).astype(np.int32)
        heads[0, 0] = 5 if step % 2 else heads[0, 0]          # heads sharing a first token
        keys = syn.ngram_rand_keys(11, step, cap)
        par, tok, n = ts.ts_ngram_build_tree(table, V, cap,
                                             torch.tensor([root], dtype=torch.int32, device="cuda"),
                                             torch.from_numpy(heads).cuda(), k,
                                             torch.from_numpy(keys).cuda(), T_max)
        torch.cuda.synchronize()
        chains = orc.ngram_retrieve(ref, root, k, keys)
        rp, rt = orc.build_draft_tree(root, heads.tolist(), chains, T_max)
        n = int(n.item())
        assert n == len(rp)
        np.testing.assert_array_equal(par.cpu().numpy()[:n], rp)
        np.testing.assert_array_equal(tok.cpu().numpy()[:n], rt)


def test_tree_from_an_empty_table_is_the_heads_tree():
    import self_speculative_ultra_gb300 as ts
    V, cap = 1000, 32
    table = ts.ngram_table(V, cap)
    heads = np.arange(9, dtype=np.int32).reshape(3, 3) + 100
    par, tok, n = ts.ts_ngram_build_tree(table, V, cap, torch.tensor([3], dtype=torch.int32, device="cuda"),
                                         torch.from_numpy(heads).cuda(), 20,
                                         torch.zeros(cap, dtype=torch.int32, device="cuda"), 64)
    rp, rt = orc.build_draft_tree(3, heads.tolist(), [], 64)
    n = int(n.item())
    assert n == 40
    np.testing.assert_array_equal(par.cpu().numpy()[:n], rp)
    np.testing.assert_array_equal(tok.cpu().numpy()[:n], rt)
