"""Pins of the token-reutilization oracle (4-gram table, retrieval, draft-tree
builder): hand-worked examples whose expected values were derived by hand
from the reading stated in the oracle, plus invariants."""
import numpy as np
import pytest

from oracle import ts_oracle as orc


def test_insert_hand_worked():
    # 4-grams of the sequence, by the position of their last token:
    # (5,1,2,3) (1,2,3,5) (2,3,5,1) (3,5,1,2) (5,1,2,4) (1,2,4,5) (2,4,5,1)
    # (4,5,1,9) (5,1,9,9)
    t = orc.ngram_insert({}, [5, 1, 2, 3, 5, 1, 2, 4, 5, 1, 9, 9], 0, cap=8)
    assert t == {5: [(1, 2, 3), (1, 2, 4), (1, 9, 9)],
                 1: [(2, 3, 5), (2, 4, 5)],
                 2: [(3, 5, 1), (4, 5, 1)],
                 3: [(5, 1, 2)],
                 4: [(5, 1, 9)]}


def test_insert_keeps_one_copy_of_a_repeated_4gram():
    # (7,8,9,10) appears twice; (8,9,10,7) (9,10,7,8) (10,7,8,9) once
    t = orc.ngram_insert({}, [7, 8, 9, 10, 7, 8, 9, 10], 0, cap=8)
    assert t == {7: [(8, 9, 10)], 8: [(9, 10, 7)], 9: [(10, 7, 8)], 10: [(7, 8, 9)]}


def test_insert_drops_the_oldest_past_the_capacity():
    toks = [1, 10, 11, 12, 1, 20, 21, 22, 1, 30, 31, 32]
    t = orc.ngram_insert({}, toks, 0, cap=2)
    assert t[1] == [(20, 21, 22), (30, 31, 32)]
    assert t[12] == [(1, 20, 21)] and t[22] == [(1, 30, 31)]


def test_incremental_insert_equals_one_shot():
    rng = np.random.default_rng(3)
    toks = rng.integers(0, 6, size=300).tolist()    # small vocabulary: many repeats
    one = orc.ngram_insert({}, toks, 0, cap=5)
    inc, prev = {}, 0
    for n in (4, 5, 17, 100, 299, 300):
        inc = orc.ngram_insert(inc, toks[:n], prev, cap=5)
        prev = n
    assert inc == one


def test_retrieve_all_when_at_most_k_else_smallest_keys():
    t = {5: [(1, 2, 3), (1, 2, 4), (1, 9, 9)]}
    assert orc.ngram_retrieve(t, 5, 3, [9, 9, 9]) == [(1, 2, 3), (1, 2, 4), (1, 9, 9)]
    assert orc.ngram_retrieve(t, 6, 3, [0, 0, 0]) == []
    # keys 7, 3, 3: slots 1 and 2 tie on 3, the lower slot first
    assert orc.ngram_retrieve(t, 5, 2, [7, 3, 3]) == [(1, 2, 4), (1, 9, 9)]
    assert orc.ngram_retrieve(t, 5, 1, [2, 3, 1]) == [(1, 9, 9)]


def test_tree_hand_worked():
    heads = [[10, 11, 12], [20, 21, 22], [30, 31, 32]]
    chains = [(10, 20, 30), (10, 99, 98), (1, 2, 3)]
    par, tok = orc.build_draft_tree(5, heads, chains, 64)
    # root, 3 depth-1, 9 depth-2, 27 depth-3 nodes = 40 in breadth-first order
    assert len(par) == 40 + 2 + 3
    assert list(tok[:4]) == [5, 10, 11, 12] and list(par[:4]) == [-1, 0, 0, 0]
    assert list(par[4:7]) == [1, 1, 1] and list(tok[4:7]) == [20, 21, 22]
    assert list(par[13:16]) == [4, 4, 4] and list(tok[13:16]) == [30, 31, 32]
    # (10,20,30) already exists: 0 -> 1 -> 4 -> 13; (10,99,98) adds 99 under
    # node 1 and 98 under it; (1,2,3) adds a new branch under the root
    assert list(par[40:]) == [1, 40, 0, 42, 43]
    assert list(tok[40:]) == [99, 98, 1, 2, 3]


def test_tree_truncates_at_T_max_in_insertion_order():
    heads = [[10, 11, 12], [20, 21, 22], [30, 31, 32]]
    par, tok = orc.build_draft_tree(5, heads, [(1, 2, 3)], 5)
    assert list(par) == [-1, 0, 0, 0, 1] and list(tok) == [5, 10, 11, 12, 20]
    # room for the head tree and two chain nodes: the chain stops after them
    par, tok = orc.build_draft_tree(5, heads, [(1, 2, 3), (4, 5, 6)], 42)
    assert list(par[40:]) == [0, 40] and list(tok[40:]) == [1, 2]


def test_tree_invariants_random():
    rng = np.random.default_rng(7)
    for _ in range(50):
        heads = rng.integers(0, 50, size=(3, 3)).tolist()
        chains = [tuple(c) for c in rng.integers(0, 50, size=(int(rng.integers(0, 21)), 3)).tolist()]
        T_max = int(rng.integers(1, 65))
        par, tok = orc.build_draft_tree(int(rng.integers(50)), heads, chains, T_max)
        assert 1 <= len(par) <= T_max and par[0] == -1
        assert all(0 <= par[i] < i for i in range(1, len(par)))
        depth = [0] * len(par)
        for i in range(1, len(par)):
            depth[i] = depth[par[i]] + 1
        assert max(depth) <= 3
        # every retrieved chain that fully fits is a root path of the tree
        kids = {}
        for i in range(1, len(par)):
            kids.setdefault((int(par[i]), int(tok[i])), i)
        for c in chains:
            cur, ok = 0, True
            for t in c:
                if (cur, t) not in kids:
                    ok = False
                    break
                cur = kids[(cur, t)]
            assert ok or len(par) == T_max
