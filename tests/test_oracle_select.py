"""Pins for the oracle's partial-KV selection and gather (CPU only)."""
import itertools

import numpy as np
import pytest

from oracle import ts_oracle as orc
import ts_synth as syn


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_best_subset(seed):
    """With distinct scores, the top-B set is the unique B-subset of the
    candidates with the largest score sum: enumerate them all."""
    rng = np.random.default_rng(seed)
    L, S, R, B = 14, 2, 3, 4
    imp = rng.permutation(np.arange(L, dtype=np.float64)) * 0.37 - 2.0
    cand = list(range(S, L - R))
    best = max(itertools.combinations(cand, B), key=lambda c: sum(imp[list(c)]))
    expect = sorted(list(range(S)) + list(best) + list(range(L - R, L)))
    np.testing.assert_array_equal(orc.select_partial(imp, L, B, S, R), expect)


@pytest.mark.parametrize("seed", range(4))
def test_defining_order_property(seed):
    """Every selected candidate beats every rejected one under
    (score desc, position asc); sizes, sinks and recent are exact."""
    rng = np.random.default_rng(100 + seed)
    L, S, R, B = 3000, 4, 64, 500
    imp = np.round(rng.standard_normal(L) * 4, 1)       # many exact ties
    idx = orc.select_partial(imp, L, B, S, R)
    assert len(idx) == S + B + R
    assert np.all(np.diff(idx) > 0)
    assert set(range(S)) <= set(idx) and set(range(L - R, L)) <= set(idx)
    chosen = np.array(sorted(set(idx) - set(range(S)) - set(range(L - R, L))))
    rejected = np.array(sorted(set(range(S, L - R)) - set(chosen)))
    worst = min(chosen, key=lambda j: (imp[j], -j))
    best_rej = max(rejected, key=lambda j: (imp[j], -j))
    assert (imp[worst], -worst) > (imp[best_rej], -best_rej)


def test_all_equal_scores_take_lowest_positions():
    L, S, R, B = 200, 4, 10, 30
    idx = orc.select_partial(np.zeros(L), L, B, S, R)
    np.testing.assert_array_equal(idx, list(range(S + B)) + list(range(L - R, L)))


@pytest.mark.parametrize("L", [1, 50, 97, 98])
def test_short_cache_keeps_everything(L):
    np.testing.assert_array_equal(orc.select_partial(np.arange(L), L, 30, 4, 64), np.arange(L))


def test_first_length_above_budget():
    L, S, R, B = 99, 4, 64, 30
    imp = -np.arange(L, dtype=np.float64)
    idx = orc.select_partial(imp, L, B, S, R)   # 31 candidates, drop the last one
    assert len(idx) == 98 and 34 not in idx


def test_planted_heavy_hitters_are_recalled():
    w = syn.scaled(syn.WORKLOADS["tiny"], L=2048, B=256)
    inp = syn.attention_inputs(w)
    q, k, v = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    _, _, imp = orc.verify_attention(q, k, v, w.L, inp["parents"], w.n_imp)
    idx = orc.select_partial(imp[0].astype(np.float32), w.L, w.B, w.S, w.R)
    assert set(inp["planted"][0].tolist()) <= set(idx.tolist())


def test_gather_is_a_bitwise_row_copy():
    rng = np.random.default_rng(3)
    cache = rng.integers(0, 2 ** 16, size=(50, 8), dtype=np.uint16)
    idx = np.array([0, 3, 4, 49])
    out = orc.gather_rows(cache, idx)
    for r, j in enumerate(idx):
        assert out[r].tobytes() == cache[j].tobytes()


# ---- incremental refresh of the partial cache
def test_incremental_refresh_hand_worked():
    # slot 2 (position 5) leaves; positions 7 and 8 join: 7 takes the freed
    # slot 2, 8 the new slot 5 (the cache grew from 5 to 6 rows)
    cache = np.arange(20 * 2, dtype=np.float64).reshape(20, 2)
    prev = [0, 1, 5, 9, 3]
    compact = np.zeros((6, 2))
    compact[:5] = cache[prev]
    slots, out, n = orc.refresh_incremental(prev, [0, 1, 3, 7, 8, 9], cache, compact)
    assert slots.tolist() == [0, 1, 7, 9, 3, 8] and n == 2
    np.testing.assert_array_equal(out, cache[[0, 1, 7, 9, 3, 8]])


def test_incremental_refresh_from_empty_is_the_full_gather():
    rng = np.random.default_rng(2)
    cache = rng.standard_normal((300, 4))
    imp = rng.standard_normal(300)
    kept = orc.select_partial(imp, 300, 20, 4, 8)
    slots, out, n = orc.refresh_incremental([], kept, cache, np.zeros((len(kept), 4)))
    assert slots.tolist() == kept.tolist() and n == len(kept)
    np.testing.assert_array_equal(out, orc.gather_rows(cache, kept))


def test_incremental_refresh_tracks_the_kept_set_over_steps():
    """Over a growing cache with drifting importance, the slots always hold
    exactly the kept set, every slot holds its position's row, and only the
    rows of newly kept positions are written."""
    rng = np.random.default_rng(4)
    S, B, R, d = 4, 40, 16, 3
    cache = rng.standard_normal((2000, d))
    base = rng.standard_normal(2000)
    slots, compact = np.zeros(0, dtype=np.int64), np.zeros((0, d))
    L = 30
    for step in range(40):
        imp = base + 0.3 * rng.standard_normal(2000)      # importance drifts step to step
        kept = orc.select_partial(imp[:L], L, B, S, R)
        grown = np.zeros((len(kept), d))
        grown[:len(compact)] = compact
        new_slots, compact, n = orc.refresh_incremental(slots, kept, cache, grown)
        assert sorted(new_slots.tolist()) == kept.tolist()
        np.testing.assert_array_equal(compact, cache[new_slots])
        assert n == len(set(kept.tolist()) - set(slots.tolist()))
        kept_slots = [s for s in range(len(slots)) if slots[s] in set(kept.tolist())]
        assert all(new_slots[s] == slots[s] for s in kept_slots)   # unchanged slots stay
        slots = new_slots
        L += int(rng.integers(1, 5))
