"""Pins for the oracle's contextual penalty, truncation, draw and acceptance
(CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import ts_oracle as orc
import ts_synth as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden", "sampling_hand_worked.json")


def _gold():
    with open(GOLD) as f:
        g = json.load(f)
    ln = math.log
    logits = np.array([1.2 * ln(8), ln(4), -ln(2) / 1.2, ln(2), 0.0, -ln(4) / 1.2], dtype=np.float32)
    return g, logits


def test_hand_worked_probabilities_at_root():
    g, x = _gold()
    win = orc.penalty_window(g["prior"], [], g["W"])
    xp = orc.penalised_logits(x, win, g["penalty"], g["temperature"])
    p = scipy.special.softmax(xp.astype(np.float64))
    np.testing.assert_allclose(p, g["expected_probabilities_root"], rtol=2e-6)


@pytest.mark.parametrize("case", range(8))
def test_hand_worked_draws(case):
    g, x = _gold()
    c = g["draws"][case]
    tok = orc.sample_node(x, g["prior"], [], g["W"], g["penalty"], g["temperature"],
                          c["top_p"], c["min_p"], c["u"])
    assert tok == c["token"]


def test_hand_worked_window_slides_along_the_tree_path():
    g, x = _gold()
    win = orc.penalty_window(g["prior"], g["depth1_drafted"], g["W"])
    assert list(win) == [2, 2, 5, 1]
    xp = orc.penalised_logits(x, win, g["penalty"], g["temperature"])
    expect = [8 ** 1.2, 4 ** (1 / 1.2), 0.5, 2.0, 1.0, 0.25]
    np.testing.assert_allclose(np.exp(xp.astype(np.float64)), expect, rtol=2e-6)


def test_penalty_direction_and_once_per_token():
    x = np.array([2.0, -2.0, 0.0, 1.0], dtype=np.float32)
    xp = orc.penalised_logits(x, [0, 0, 0, 1, 2], 1.2, 1.0)
    assert xp[0] < 2.0 and abs(xp[0] - 2 / 1.2) < 1e-6      # once, not three times
    assert xp[1] < -2.0 and abs(xp[1] + 2.4) < 1e-6
    assert xp[2] == 0.0 and xp[3] == 1.0


def test_temperature_scales_logits():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50).astype(np.float32)
    a = orc.penalised_logits(x, [], 1.2, 2.0)
    np.testing.assert_allclose(a, x / 2, rtol=1e-7)


def test_untruncated_draw_is_the_categorical_distribution():
    """top_p = 1, min_p = 0: the inverse-CDF draw maps the interval of u of
    length p_t to token t, so a uniform grid of N values of u hits token t
    N*p_t times up to one (p from the library softmax)."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(12) * 1.5).astype(np.float32)
    p = scipy.special.softmax(x.astype(np.float64))
    N = 20000
    counts = np.zeros(12)
    for n in range(N):
        counts[orc.sample_from_logits(x, 1.0, 0.0, (n + 0.5) / N)] += 1
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-9)


@pytest.mark.parametrize("top_p,min_p", [(1e-9, 0.0), (1.0, 1.0), (0.9, 1.0)])
def test_degenerate_truncation_is_greedy(top_p, min_p):
    rng = np.random.default_rng(4)
    x = rng.standard_normal(300).astype(np.float32)
    for u in (0.0, 0.3, 0.999):
        assert orc.sample_from_logits(x, top_p, min_p, u) == int(np.argmax(x))


def test_equal_probabilities_rank_by_token_id():
    x = np.zeros(5, dtype=np.float32)
    # five equal probabilities 0.2: top-p 0.5 keeps ranks with mass-before <= .5 -> ids 0,1,2
    assert orc.sample_from_logits(x, 0.5, 0.0, 0.99) == 2
    assert orc.sample_from_logits(x, 0.5, 0.0, 0.0) == 0


def _chain(depth, V=50):
    parents = np.array([-1] + list(range(depth)), dtype=np.int32)
    toks = np.arange(10, 10 + depth + 1, dtype=np.int32)
    return parents, toks


def test_chain_tree_known_path():
    parents, toks = _chain(3)
    V = 50
    logits = np.zeros((4, V), dtype=np.float32)
    logits[0, 11] = 40.0    # root predicts node 1's token
    logits[1, 12] = 40.0    # node 1 predicts node 2's token
    logits[2, 33] = 40.0    # node 2 predicts something else -> stop at node 2
    logits[3, 5] = 40.0
    prior = np.arange(20, 30, dtype=np.int32)
    prior[-1] = toks[0]
    u = np.full(4, 0.5, dtype=np.float32)
    args = (logits, prior, parents, toks, 8, 1.2, 1.0, 0.9, 0.05, u)
    path, bonus = orc.sample_accept_sequential(*args)
    assert path == [0, 1, 2] and bonus == 33
    samp = orc.sample_all_nodes(*args)
    assert orc.accept_from_samples(parents, toks, samp) == (path, bonus)


@pytest.mark.parametrize("wname,seed", [("tiny", 0), ("tiny", 1), ("tiny", 2)])
def test_parallel_form_equals_sequential_form(wname, seed):
    w = syn.scaled(syn.WORKLOADS[wname], V=2000, seed=seed)
    inp = syn.sampling_inputs(w, step=seed)
    args = (inp["logits"], inp["prior"], inp["parents"], inp["tokens"], w.W, w.penalty,
            w.temperature, w.top_p, w.min_p, inp["uniforms"])
    samp = orc.sample_all_nodes(*args)
    path, bonus = orc.accept_from_samples(inp["parents"], inp["tokens"], samp)
    assert (path, bonus) == orc.sample_accept_sequential(*args)
    # invariants: a root path whose every drafted token matches its parent's draw
    assert path[0] == 0
    for a, b in zip(path[:-1], path[1:]):
        assert inp["parents"][b] == a and inp["tokens"][b] == samp[a]
    assert bonus == samp[path[-1]]


def test_deepest_path_ties_go_to_lower_node():
    parents = np.array([-1, 0, 0, 1, 2], dtype=np.int32)
    toks = np.array([0, 7, 7, 8, 8], dtype=np.int32)
    sampled = np.array([7, 8, 8, 1, 2])
    path, bonus = orc.accept_from_samples(parents, toks, sampled)
    assert path == [0, 1, 3] and bonus == 1


def test_kv_commit_moves_accepted_rows():
    cache = np.arange(2 * 12 * 3).reshape(2, 12, 3)
    out = orc.kv_commit(cache, 5, [0, 2, 4])
    np.testing.assert_array_equal(out[:, 6], cache[:, 7])
    np.testing.assert_array_equal(out[:, 7], cache[:, 9])
    np.testing.assert_array_equal(out[:, :6], cache[:, :6])


def test_top_p_boundary_exceeds():
    """§D.1: the smallest set whose cumulative probability exceeds p.  Four
    equal probabilities 0.25, top_p 0.5: ranks 0 and 1 hold exactly 0.5,
    which does not exceed 0.5, so rank 2 joins (mass 0.75 > 0.5) and rank 3
    does not (the mass before it, 0.75, already exceeds 0.5)."""
    x = np.zeros(4, dtype=np.float32)
    assert orc.sample_from_logits(x, 0.5, 0.0, 0.99) == 2
    assert orc.sample_from_logits(x, 0.4999999, 0.0, 0.99) == 1
    assert orc.sample_from_logits(x, 0.7500001, 0.0, 0.99) == 3


def test_top_p_one_keeps_every_token():
    """No set can exceed a probability of 1: top_p = 1 keeps the whole
    vocabulary, so the last token of a long tail is still drawn at u near 1."""
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(5000) * 3).astype(np.float32)
    p = scipy.special.softmax(x.astype(np.float64))
    last = int(np.lexsort((np.arange(5000), -p))[-1])
    assert orc.sample_from_logits(x, 1.0, 0.0, 1.0 - 1e-12) == last
    _, info = orc.sample_from_logits(x, 1.0, 0.0, 0.5, return_info=True)
    assert info["n_keep"] == 5000


# --------------------------------------------------------------------------
# η-sampling (hand-worked: p = [1/2, 1/4, 1/8, 1/8])
# H = 1/2 ln 2 + 1/4 ln 4 + 2 * 1/8 ln 8 = (1/2 + 1/2 + 3/4) ln 2 = 1.75 ln 2
# exp(-H) = 2^-1.75 = 0.29730; with eps = 0.2, alpha = sqrt(0.2) = 0.44721:
# alpha exp(-H) = 0.13296 -> eta = 0.13296: K = {0, 1} (1/8 < eta), mass 3/4
# with eps = 0.1: alpha = sqrt(0.1), alpha exp(-H) = 0.09401 = eta -> K = all four
# --------------------------------------------------------------------------
def test_eta_hand_worked():
    x = np.log(np.array([0.5, 0.25, 0.125, 0.125]))
    p = np.array([0.5, 0.25, 0.125, 0.125])
    assert orc.eta_threshold(p, 0.2, np.sqrt(0.2)) == pytest.approx(np.sqrt(0.2) * 2 ** -1.75, rel=1e-12)
    assert orc.eta_threshold(p, 0.1, np.sqrt(0.1)) == pytest.approx(np.sqrt(0.1) * 2 ** -1.75, rel=1e-12)
    assert orc.eta_threshold(p, 0.05, 1.0) == pytest.approx(0.05, rel=1e-12)
    # K = {0, 1}: u*0.75 against cumulative 0.5, 0.75
    assert orc.sample_from_logits_eta(x, 0.2, np.sqrt(0.2), 0.5) == 0    # target .375
    assert orc.sample_from_logits_eta(x, 0.2, np.sqrt(0.2), 0.8) == 1    # target .6
    # K = all: ties between ids 2 and 3 rank id 2 first; cumulative .5 .75 .875 1
    assert orc.sample_from_logits_eta(x, 0.1, np.sqrt(0.1), 0.86) == 2   # target .86
    assert orc.sample_from_logits_eta(x, 0.1, np.sqrt(0.1), 0.9) == 3    # target .9


def test_eta_zero_epsilon_is_plain_categorical():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 3, size=200)
    p = np.exp(x - x.max())
    p /= p.sum()
    order = np.lexsort((np.arange(200), -p))
    c = np.cumsum(p[order])
    for u in rng.random(50):
        ref = int(order[int(np.argmax(c > u))])
        assert orc.sample_from_logits_eta(x, 0.0, 0.0, u) == ref


def test_literal_ctrl_penalty_divides_every_windowed_logit():
    """The literal CTRL form divides a windowed logit by theta whatever its
    sign: a negative logit moves toward zero (its token becomes MORE likely,
    the reason the sign-aware form is the default), zero stays zero."""
    x = np.array([2.0, -2.0, 0.0, 1.0], dtype=np.float32)
    xp = orc.penalised_logits(x, [0, 0, 1, 2], 1.2, 1.0, literal=True)
    assert abs(xp[0] - 2 / 1.2) < 1e-6 and abs(xp[1] + 2 / 1.2) < 1e-6
    assert xp[2] == 0.0 and xp[3] == 1.0
    # with every windowed logit positive the two forms agree
    y = np.array([0.5, 3.0, -1.0, 2.0], dtype=np.float32)
    np.testing.assert_array_equal(orc.penalised_logits(y, [0, 1, 3], 1.2, 0.7, literal=True),
                                  orc.penalised_logits(y, [0, 1, 3], 1.2, 0.7))


def test_literal_penalty_hand_worked_draw():
    """V = 3, logits [ln 2, -ln 2 * 1.2, 0], window {1}, theta 1.2, literal:
    x' = [ln 2, -ln 2, 0] so p = [2, 1/2, 1] / 3.5; with top_p = 1, min_p = 0
    the ranked order is (0, 2, 1) with cumulative [4/7, 6/7, 1]: u = 0.5 draws
    token 0, u = 0.6 token 2, u = 0.88 token 1.  The sign-aware form gives
    x'[1] = -1.44 ln 2 instead: p = [2, 2^-1.44, 1] / (3 + 2^-1.44), cumulative
    [0.594, 0.891, 1], so u = 0.88 draws token 2 there."""
    ln2 = math.log(2)
    x = np.array([ln2, -ln2 * 1.2, 0.0], dtype=np.float32)
    for u, tok in ((0.5, 0), (0.6, 2), (0.88, 1)):
        assert orc.sample_node(x, [1], [], 1, 1.2, 1.0, 1.0, 0.0, u, literal=True) == tok
    assert orc.sample_node(x, [1], [], 1, 1.2, 1.0, 1.0, 0.0, 0.88) == 2


def test_kv_append_places_rows_then_commit_moves_them():
    """Append then commit: the accepted nodes' own rows end at L, L+1, ...
    (hand-checked on a 1-head cache of 1-element rows)."""
    cache = np.zeros((1, 10, 1))
    rows = np.array([[[10.0], [11.0], [12.0], [13.0]]])       # nodes 0..3
    c = orc.kv_append(cache, 5, rows)
    assert c[0, :, 0].tolist() == [0, 0, 0, 0, 0, 10, 11, 12, 13, 0]
    c = orc.kv_commit(c, 5, [0, 2, 3])                         # path root -> 2 -> 3
    assert c[0, 5:8, 0].tolist() == [10, 12, 13]
