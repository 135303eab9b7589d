"""Pins for the oracle's tie accounting (CPU only).

The GPU parity tests forgive a differing draw or selected position only when
the oracle says its deciding quantity lies within 1e-5 of a cut.  These tests
pin the distances that decide that forgiveness to hand-worked values
(tests/golden/sampling_hand_worked.json, §D.1 / Table 11 of the paper
summary), check that the comparison helpers reject a difference outside the
band, and plant single mistakes in copies of the oracle's functions (on the
CPU) to show that each pin catches them.
"""
import inspect
import json
import math
import os
import types

import numpy as np
import pytest

from oracle import ts_oracle as orc
import parity_util as pu

GOLD = os.path.join(os.path.dirname(__file__), "golden", "sampling_hand_worked.json")
DIST_KEYS = ("top_p_last", "min_p_last", "first_cut", "draw_hi", "draw_lo")


def _gold():
    with open(GOLD) as f:
        g = json.load(f)
    ln = math.log
    logits = np.array([1.2 * ln(8), ln(4), -ln(2) / 1.2, ln(2), 0.0, -ln(4) / 1.2], dtype=np.float32)
    return g, logits


# --------------------------------------------------------------------------
# pins (each takes the oracle module, so the mutation tests can reuse them)
# --------------------------------------------------------------------------
def pin_sampling_margins(mod):
    """The hand-worked distances (exact fractions); the logits are fp32, so
    the oracle's p carries their rounding: relative tolerance 2e-6."""
    g, x = _gold()
    for e in g["margins"]:
        tok, info = mod.sample_node(x, g["prior"], [], g["W"], g["penalty"], g["temperature"],
                                    e["top_p"], e["min_p"], e["u"], return_info=True)
        assert tok == e["token"]
        assert info["n_keep"] == e["n_keep"] and info["rank"] == e["rank"]
        for k in DIST_KEYS:
            want = math.inf if e[k] is None else e[k]
            assert info["dist"][k] == pytest.approx(want, rel=2e-6, abs=1e-9), (k, e)
        assert info["margin"] == pytest.approx(min(math.inf if e[k] is None else e[k]
                                                   for k in DIST_KEYS), rel=2e-6)


def pin_eta_margins(mod):
    """p = [1/2, 1/4, 1/8, 1/8], eps = 0.2, alpha = sqrt(0.2):
    eta = sqrt(0.2) * 2^-1.75 = 0.132957; the pool is ranks {0, 1} (mass 3/4).
    eta_last = 0.25/eta - 1 = 0.880305; eta_first_cut = |0.125/eta - 1| =
    0.059848; u = 0.5: cumulative 2/3, 1 -> rank 0, draw_hi = 2/3 - 1/2."""
    x = np.log(np.array([0.5, 0.25, 0.125, 0.125]))
    eta = math.sqrt(0.2) * 2 ** -1.75
    tok, info = mod.sample_from_logits_eta(x, 0.2, math.sqrt(0.2), 0.5, return_info=True)
    assert tok == 0 and info["n_keep"] == 2 and info["rank"] == 0
    assert info["dist"]["eta_last"] == pytest.approx(0.25 / eta - 1, rel=1e-9)
    assert info["dist"]["eta_first_cut"] == pytest.approx(1 - 0.125 / eta, rel=1e-9)
    assert info["dist"]["draw_hi"] == pytest.approx(2 / 3 - 0.5, rel=1e-9)
    assert info["dist"]["draw_lo"] == math.inf
    assert info["margin"] == pytest.approx(1 - 0.125 / eta, rel=1e-9)


def pin_select_cut(mod):
    """Scores [9, 1, 5, 3, 7, 3, 8, 2], S = 1 sink, R = 1 recent, B = 3:
    the candidates are positions 1..6 with scores [1, 5, 3, 7, 3, 8]; ranked
    8, 7, 5, 3, 3, 1, the B-th best is 5, and their distances to it are
    [4, 0, 2, 2, 2, 3]."""
    imp = np.array([9, 1, 5, 3, 7, 3, 8, 2], dtype=np.float32)
    s_cut, dist = mod.select_cut_margin(imp, 8, 3, 1, 1)
    assert s_cut == 5.0
    np.testing.assert_array_equal(dist, [4, 0, 2, 2, 2, 3])
    # within the budget there is no cut
    s_cut, dist = mod.select_cut_margin(imp, 8, 6, 1, 1)
    assert s_cut == math.inf and dist.size == 0


def pin_top_p_exceeds(mod):
    """§D.1 wording: four equal masses 0.25 and top_p 0.5 keep three ranks."""
    x = np.zeros(4, dtype=np.float32)
    assert mod.sample_from_logits(x, 0.5, 0.0, 0.99) == 2
    assert mod.sample_from_logits(x, 0.4999999, 0.0, 0.99) == 1


def test_sampling_margins_hand_worked():
    pin_sampling_margins(orc)


def test_eta_margins_hand_worked():
    pin_eta_margins(orc)


def test_select_cut_margin_hand_worked():
    pin_select_cut(orc)


def test_top_p_exceeds():
    pin_top_p_exceeds(orc)


# --------------------------------------------------------------------------
# planted mistakes: each single-token change of the oracle's source must make
# its pin fail
# --------------------------------------------------------------------------
MUTATIONS = [
    # (original text, mutated text, pin)
    ("s_cut = np.sort(cand)[::-1][B - 1]", "s_cut = np.sort(cand)[::-1][B]", pin_select_cut),
    ("cand = imp_row[S:L - R]", "cand = imp_row[S:L - R + 1]", pin_select_cut),
    ("cand = imp_row[S:L - R]", "cand = imp_row[S - 1:L - R]", pin_select_cut),
    ('"top_p_last": abs(before[last] - top_p)', '"top_p_last": abs(before[last - 1] - top_p)',
     pin_sampling_margins),
    ('"top_p_last": abs(before[last] - top_p)', '"top_p_last": abs(before[last + 1] - top_p)',
     pin_sampling_margins),
    ('"min_p_last": abs(ratio[last] - min_p)', '"min_p_last": abs(ps[last] - min_p)',
     pin_sampling_margins),
    ('dist["first_cut"] = float(max(fails))', 'dist["first_cut"] = float(min(fails))',
     pin_sampling_margins),
    ('"draw_hi": abs(c[r] / c[-1] - u),\n            "draw_lo": abs(c[r - 1] / c[-1] - u) if r > 0 else inf}',
     '"draw_hi": abs(c[r] - u),\n            "draw_lo": abs(c[r - 1] / c[-1] - u) if r > 0 else inf}',
     pin_sampling_margins),
    ('"draw_hi": abs(c[r] / c[-1] - u),\n            "draw_lo": abs(c[r - 1] / c[-1] - u) if r > 0 else inf}',
     '"draw_hi": abs(c[r] / c[-1] - u),\n            "draw_lo": abs(c[r - 1] / c[-1] - u) if r > 1 else inf}',
     pin_sampling_margins),
    ('"eta_first_cut": rel(ps[n_keep]) if n_keep < V else inf',
     '"eta_first_cut": rel(ps[n_keep - 1]) if n_keep < V else inf', pin_eta_margins),
    ("rel = (lambda v: abs(v / eta - 1.0))", "rel = (lambda v: abs(v - eta))", pin_eta_margins),
    ("    return before <= top_p\n", "    return before < top_p\n", pin_top_p_exceeds),
]


def _mutated_oracle(original: str, mutated: str):
    src = inspect.getsource(orc)
    assert src.count(original) >= 1, f"mutation target not found: {original!r}"
    mod = types.ModuleType("ts_oracle_mutant")
    exec(compile(src.replace(original, mutated, 1), "ts_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("k", range(len(MUTATIONS)))
def test_pins_catch_planted_mistake(k):
    original, mutated, pin = MUTATIONS[k]
    pin(_mutated_oracle(original, original))      # the unmutated copy passes
    with pytest.raises((AssertionError, IndexError)):
        pin(_mutated_oracle(original, mutated))


# --------------------------------------------------------------------------
# the comparison helpers of the GPU parity tests
# --------------------------------------------------------------------------
def _with_clean_counts(fn):
    saved = {k: list(v) for k, v in pu.TIE_COUNTS.items()}
    try:
        return fn()
    finally:
        pu.TIE_COUNTS.clear()
        pu.TIE_COUNTS.update(saved)


def test_compare_draws_fails_outside_the_tie_band():
    g, x = _gold()
    xs = orc.penalised_logits(x, orc.penalty_window(g["prior"], [], g["W"]), g["penalty"],
                              g["temperature"])
    # u = 0.1 lies far from every cut (margin 0.05): a different token fails
    tok, info = orc.sample_from_logits(xs, 0.9, 0.2, 0.1, return_info=True)
    assert info["margin"] > pu.TIE
    with pytest.raises(AssertionError):
        _with_clean_counts(lambda: pu.compare_draws([tok + 1], [tok], [info]))
    assert _with_clean_counts(lambda: pu.compare_draws([tok], [tok], [info])) == 0
    # u one part in 10^7 below the cumulative kept mass of rank 0 (8/14):
    # draw_hi is ~1e-7, so a neighbouring token is a counted tie
    u = 8 / 14 - 1e-7
    tok, info = orc.sample_from_logits(xs, 0.9, 0.2, u, return_info=True)
    assert info["margin"] < pu.TIE and tok == 0
    assert _with_clean_counts(lambda: pu.compare_draws([1], [tok], [info])) == 1


def test_compare_selection_fails_outside_the_tie_band():
    imp = np.array([9, 1, 5, 3, 7, 3, 8, 2], dtype=np.float32)
    L, B, S, R = 8, 3, 1, 1
    ref = orc.select_partial(imp, L, B, S, R)                 # {0, 2, 4, 6, 7}
    assert ref.tolist() == [0, 2, 4, 6, 7]
    # position 3 (score 3) in place of position 2 (score 5, the cut): the
    # score 3 lies 2 away from the cut, far outside the band
    bad = np.array([[0, 3, 4, 6, 7]])
    with pytest.raises(AssertionError):
        _with_clean_counts(lambda: pu.compare_selection(bad, ref[None], imp[None], L, B, S, R))
    # an exact tie at the cut: scores [.., 5, .., 5, ..] at positions 2 and 3
    imp2 = np.array([9, 1, 5, 5, 7, 3, 8, 2], dtype=np.float32)
    ref2 = orc.select_partial(imp2, L, B, S, R)               # lower position wins
    assert ref2.tolist() == [0, 2, 4, 6, 7]
    swapped = np.array([[0, 3, 4, 6, 7]])
    assert _with_clean_counts(
        lambda: pu.compare_selection(swapped, ref2[None], imp2[None], L, B, S, R)) == 2
    # a sink that differs is never a tie
    nosink = np.array([[1, 2, 4, 6, 7]])
    with pytest.raises(AssertionError):
        _with_clean_counts(lambda: pu.compare_selection(nosink, ref[None], imp[None], L, B, S, R))
