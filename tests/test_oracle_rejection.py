"""Pins of the rejection-sampling acceptance oracle (App. A of the TokenSwift
paper: acceptance and rejection cases together reproduce the target's
distribution).  Hand-worked cases, the two degenerate drafts, and the
losslessness itself checked by a seeded Monte Carlo run against the target
distribution."""
import math

import numpy as np
import pytest
import scipy.special

from oracle import ts_oracle as orc

NOPEN = dict(prior=np.zeros(0, np.int32), W=0, penalty=1.2, temperature=1.0, top_p=1.0, min_p=0.0)


def _run(logits, q, parents, tokens, u_acc, u_draw, **kw):
    a = dict(NOPEN)
    a.update(kw)
    return orc.accept_rejection(np.asarray(logits, np.float32), q, a["prior"], parents, tokens,
                                a["W"], a["penalty"], a["temperature"], a["top_p"], a["min_p"],
                                u_acc, u_draw)


def test_hand_worked_two_tokens():
    """p = [3/4, 1/4], q = [1/4, 3/4], one child with token 1: it is accepted
    with probability p(1)/q(1) = 1/3.  u = 0.2 accepts (0.2 * 3/4 < 1/4); the
    bonus is then drawn at the child (p = [1/2, 1/2], u = 0.3 -> token 0).
    u = 0.5 rejects; the residual max(p - q, 0) = [1/2, 0] leaves token 0."""
    logits = [[math.log(0.75), math.log(0.25)], [0.0, 0.0]]
    q = [[0.25, 0.75], [0.5, 0.5]]
    parents, tokens = [-1, 0], [0, 1]
    assert _run(logits, q, parents, tokens, [0.0, 0.2], [0.9, 0.3]) == ([0, 1], 0)
    assert _run(logits, q, parents, tokens, [0.0, 0.2], [0.9, 0.7]) == ([0, 1], 1)
    for ud in (0.0, 0.5, 0.99):
        assert _run(logits, q, parents, tokens, [0.0, 0.5], [ud, 0.3]) == ([0], 0)


def test_draft_equal_to_target_accepts_the_first_child():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((4, 6)).astype(np.float32)
    q = np.stack([scipy.special.softmax(x.astype(np.float64)) for x in logits])
    parents, tokens = [-1, 0, 0, 0], [0, 2, 0, 5]
    for _ in range(50):
        path, _ = _run(logits, q, parents, tokens, rng.random(4), rng.random(4))
        assert path == [0, 1]


def test_draft_outside_the_target_support_rejects_and_keeps_the_target():
    """min_p = 0.5 keeps only token 0 of the root; a draft concentrated on
    token 3 is rejected at every child and the residual is the target
    itself, so the bonus is token 0 whatever the uniform."""
    logits = np.array([[3.0, 0.0, 0.0, -2.0], [0, 0, 0, 0], [0, 0, 0, 0]], np.float32)
    q = np.array([[0, 0, 0, 1.0], [0.25] * 4, [0.25] * 4])
    for ud in (0.0, 0.5, 0.99):
        assert _run(logits, q, [-1, 0, 0], [0, 3, 3], [0.0, 0.1, 0.9], [ud, 0, 0],
                    min_p=0.5) == ([0], 0)
    # without truncation a rejected draft leaves the full target: the bonus
    # is the plain inverse-CDF draw over token ids
    p = orc.target_distribution(logits[0], 1.0, 0.0)
    q2 = np.array([[0, 0, 0, 1.0], [0.25] * 4, [0.25] * 4])
    for ud in (0.05, 0.6, 0.97):
        p_res = np.maximum(p - q2[0], 0)
        want = orc.draw_in_id_order(p_res / p_res.sum(), ud)
        # token 3 is accepted iff u * 1 < p(3); take u above it
        assert _run(logits, q2, [-1, 0], [0, 3], [0.0, 0.999], [ud, 0])[1] == want


def test_lossless_first_token_follows_the_target():
    """App. A's claim: with the children drawn i.i.d. from q, the first
    committed token (the accepted child's token, else the bonus) is
    distributed as the target p, whatever q.  20,000 seeded trials per
    draft; every token's frequency within 5 standard errors of p."""
    rng = np.random.default_rng(12345)
    logits = np.array([[1.0, 0.2, -0.5, 0.7], [0, 0, 0, 0], [0, 0, 0, 0], [0, 0, 0, 0]],
                      np.float32)
    p = orc.target_distribution(logits[0], 1.0, 0.0)
    n = 20000
    for qrow in ([0.1, 0.5, 0.3, 0.1], [0.7, 0.1, 0.1, 0.1]):
        q = np.array([qrow, [0.25] * 4, [0.25] * 4, [0.25] * 4])
        counts = np.zeros(4)
        for _ in range(n):
            toks = rng.choice(4, size=3, p=q[0])
            path, bonus = _run(logits, q, [-1, 0, 0, 0], [0, *toks], rng.random(4), rng.random(4))
            first = int(toks[path[1] - 1]) if len(path) > 1 else bonus
            counts[first] += 1
        f = counts / n
        se = np.sqrt(p * (1 - p) / n)
        assert np.all(np.abs(f - p) <= 5 * se), (qrow, f, p)
