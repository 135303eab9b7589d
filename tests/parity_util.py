"""Helpers shared by the GPU parity tests: upload seeded inputs, run the
oracle, compare with the tolerances and tie accounting of the hot path.

Tolerances:
  attention output: per (node, head) row, ||o - o_ref||_2 / ||o_ref||_2 <= 2e-3;
  log-sum-exp: |lse - lse_ref| <= 2e-3;
  importance: |imp - imp_ref| <= 1e-5 * ||qsum|| * ||k_j|| / sqrt(d)
      (a float32 dot product of d terms errs by at most ~d * 2^-24 of the
      Cauchy-Schwarz bound; 1e-5 leaves room for d = 128);
  index sets and tokens: bit-exact, except positions or nodes whose deciding
      quantity lies within 1e-5 of its cut (counted and reported as ties).
"""
from __future__ import annotations

import collections

import numpy as np
import torch

from oracle import ts_oracle as orc

ATTN_RTOL = 2e-3
LSE_ATOL = 2e-3
TIE = 1e-5

# near-ties seen in this pytest session, by kind ("draw", "selection", ...):
# [number of compared items, number of counted ties]; printed by the
# terminal-summary hook of conftest.py
TIE_COUNTS: dict = collections.defaultdict(lambda: [0, 0])


def record_ties(kind: str, compared: int, ties: int) -> None:
    TIE_COUNTS[kind][0] += int(compared)
    TIE_COUNTS[kind][1] += int(ties)


def compare_draws(got, ref, infos, kind: str = "draw") -> int:
    """Sampled tokens must equal the oracle's, except at nodes whose oracle
    margin (the smallest distance of a deciding quantity to its cut, from
    sample_from_logits / sample_from_logits_eta with return_info) is below
    TIE.  Returns the number of such tied nodes that differ; raises on any
    other difference."""
    got = np.asarray(got).tolist()
    ref = np.asarray(ref).tolist()
    assert len(got) == len(ref), f"{len(got)} draws against {len(ref)}"
    ties = 0
    for i, (g, r) in enumerate(zip(got, ref)):
        if g != r:
            m = infos[i]["margin"]
            assert m < TIE, (f"node {i}: gpu {g} oracle {r} margin {m:.2e} "
                             f"({infos[i].get('dist')})")
            ties += 1
    record_ties(kind, len(ref), ties)
    return ties


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def attention_rel_err(o: np.ndarray, o_ref: np.ndarray) -> np.ndarray:
    num = np.linalg.norm(o - o_ref, axis=-1)
    den = np.linalg.norm(o_ref, axis=-1)
    return num / np.maximum(den, 1e-30)


# largest attention row error (relative, per row) and LSE error seen by the
# parity checks of this session, reported in the pytest summary
ERR_MAX = {"attention rel": 0.0, "lse abs": 0.0}


def check_attention(o, lse, o_ref, lse_ref):
    rel = attention_rel_err(o.astype(np.float64), o_ref)
    ERR_MAX["attention rel"] = max(ERR_MAX["attention rel"], float(rel.max()))
    assert rel.max() <= ATTN_RTOL, f"attention rel err {rel.max():.3e} > {ATTN_RTOL}"
    if lse is not None:
        d = np.abs(lse.astype(np.float64) - lse_ref)
        ERR_MAX["lse abs"] = max(ERR_MAX["lse abs"], float(d.max()))
        assert d.max() <= LSE_ATOL, f"lse abs err {d.max():.3e}"
    return float(rel.max())


def check_importance(imp, imp_ref, q64, k64, n_imp, G):
    T, Hq, d = q64.shape
    Hkv, L = imp_ref.shape
    worst = 0.0
    if L == 0:
        return worst
    for kv in range(Hkv):
        qs = q64[T - n_imp:, kv * G:(kv + 1) * G, :].sum(axis=(0, 1))
        bound = 1e-5 * np.linalg.norm(qs) * np.linalg.norm(k64[kv, :L], axis=1) / np.sqrt(d)
        err = np.abs(imp[kv].astype(np.float64) - imp_ref[kv])
        assert np.all(err <= bound + 1e-30), f"imp err {err.max():.3e} (head {kv})"
        worst = max(worst, float((err / np.maximum(bound, 1e-30)).max()))
    return worst


def compare_selection(idx_gpu, idx_ref, imp_rank, L, B, S, R):
    """Kept sets must agree except for positions whose ranking score lies
    within TIE * max(1, |s_cut|) of the B-th best score.  Returns the number
    of such tied positions that differ."""
    ties = 0
    for kv in range(idx_ref.shape[0]):
        a, b = set(idx_gpu[kv].tolist()), set(idx_ref[kv].tolist())
        if a == b:
            continue
        s_cut, _ = orc.select_cut_margin(imp_rank[kv], L, B, S, R)
        band = TIE * max(1.0, abs(s_cut))
        for j in a ^ b:
            assert S <= j < L - R, f"head {kv}: sink/recent position {j} differs"
            assert abs(imp_rank[kv][j] - s_cut) <= band, (
                f"head {kv}: position {j} score {imp_rank[kv][j]} differs outside the tie band "
                f"around {s_cut}")
            ties += 1
    record_ties("selection", int(np.asarray(idx_ref).size), ties)
    return ties
