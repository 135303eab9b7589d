"""KV-head sharding of one decode stream across ranks.

Verification attention, importance, top-B selection and gather are
independent per (layer, KV head) ("TokenSwift: Lossless Acceleration of Ultra
Long Sequence Generation", §3.3: GQA query heads are partitioned per KV head
and their scores aggregated), so one stream can be split across ranks by KV
head with no exchange inside the hot path: rank r owns KV heads
[lo_r, hi_r) and the query heads of their groups.  Only the step's sampling
needs the whole vocabulary row, which the model's output layer already gives
every rank.  This module holds the host-side bookkeeping; every rank runs the
ordinary library calls on its slices.
"""
from __future__ import annotations


def kv_head_range(Hkv: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced KV-head range [lo, hi) owned by `rank`."""
    if not (0 <= rank < world) or Hkv < 1:
        raise ValueError("need 0 <= rank < world and Hkv >= 1")
    base, extra = divmod(Hkv, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def query_head_range(Hq: int, Hkv: int, rank: int, world: int) -> tuple[int, int]:
    """Query heads of the groups owned by `rank` (head h belongs to KV head h // G)."""
    G = Hq // Hkv
    lo, hi = kv_head_range(Hkv, rank, world)
    return lo * G, hi * G


def shard_layer(q, k, v, rank: int, world: int):
    """Slices of one layer's tensors owned by `rank`: q [T, Hq, d] -> its query
    heads, k/v [Hkv, L_cap, d] -> its KV heads (views; contiguous for k/v)."""
    Hq, Hkv = q.shape[1], k.shape[0]
    qlo, qhi = query_head_range(Hq, Hkv, rank, world)
    lo, hi = kv_head_range(Hkv, rank, world)
    return q[:, qlo:qhi], k[lo:hi], v[lo:hi]
