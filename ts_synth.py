"""Seeded synthetic inputs for the TokenSwift decode hot path.

This module only *makes inputs*: query/key/value tensors, draft trees, logits,
penalty windows and the per-node uniforms.  It holds none of the method's
arithmetic (no attention, no selection, no sampling), so both the CPU oracle
tests and the CUDA path tests can take their inputs from here without sharing
any computation.

The workloads stand in for the PG-19 prompts and the LLaMA / Qwen models of
"TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation"
(§4.1 Setup): the datasets and weights are not available, so the tensors are
seeded Gaussians with the shapes of those models, planted heavy-hitter keys,
a [1,3,3,3] draft tree merged with n-gram chains (§4.4.1, §B.2), and
N(0, 3^2) logits.

bf16 values are carried as raw uint16 bit patterns (round-to-nearest-even from
float32), so every consumer decodes exactly the same numbers.
"""
from __future__ import annotations

import dataclasses
import numpy as np

MASK64 = (1 << 64) - 1


# --------------------------------------------------------------------------
# workload shapes
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    Hq: int
    Hkv: int
    d: int
    L: int            # committed cache length
    T: int            # draft tree nodes
    tree: str         # "random" or "trie"
    B: int            # partial-cache budget (top-B)
    S: int            # attention-sink tokens kept
    R: int            # recent tokens kept
    n_imp: int        # importance computed from the last n_imp tree queries
    V: int            # vocabulary
    W: int            # contextual-penalty window
    planted: int      # planted heavy-hitter keys per KV head
    seed: int
    penalty: float = 1.2
    temperature: float = 1.0
    top_p: float = 0.9
    min_p: float = 0.05

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def L_cap(self) -> int:
        return self.L + self.T

    @property
    def N(self) -> int:
        return min(self.L, self.S + self.B + self.R)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 1, 64, 4096, 16, "random", 1024, 4, 64, 16,
                     32000, 1024, 32, 0),
    "qwen2.5-1.5b": Workload("qwen2.5-1.5b", 28, 12, 2, 128, 32768, 64, "trie",
                             4096, 4, 64, 64, 151936, 1024, 256, 1),
    "llama3.1-8b": Workload("llama3.1-8b", 32, 32, 8, 128, 102400, 64, "trie",
                            4096, 4, 64, 64, 128256, 1024, 256, 2),
    "mha-7b": Workload("mha-7b", 32, 32, 32, 128, 102400, 64, "trie",
                       4096, 4, 64, 64, 32000, 1024, 256, 3),
    "qwen2.5-14b": Workload("qwen2.5-14b", 48, 40, 8, 128, 102400, 64, "trie",
                            4096, 4, 64, 64, 152064, 1024, 256, 4),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    return dataclasses.replace(w, **kw)


# --------------------------------------------------------------------------
# bf16 bit patterns
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# counter-based uniforms (one per tree node)
# --------------------------------------------------------------------------
def splitmix64(x: int) -> int:
    """SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def node_uniforms(seed: int, step: int, T: int) -> np.ndarray:
    """u[i] = top 24 bits of splitmix64(seed ^ step<<32 ^ i) * 2^-24, in [0, 1)."""
    out = np.empty(T, dtype=np.float32)
    for i in range(T):
        z = splitmix64((seed ^ ((step << 32) & MASK64) ^ i) & MASK64)
        out[i] = np.float32((z >> 40) * (2.0 ** -24))
    return out


def ngram_rand_keys(seed: int, step: int, cap: int) -> np.ndarray:
    """Random keys of the root's stored n-gram continuations for one step
    (slot i, oldest first): top 31 bits of splitmix64(seed ^ step<<32 ^
    (1<<31 | i)), as int32 (non-negative)."""
    out = np.empty(cap, dtype=np.int32)
    for i in range(cap):
        z = splitmix64((seed ^ ((step << 32) & MASK64) ^ (0x80000000 | i)) & MASK64)
        out[i] = np.int32(z >> 33)
    return out


# --------------------------------------------------------------------------
# draft trees
# --------------------------------------------------------------------------
def random_tree(rng: np.random.Generator, T: int, V: int, max_depth: int = 3):
    """Random parent array: parent[i] uniform over earlier nodes whose depth is
    below max_depth, so every root-to-leaf path has at most max_depth+1 nodes."""
    parents = np.full(T, -1, dtype=np.int32)
    depth = np.zeros(T, dtype=np.int32)
    for i in range(1, T):
        ok = np.nonzero(depth[:i] < max_depth)[0]
        p = int(ok[rng.integers(len(ok))])
        parents[i] = p
        depth[i] = depth[p] + 1
    tokens = rng.integers(0, V, size=T, dtype=np.int64).astype(np.int32)
    return parents, tokens


def trie_tree(rng: np.random.Generator, T: int, V: int,
              branching=(3, 3, 3), n_ngrams: int = 20, ngram_len: int = 3):
    """Draft tree of the shape the pages use: the ternary full tree [1,3,3,3]
    (§4.4.1 Tree Configuration, §B.2 Inference Details) holding the extra
    heads' candidates, with up to k=20 retrieved n-gram continuations
    (Table 11) merged in as a trie under the root.  Nodes are numbered in
    insertion order, so parent[i] < i.  Trimmed, or padded with extra
    children of shallow nodes, to exactly T nodes; depth <= len(branching)."""
    max_depth = len(branching)
    parents, tokens, depth = [-1], [int(rng.integers(V))], [0]
    kids = [dict()]

    def add(p, tok):
        parents.append(p)
        tokens.append(tok)
        depth.append(depth[p] + 1)
        kids.append(dict())
        kids[p][tok] = len(parents) - 1
        return len(parents) - 1

    level = [0]
    for b in branching:
        nxt = []
        for p in level:
            for _ in range(b):
                if len(parents) >= T:
                    break
                tok = int(rng.integers(V))
                while tok in kids[p]:
                    tok = int(rng.integers(V))
                nxt.append(add(p, tok))
        level = nxt
    for _ in range(n_ngrams):
        seq = [int(t) for t in rng.integers(0, V, size=ngram_len)]
        node = 0
        for tok in seq:
            if tok in kids[node]:
                node = kids[node][tok]
            elif len(parents) < T and depth[node] < max_depth:
                node = add(node, tok)
            else:
                break
    while len(parents) < T:
        shallow = [i for i in range(len(parents)) if depth[i] < max_depth]
        p = shallow[int(rng.integers(len(shallow)))]
        tok = int(rng.integers(V))
        if tok not in kids[p]:
            add(p, tok)
    return np.asarray(parents[:T], dtype=np.int32), np.asarray(tokens[:T], dtype=np.int32)


def make_tree(w: Workload, rng: np.random.Generator):
    if w.tree == "random":
        return random_tree(rng, w.T, w.V)
    return trie_tree(rng, w.T, w.V)


# --------------------------------------------------------------------------
# attention inputs
# --------------------------------------------------------------------------
def layer_rng(w: Workload, layer: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, layer, stream]))


def attention_inputs(w: Workload, layer: int = 0, L: int | None = None,
                     plant: bool = True, tree=None):
    """Q [T,Hq,d], K/V [Hkv,L_cap,d] as bf16 bits, plus the tree parents.

    K/V rows [0, L) are the committed cache, rows [L, L+T) are the tree's own
    keys/values (written by the verification forward), rows beyond are zero.
    Heavy hitters: `planted` keys per KV head at random positions in
    [S, L-R), each sqrt(d) * normalize(0.9*qhat + 0.1*xi) where qhat is the
    unit direction of the summed importance queries of that head's group and
    xi a random unit vector (cosine to qhat > 0.8 after bf16 rounding).
    """
    L = w.L if L is None else L
    rng = layer_rng(w, layer)
    T, Hq, Hkv, d = w.T, w.Hq, w.Hkv, w.d
    L_cap = L + T
    if tree is None:
        parents, tokens = make_tree(w, rng)
    else:
        parents, tokens = tree
    q = rng.standard_normal((T, Hq, d), dtype=np.float32)
    qb = f32_to_bf16_bits(q)
    qd = bf16_bits_to_f32(qb).astype(np.float64)
    kb = np.zeros((Hkv, L_cap, d), dtype=np.uint16)
    vb = np.zeros((Hkv, L_cap, d), dtype=np.uint16)
    lo, hi = w.S, L - w.R
    n_pl = min(w.planted, max(hi - lo, 0)) if plant else 0
    planted = np.zeros((Hkv, n_pl), dtype=np.int64)
    G = w.G
    n_imp = w.n_imp if w.n_imp > 0 else T
    for h in range(Hkv):
        kh = rng.standard_normal((L + T, d), dtype=np.float32)
        vh = rng.standard_normal((L + T, d), dtype=np.float32)
        if n_pl > 0:
            direction = qd[T - n_imp:, h * G:(h + 1) * G, :].reshape(-1, d).sum(axis=0)
            qhat = direction / np.linalg.norm(direction)
            pos = np.sort(rng.choice(np.arange(lo, hi), size=n_pl, replace=False))
            planted[h] = pos
            for j in pos:
                xi = rng.standard_normal(d)
                xi /= np.linalg.norm(xi)
                kk = 0.9 * qhat + 0.1 * xi
                kh[j] = (np.sqrt(d) * kk / np.linalg.norm(kk)).astype(np.float32)
        kb[h, :L + T] = f32_to_bf16_bits(kh)
        vb[h, :L + T] = f32_to_bf16_bits(vh)
    return dict(q=qb, k=kb, v=vb, parents=parents, tokens=tokens, L=L,
                L_cap=L_cap, planted=planted)


# --------------------------------------------------------------------------
# sampling inputs
# --------------------------------------------------------------------------
def sampling_inputs(w: Workload, step: int = 0, tree=None, plant_accept: float = 0.7,
                    logit_std: float = 3.0):
    """Logits [T,V] fp32 ~ N(0, logit_std^2), a window of W uniform prior
    token ids ending with the root token, the tree, and one uniform per node.

    To make acceptance non-trivial, with probability `plant_accept` a node's
    first child's token gets +30 on that node's logits (so the target's own
    sample tends to match the draft)."""
    rng = np.random.Generator(np.random.PCG64([w.seed, 1_000_003, step]))
    if tree is None:
        parents, tokens = make_tree(w, rng)
    else:
        parents, tokens = tree
    T, V, W = w.T, w.V, w.W
    logits = (rng.standard_normal((T, V), dtype=np.float32) * np.float32(logit_std)).astype(np.float32)
    first_child = np.full(T, -1, dtype=np.int64)
    for i in range(T - 1, 0, -1):
        first_child[parents[i]] = i
    for i in range(T):
        c = first_child[i]
        if c >= 0 and rng.random() < plant_accept:
            logits[i, tokens[c]] += np.float32(30.0)
    prior = rng.integers(0, V, size=W, dtype=np.int64).astype(np.int32)
    prior[-1] = tokens[0]
    u = node_uniforms(w.seed, step, T)
    return dict(logits=logits, prior=prior, parents=np.asarray(parents, np.int32),
                tokens=np.asarray(tokens, np.int32), uniforms=u)


# --------------------------------------------------------------------------
# standalone importance scores (selection tests)
# --------------------------------------------------------------------------
def importance_scores(Hkv: int, L: int, seed: int, std: float = 16.0,
                      grid: float | None = None, n_heavy: int = 256):
    """fp32 importance-like scores [Hkv, L]: N(0, std^2), optionally rounded
    to a grid (creating exact ties), with n_heavy positions raised far above
    the rest (the heavy hitters)."""
    rng = np.random.Generator(np.random.PCG64([seed, 77]))
    s = rng.standard_normal((Hkv, L)) * std
    if grid:
        s = np.round(s / grid) * grid
    for h in range(Hkv):
        if n_heavy and L > 0:
            pos = rng.choice(L, size=min(n_heavy, L), replace=False)
            s[h, pos] += 10 * std
    return s.astype(np.float32)
