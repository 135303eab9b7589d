"""CPU oracle for the TokenSwift per-step decode hot path.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain, fp64 statement of
what the hot path computes, used to check the CUDA library.  Only the test
suite, the package's smoke check and the benchmark's CPU-baseline leg may
import it; the product path never does.  It shares no code with the CUDA
path: its only inputs are numpy arrays (bf16 arrives as uint16 bit patterns,
decoded here).

Source: "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation"
(Wu, Shen, Jia, Wang, Zheng; ICML 2025), as summarised on the pages studied:
  * §3.1 Overview / Figure 2: drafting on a partial KV cache, verification on
    the full cache, exact-match acceptance of the longest valid draft, then
    n-gram table and KV cache update.
  * §E Tree-Based Attention: each tree token attends only to its predecessors.
  * §3.3 Dynamic KV Cache Management: fixed budget, the initial |S| pairs are
    kept, importance = query-key dot products, GQA scores aggregated per group.
  * §3.4 Contextual Penalty: a penalty on the most recent W tokens.
  * §D.1 Sampling algorithms: top-p keeps the smallest set whose cumulative
    probability exceeds p; min-p keeps tokens above p_base * p_max.
  * Table 11: k=20, temperature 1.0, top-p 0.9, min-p 0.05, penalty 1.2,
    penalty length 1024.
  * A. Lossless Nature of Speculative Decoding: acceptance and rejection
    cases together reproduce the target distribution (accept_rejection).

Readings taken where the pages are silent: CTRL-style penalty is sign-aware
(positive logits divided by theta, non-positive multiplied); a windowed token
is penalised once whatever its count; top-p and min-p are intersected on the
same post-temperature distribution; top-p keeps rank r iff the mass before r
is <= p (the smallest set whose mass exceeds p), and everything when p >= 1; one uniform per node drives an inverse-CDF draw over the kept
set in (p desc, id asc) order; importance is the raw scaled dot product summed
over the group's heads and the last n_imp tree queries; sinks and the recent
window are kept outside the top-B competition; ties in importance go to the
lower position.

Precision: scores, softmax and importance in fp64.  Where floating point
decides an integer, the decision is taken in the precision the library
stores the deciding quantity in: importance is rounded to fp32 before the
top-B ranking (the library's imp array is fp32), and the penalised,
temperature-scaled logits are formed with fp32 operations before ranking
(the logits arrive as fp32).  Probabilities and their sums stay fp64.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# input decoding
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# draft tree
# --------------------------------------------------------------------------
def root_paths(parents) -> list[list[int]]:
    """For every node i, the nodes from the root down to i (inclusive).

    §E Tree-Based Attention: a tree token attends to its predecessors, i.e.
    the chain of parents up to the root, plus itself."""
    T = len(parents)
    paths = []
    for i in range(T):
        chain = []
        a = i
        while a != -1:
            chain.append(a)
            a = int(parents[a])
        paths.append(chain[::-1])
    return paths


# --------------------------------------------------------------------------
# (a1, a2) tree verification attention + attention importance
# --------------------------------------------------------------------------
def verify_attention(q, k, v, L: int, parents, n_imp: int = 0):
    """Tree-masked GQA/MHA attention of the T draft-tree queries against the
    full KV cache, and the per-position importance of the cache.

    q: [T, Hq, d] float64 (post-RoPE queries of the tree tokens)
    k, v: [Hkv, >= L+T, d] float64; rows [0, L) are the committed cache,
          row L+a holds tree node a's own key/value.
    parents: [T] int, parents[0] = -1, parents[i] < i.

    For node i and query head h (KV head kv = h // G, contiguous grouping):
        s_j = q[i,h] . k[kv,j] / sqrt(d),  j in [0, L)  or  j = L+a, a on the
              root path of i                                   (§3.1, §E)
        O[i,h]   = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m),  m = max_j s_j
        LSE[i,h] = m + ln sum_j exp(s_j - m)
    Importance (§3.3: query-key dot products; GQA queries partitioned, their
    scores aggregated per group):
        imp[kv, j] = sum over the last n_imp nodes i and the heads h of group
                     kv of s_{i,h,j},  for cache positions j in [0, L) only.
    Returns O [T,Hq,d], LSE [T,Hq], imp [Hkv, L] (all float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[0]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    n_imp = T if n_imp <= 0 else n_imp
    scale = 1.0 / np.sqrt(d)
    paths = root_paths(parents)

    O = np.zeros((T, Hq, d))
    LSE = np.zeros((T, Hq))
    imp = np.zeros((Hkv, L))
    for h in range(Hq):
        kv = h // G
        # scores of every tree query of head h against the committed cache
        s_cache = (q[:, h, :] @ k[kv, :L, :].T) * scale           # [T, L]
        # scores against the tree rows each node may see (its root path)
        s_tree = [(k[kv, [L + a for a in paths[i]], :] @ q[i, h, :]) * scale for i in range(T)]
        m = np.array([max(s_cache[i].max() if L > 0 else -np.inf, s_tree[i].max())
                      for i in range(T)])                          # row maxima
        w_cache = np.exp(s_cache - m[:, None])                     # [T, L]
        num = w_cache @ v[kv, :L, :]                               # [T, d]
        Z = w_cache.sum(axis=1)
        for i in range(T):
            w_tree = np.exp(s_tree[i] - m[i])
            num[i] += w_tree @ v[kv, [L + a for a in paths[i]], :]
            Z[i] += w_tree.sum()
        O[:, h, :] = num / Z[:, None]
        LSE[:, h] = m + np.log(Z)
        for i in range(T - n_imp, T):
            imp[kv] += s_cache[i]
    return O, LSE, imp


def importance_softmax(q, k, L: int, lse, n_imp: int = 0):
    """(NEXT-4) Softmax-weighted importance: the attention probability each
    committed cache position receives from the importance queries of its
    KV head's group.

    §3.3 Dynamic KV Cache Management ranks cache pairs by query-key scores,
    the queries of a GQA group partitioned and their scores aggregated.  This
    variant aggregates the normalised attention weights instead of the raw
    scores (the pages do not define this variant; this is the plain reading
    of "aggregate the group's attention" with softmax weights):

        imp[kv, j] = sum over the last n_imp nodes i and the heads h of
                     group kv of exp(q[i,h] . k[kv,j] / sqrt(d) - lse[i,h]),
                     j in [0, L),

    lse [T, Hq] being each row's log-sum-exp over everything the row attends
    to (the committed cache and its root path of the tree), as returned by
    verify_attention.  q [T,Hq,d], k [Hkv, >= L, d] float64.  Returns
    imp [Hkv, L] float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    n_imp = T if n_imp <= 0 else n_imp
    scale = 1.0 / np.sqrt(d)
    imp = np.zeros((Hkv, L))
    for h in range(Hq):
        kv = h // G
        for i in range(T - n_imp, T):
            s = (k[kv, :L, :] @ q[i, h, :]) * scale
            imp[kv] += np.exp(s - lse[i, h])
    return imp


# --------------------------------------------------------------------------
# (a3, a4) partial KV cache: top-B selection + gather
# --------------------------------------------------------------------------
def select_partial(imp_row, L: int, B: int, S: int, R: int) -> np.ndarray:
    """Positions kept in one KV head's partial (draft) cache, ascending.

    §3.3: a fixed budget; the initial |S| pairs (attention sinks) are always
    preserved and less important pairs are replaced.  The recent window of R
    positions is also always kept.  The top-B competition runs over
    [S, L-R) ranked by (importance desc, position asc).  When the whole
    cache fits the budget (L <= S+B+R) every position is kept.

    imp_row: importance of positions [0, L), in the precision the library
    ranks it (fp32 values, carried here as float64)."""
    imp_row = np.asarray(imp_row, dtype=np.float64)
    if L <= S + B + R:
        return np.arange(L, dtype=np.int64)
    cand = np.arange(S, L - R, dtype=np.int64)
    order = np.lexsort((cand, -imp_row[cand]))   # primary: -imp asc; then position asc
    top = cand[order[:B]]
    keep = np.concatenate([np.arange(S), top, np.arange(L - R, L)])
    return np.sort(keep)


def gather_rows(cache_head, idx) -> np.ndarray:
    """Compact draft cache of one KV head: rows idx of the full cache, copied
    bit for bit (§3.1: the partial KV cache used for drafting)."""
    return np.asarray(cache_head)[np.asarray(idx, dtype=np.int64)].copy()


def refresh_incremental(slots_prev, kept_new, cache_head, compact_prev):
    """(NEXT-4) Incremental update of one KV head's partial cache.

    §3.3: the budgeted cache keeps its initial |S| pairs and replaces the
    less important pairs as generation proceeds.  The pages give no slot
    rule; the one taken here: a slot keeps its row while its position stays
    selected; the rows of newly selected positions are written into the slots whose positions
    left the selection, and past the old slot count while the cache is still
    growing (L <= S+B+R).  Freed slots are filled in ascending slot order by
    the added positions in ascending position order.  Attention over the
    partial cache does not depend on the slot order.

    slots_prev   [N_prev] positions held by slots 0..N_prev-1 (distinct)
    kept_new     the new kept positions (select_partial's output)
    cache_head   [>= L, d] the full cache rows of this head
    compact_prev [>= N_new, d] the partial cache rows before the update
    Returns (slots_new [N_new], compact_new [N_new, d], rows_written)."""
    slots_prev = [int(x) for x in slots_prev]
    kept = [int(x) for x in kept_new]
    N_prev, N_new = len(slots_prev), len(kept)
    assert N_new >= N_prev, "the kept set never shrinks"
    kept_set, prev_set = set(kept), set(slots_prev)
    freed = [s for s in range(N_prev) if slots_prev[s] not in kept_set]
    added = sorted(j for j in kept if j not in prev_set)
    targets = freed + list(range(N_prev, N_new))
    assert len(targets) == len(added)
    slots = slots_prev + [-1] * (N_new - N_prev)
    out = np.array(compact_prev[:N_new], copy=True)
    for s, j in zip(targets, added):
        slots[s] = j
        out[s] = cache_head[j]
    return np.asarray(slots, dtype=np.int64), out, len(added)


def select_cut_margin(imp_row, L: int, B: int, S: int, R: int) -> tuple[float, np.ndarray]:
    """The B-th best candidate score s_cut, and for every candidate its
    distance to s_cut (used to count near-ties between implementations)."""
    imp_row = np.asarray(imp_row, dtype=np.float64)
    if L <= S + B + R:
        return np.inf, np.zeros(0)
    cand = imp_row[S:L - R]
    s_cut = np.sort(cand)[::-1][B - 1]
    return float(s_cut), np.abs(cand - s_cut)


# --------------------------------------------------------------------------
# (a5, a6) contextual penalty + temperature + top-p / min-p + draw
# --------------------------------------------------------------------------
def penalty_window(prior, path_tokens, W: int) -> np.ndarray:
    """The most recent W tokens at a tree node (§3.4): the committed history
    `prior` (which ends with the root token) followed by the drafted tokens
    on the root path of the node, root excluded; the last W of these."""
    seq = np.concatenate([np.asarray(prior, dtype=np.int64),
                          np.asarray(path_tokens, dtype=np.int64)])
    return seq[len(seq) - W:] if W > 0 else seq[:0]


def penalised_logits(x, window, penalty: float, temperature: float,
                     literal: bool = False) -> np.ndarray:
    """CTRL-style contextual penalty on the windowed tokens, then temperature.

    Each distinct token in the window is penalised once: x/theta if x > 0,
    x*theta otherwise (§3.4, §4.3.3, Table 11 theta = 1.2); with `literal`,
    the CTRL form as written, x/theta whatever the sign.  Every logit is
    then divided by the temperature.  Formed with fp32 operations, the
    precision the logits arrive in."""
    x = np.asarray(x, dtype=np.float32).copy()
    th = np.float32(penalty)
    for t in np.unique(np.asarray(window, dtype=np.int64)):
        xt = x[t]
        x[t] = xt / th if (literal or xt > 0) else xt * th
    return (x / np.float32(temperature)).astype(np.float32)


def _top_p_keep(before, top_p: float) -> np.ndarray:
    """top-p (§D.1): the smallest set of leading ranks whose cumulative
    probability exceeds p.  Rank r belongs to it iff the ranks before r do
    not yet exceed p, i.e. their mass is <= top_p.  With top_p >= 1 no set
    can exceed p and every rank is kept."""
    if top_p >= 1.0:
        return np.ones(len(before), dtype=bool)
    return before <= top_p


def sample_from_logits(x_pen, top_p: float, min_p: float, u: float, return_info: bool = False):
    """Draw one token from penalised logits with top-p and min-p truncation.

    p = softmax(x') in fp64.  Tokens are ranked by (p desc, id asc).
    top-p (§D.1): keep the smallest prefix of ranks whose mass exceeds p:
        rank r is kept iff the mass of ranks before r is <= top_p
        (top_p >= 1 keeps every rank).
    min-p (§D.1): keep tokens with p >= min_p * p_max.
    Both are applied (Table 11 sets both); the kept set K is their
    intersection, which always holds rank 0.  The draw is the smallest rank r
    in K whose cumulative mass over K exceeds u * mass(K).

    With return_info, also the distance of each deciding quantity to its cut
    (used to recognise near-ties between implementations):
      top_p_last  mass before the last kept rank vs top_p
      min_p_last  p/p_max of the last kept rank vs min_p
      first_cut   the first cut rank: it would join K only if every filter
                  that cuts it flipped, so the largest of their distances
      draw_hi     cumulative kept mass at the drawn rank / mass(K) vs u
      draw_lo     the same one rank earlier
    Distances are inf where the quantity does not exist (rank 0 is never
    cut; no rank follows the last).  margin = the smallest of them.
    """
    x = np.asarray(x_pen, dtype=np.float64)
    V = x.shape[0]
    m = x.max()
    e = np.exp(x - m)
    p = e / e.sum()
    ids = np.arange(V)
    order = np.lexsort((ids, -p))
    ps = p[order]
    before = np.concatenate([[0.0], np.cumsum(ps)[:-1]])
    ratio = ps / ps[0]
    keep = _top_p_keep(before, top_p) & (ratio >= min_p)
    keep[0] = True
    n_keep = int(np.argmin(keep)) if not keep.all() else V   # keep is a prefix
    kept = ps[:n_keep]
    c = np.cumsum(kept)
    target = u * c[-1]
    r = int(np.argmax(c > target)) if (c > target).any() else n_keep - 1
    tok = int(order[r])
    if not return_info:
        return tok
    inf = float("inf")
    last = n_keep - 1
    dist = {"top_p_last": abs(before[last] - top_p) if (last > 0 and top_p < 1.0) else inf,
            "min_p_last": abs(ratio[last] - min_p) if last > 0 else inf,
            "first_cut": inf,
            "draw_hi": abs(c[r] / c[-1] - u),
            "draw_lo": abs(c[r - 1] / c[-1] - u) if r > 0 else inf}
    if n_keep < V:
        fails = []
        if top_p < 1.0 and before[n_keep] > top_p:
            fails.append(before[n_keep] - top_p)
        if ratio[n_keep] < min_p:
            fails.append(min_p - ratio[n_keep])
        dist["first_cut"] = float(max(fails))
    dist = {k: float(v) for k, v in dist.items()}
    return tok, dict(n_keep=n_keep, rank=r, dist=dist, margin=min(dist.values()))


def sample_node(logits_row, prior, path_tokens, W, penalty, temperature, top_p,
                min_p, u, return_info=False, literal=False):
    """One tree node's draw: window, penalty, temperature, truncation, draw."""
    win = penalty_window(prior, path_tokens, W)
    xp = penalised_logits(logits_row, win, penalty, temperature, literal)
    return sample_from_logits(xp, top_p, min_p, u, return_info)


def eta_threshold(p, epsilon: float, alpha: float) -> float:
    """η of η-sampling (§D.1: the pool is the tokens with probability at
    least η; η is formed from the entropy, α and ε): η = min(ε, α·exp(-H)),
    H = -sum p log p the entropy in nats of the (penalised, tempered)
    distribution, the truncation-sampling form of the paper the pages cite
    for it (§5.2)."""
    p = np.asarray(p, dtype=np.float64)
    nz = p[p > 0]
    H = float(-(nz * np.log(nz)).sum())
    return min(float(epsilon), float(alpha) * float(np.exp(-H)))


def sample_from_logits_eta(x_pen, epsilon: float, alpha: float, u: float,
                           return_info: bool = False):
    """Draw one token with η-sampling: p = softmax(x') in fp64, ranks by
    (p desc, id asc), the kept set K = {p >= η} (a rank prefix holding rank
    0, as α <= 1 puts η at or below p_max), and the smallest rank in K whose
    cumulative mass exceeds u * mass(K).

    With return_info, the distances of the deciding quantities to their cuts:
      eta_last, eta_first_cut  p/η - 1 of the last kept and first cut rank
                               (relative: η itself is small)
      draw_hi, draw_lo         as in sample_from_logits
    and margin = the smallest."""
    x = np.asarray(x_pen, dtype=np.float64)
    V = x.shape[0]
    e = np.exp(x - x.max())
    p = e / e.sum()
    eta = eta_threshold(p, epsilon, alpha)
    order = np.lexsort((np.arange(V), -p))
    ps = p[order]
    keep = ps >= eta
    keep[0] = True
    n_keep = int(np.argmin(keep)) if not keep.all() else V
    c = np.cumsum(ps[:n_keep])
    target = u * c[-1]
    r = int(np.argmax(c > target)) if (c > target).any() else n_keep - 1
    tok = int(order[r])
    if not return_info:
        return tok
    inf = float("inf")
    last = n_keep - 1
    rel = (lambda v: abs(v / eta - 1.0)) if eta > 0 else (lambda v: inf)
    dist = {"eta_last": rel(ps[last]) if last > 0 else inf,
            "eta_first_cut": rel(ps[n_keep]) if n_keep < V else inf,
            "draw_hi": abs(c[r] / c[-1] - u),
            "draw_lo": abs(c[r - 1] / c[-1] - u) if r > 0 else inf}
    dist = {k: float(v) for k, v in dist.items()}
    return tok, dict(n_keep=n_keep, rank=r, dist=dist, margin=min(dist.values()), eta=eta)


def sample_all_nodes_eta(logits, prior, parents, tree_tokens, W, penalty, temperature,
                         epsilon, alpha, uniforms, return_info=False):
    """Every node's η-sampling draw (window and penalty as sample_node)."""
    paths = root_paths(parents)
    out, infos = [], []
    for i in range(len(parents)):
        drafted = [int(tree_tokens[a]) for a in paths[i][1:]]
        win = penalty_window(prior, drafted, W)
        xp = penalised_logits(logits[i], win, penalty, temperature)
        r = sample_from_logits_eta(xp, epsilon, alpha, float(uniforms[i]), return_info)
        if return_info:
            out.append(r[0])
            infos.append(r[1])
        else:
            out.append(r)
    out = np.asarray(out, dtype=np.int64)
    return (out, infos) if return_info else out


# --------------------------------------------------------------------------
# (a7) exact-match tree acceptance
# --------------------------------------------------------------------------
def accept_from_samples(parents, tree_tokens, sampled):
    """Parallel form: every node has its own target sample.  The root is
    accepted; node c is accepted iff its parent is accepted and its drafted
    token equals the parent's sample (§3.1: exact-match verification).  The
    longest accepted root path wins (deepest node; ties to the smaller node
    index), and the bonus token is the sample at that node.
    Returns (path list, bonus token)."""
    T = len(parents)
    accepted = np.zeros(T, dtype=bool)
    depth = np.zeros(T, dtype=np.int64)
    accepted[0] = True
    for c in range(1, T):
        p = int(parents[c])
        depth[c] = depth[p] + 1
        accepted[c] = accepted[p] and int(tree_tokens[c]) == int(sampled[p])
    best = 0
    for c in range(T):
        if accepted[c] and depth[c] > depth[best]:
            best = c
    path = root_paths(parents)[best]
    return path, int(sampled[best])


def sample_accept_sequential(logits, prior, parents, tree_tokens, W, penalty,
                             temperature, top_p, min_p, uniforms, literal=False):
    """Sequential form of one verification step: starting at the root, sample
    the current node, move to the lowest-index child whose drafted token
    equals that sample, repeat; stop when no child matches.  Only nodes on
    the accepted path are sampled.  Returns (path, bonus token)."""
    T = len(parents)
    children = [[] for _ in range(T)]
    for c in range(1, T):
        children[int(parents[c])].append(c)
    node, path, drafted = 0, [0], []
    while True:
        tok = sample_node(logits[node], prior, drafted, W, penalty, temperature,
                          top_p, min_p, float(uniforms[node]), literal=literal)
        nxt = [c for c in children[node] if int(tree_tokens[c]) == tok]
        if not nxt:
            return path, tok
        node = min(nxt)
        path.append(node)
        drafted.append(int(tree_tokens[node]))


def sample_all_nodes(logits, prior, parents, tree_tokens, W, penalty,
                     temperature, top_p, min_p, uniforms, return_info=False,
                     literal=False):
    """Every node's draw (the parallel form's input).  Node i's window holds
    the drafted tokens on its root path, root excluded."""
    paths = root_paths(parents)
    out, infos = [], []
    for i in range(len(parents)):
        drafted = [int(tree_tokens[a]) for a in paths[i][1:]]
        r = sample_node(logits[i], prior, drafted, W, penalty, temperature,
                        top_p, min_p, float(uniforms[i]), return_info, literal)
        if return_info:
            out.append(r[0])
            infos.append(r[1])
        else:
            out.append(r)
    out = np.asarray(out, dtype=np.int64)
    return (out, infos) if return_info else out


# --------------------------------------------------------------------------
# (NEXT-3) rejection-sampling acceptance (App. A)
# --------------------------------------------------------------------------
def target_distribution(x_pen, top_p: float, min_p: float) -> np.ndarray:
    """The distribution the exact-match path draws from, as a vector: the
    kept set of sample_from_logits (top-p and min-p on p = softmax(x')), its
    probabilities renormalised over the set, zero elsewhere (fp64)."""
    x = np.asarray(x_pen, dtype=np.float64)
    e = np.exp(x - x.max())
    p = e / e.sum()
    order = np.lexsort((np.arange(x.shape[0]), -p))
    ps = p[order]
    before = np.concatenate([[0.0], np.cumsum(ps)[:-1]])
    keep = _top_p_keep(before, top_p) & (ps / ps[0] >= min_p)
    keep[0] = True
    n_keep = int(np.argmin(keep)) if not keep.all() else x.shape[0]
    out = np.zeros_like(p)
    out[order[:n_keep]] = ps[:n_keep]
    return out / out.sum()


def draw_in_id_order(p, u: float) -> int:
    """Inverse-CDF draw over token ids in ascending order: the smallest id
    whose cumulative mass exceeds u * sum(p)."""
    c = np.cumsum(np.asarray(p, dtype=np.float64))
    hit = np.nonzero(c > u * c[-1])[0]
    return int(hit[0]) if hit.size else int(np.nonzero(p)[0][-1])


def accept_rejection(logits, q, prior, parents, tree_tokens, W, penalty, temperature, top_p,
                     min_p, u_accept, u_draw, literal=False):
    """Speculative-sampling acceptance over the draft tree (App. A: acceptance
    and rejection cases together reproduce the target's distribution).

    The pages give the chain argument only; the tree form taken here is
    multi-candidate recursive rejection: from the root, at each accepted node n the children are tried in index
    order as draft candidates drawn from q[n] (the draft distribution that
    proposed n's children, one row per node).  Child c with token x is
    accepted iff u_accept[c] * q[n][x] < p(x), p being n's target
    distribution (penalty window along n's root path, temperature, top-p and
    min-p, as the exact-match path uses); on rejection p becomes
    max(p - q[n], 0) renormalised and the next child is tried.  When no child
    is accepted, the bonus token is drawn from the current p with u_draw[n]
    (inverse CDF in token-id order).  Returns (path, bonus)."""
    T = len(parents)
    children = [[] for _ in range(T)]
    for c in range(1, T):
        children[int(parents[c])].append(c)
    node, path, drafted = 0, [0], []
    while True:
        win = penalty_window(prior, drafted, W)
        p = target_distribution(penalised_logits(logits[node], win, penalty, temperature, literal),
                                top_p, min_p)
        qn = np.asarray(q[node], dtype=np.float64)
        nxt = None
        for c in children[node]:
            x = int(tree_tokens[c])
            if float(u_accept[c]) * qn[x] < p[x]:
                nxt = c
                break
            r = np.maximum(p - qn, 0.0)
            if r.sum() > 0.0:   # r == 0 only if p == q, where a rejection leaves p as it is
                p = r / r.sum()
        if nxt is None:
            return path, draw_in_id_order(p, float(u_draw[node]))
        node = nxt
        path.append(node)
        drafted.append(int(tree_tokens[node]))


# --------------------------------------------------------------------------
# (a8) KV commit of the accepted path
# --------------------------------------------------------------------------
def kv_append(cache, L: int, rows) -> np.ndarray:
    """The tree tokens' own K (or V) rows written by the verification forward
    (§3.1): rows [L, L+T) of every head take rows[h, 0:T].  cache
    [Hkv, L_cap, d]; rows [Hkv, T, d]; returns the updated copy."""
    out = np.array(cache, copy=True)
    rows = np.asarray(rows)
    out[:, L:L + rows.shape[1]] = rows
    return out


def kv_commit(cache, L: int, path) -> np.ndarray:
    """After acceptance the cache update (§3.1) keeps the accepted tree rows:
    row L+path[t] moves to row L+t for t = 1..len(path)-1 (the root's row is
    already at L).  cache: [Hkv, L_cap, d]; returns the updated copy."""
    out = np.array(cache, copy=True)
    for t in range(1, len(path)):
        out[:, L + t] = cache[:, L + path[t]]
    return out


# --------------------------------------------------------------------------
# (NEXT-2) token reutilization: the 4-gram table and the draft-tree builder
# --------------------------------------------------------------------------
# §3.1 Overview: after verification the n-gram table is updated; §3.2 and
# §3.4: frequent n-grams supply extra draft candidates, with random selection
# among several valid ones; §B.2 Inference Details / Table 10: 4-grams, at
# most k retrieved n-grams (k = 20, Table 11); §4.4.1 / §B.2: the extra heads'
# candidates form the ternary full tree [1,3,3,3].
#
# Readings (the pages give no data structure): a 4-gram (a, b, c, d) is
# stored under its first token a as the continuation (b, c, d); each key keeps
# its distinct continuations, at most `cap` of them, oldest dropped first, a
# repeated continuation neither duplicated nor moved.  Retrieval for the root
# token returns every stored continuation (oldest first) when there are at
# most k, else the k whose caller-supplied random keys are smallest (ties to
# the lower slot), in that order.  The tree is the root, then the head tree in
# breadth-first order (depth-d nodes carry head d's candidates), then each
# retrieved continuation merged as a path from the root: an existing child
# with the same token is followed, else a node is appended while fewer than
# T_max nodes exist.


def ngram_insert(table: dict, tokens, start: int, cap: int) -> dict:
    """Insert the 4-grams ending at positions start .. len(tokens)-1 (those
    with a full 4-gram, p >= 3) into `table` (key -> list of continuations,
    oldest first), in position order.  Returns the table."""
    toks = [int(t) for t in tokens]
    for p in range(max(start, 3), len(toks)):
        key = toks[p - 3]
        cont = (toks[p - 2], toks[p - 1], toks[p])
        lst = table.setdefault(key, [])
        if cont in lst:
            continue
        lst.append(cont)
        if len(lst) > cap:
            lst.pop(0)
    return table


def ngram_retrieve(table: dict, root: int, k: int, rand_keys) -> list:
    """Continuations stored under `root`: all of them (oldest first) if there
    are at most k, else the k with the smallest (rand_keys[slot], slot), where
    slot is the entry's position oldest-first, in increasing key order."""
    lst = table.get(int(root), [])
    if len(lst) <= k:
        return list(lst)
    order = sorted(range(len(lst)), key=lambda s: (int(rand_keys[s]), s))
    return [lst[s] for s in order[:k]]


def build_draft_tree(root_token: int, head_topk, chains, T_max: int):
    """Draft tree of the root, the extra heads' ternary tree and the retrieved
    chains, as (parents, tokens) int32 arrays of n <= T_max nodes with
    parents[i] < i.  head_topk[d][c]: candidate c of head d+1."""
    parents, tokens = [-1], [int(root_token)]
    children = [[]]

    def add(p, tok):
        parents.append(p)
        tokens.append(int(tok))
        children.append([])
        children[p].append(len(parents) - 1)
        return len(parents) - 1

    level = [0]
    for d in range(len(head_topk)):
        nxt = []
        for p in level:
            for tok in head_topk[d]:
                if len(parents) >= T_max:
                    break
                nxt.append(add(p, tok))
        level = nxt
    for chain in chains:
        cur = 0
        for tok in chain:
            hit = next((c for c in children[cur] if tokens[c] == int(tok)), None)
            if hit is None:
                if len(parents) >= T_max:
                    break
                hit = add(cur, tok)
            cur = hit
    return np.asarray(parents, dtype=np.int32), np.asarray(tokens, dtype=np.int32)
