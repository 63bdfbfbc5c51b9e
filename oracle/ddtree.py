"""DDTree: optimal draft tree under a node budget, from factorized per-position distributions.

[DDTree] section "핵심 아이디어": the drafter emits one distribution per future
position in a single pass, and the tree builder treats the positions as independent
(a factorized distribution).
[DDTree] section "방법론 자세히 보기": the expected acceptance length equals the sum
of the prefix probabilities of the tree's nodes, so the best tree under a budget of B
nodes is the set of the B most probable prefixes; a best-first max-heap finds them in
O(B log B).

Readings (the pages give no more detail):
  * log-probabilities are float32; a prefix score is the float32 sum of its
    positions' log-probs, added root first.
  * total order on prefixes: score descending, then depth ascending, then the
    parent's place in this same order, then the rank of the last token in its
    position's sorted list.  Both the heap and the brute force below use it.
  * per-position candidates are sorted by (log-prob descending, token id ascending);
    only the first K = min(B, V) can enter a B-node tree.
  * successor rule of the best-first search: popping prefix (..., r) proposes its
    first child (..., r, 1) and its next sibling (..., r + 1).
"""
from __future__ import annotations

import functools
import heapq
import itertools

import numpy as np


class TreeError(ValueError):
    pass


def log_softmax(logits) -> np.ndarray:
    """Per-row log-softmax in float64, returned as float32."""
    x = np.asarray(logits, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True))
    return (x - lse).astype(np.float32)


def topk_sorted(lp_row: np.ndarray, K: int):
    """The K best (log-prob desc, token id asc) entries of one position."""
    lp_row = np.asarray(lp_row, dtype=np.float32)
    if np.isnan(lp_row).any():
        raise TreeError("NaN log-probability")
    ids = np.arange(lp_row.shape[0])
    order = np.lexsort((ids, -lp_row.astype(np.float64)))[:K]
    return order.astype(np.int32), lp_row[order]


def n_prefixes(V: int, D: int) -> int:
    return sum(V ** k for k in range(1, D + 1))


def build_tree(lp: np.ndarray, B: int):
    """Best-first max-heap selection of the top-B prefixes.

    lp: float32 [D, V] log-probabilities of draft positions 1..D.
    Returns dict of arrays of length B+1 (index 0 = root, i.e. the bonus token):
      tok (root: -1), parent (root: -1), depth (root: 0), score (float32, root 0),
      rank (0-based rank of the node's token at its depth; root: -1).
    Node indices are the pop order, so every parent precedes its children.
    """
    lp = np.asarray(lp, dtype=np.float32)
    D, V = lp.shape
    if B < 0 or B > n_prefixes(V, D):
        raise TreeError("budget exceeds the number of prefixes")
    K = min(B, V)
    ids, vals = [], []
    for d in range(D):
        i, v = topk_sorted(lp[d], max(K, 1))
        ids.append(i)
        vals.append(v)

    tok = [-1]
    parent = [-1]
    depth = [0]
    score = [np.float32(0.0)]
    rank = [-1]
    heap = []

    def push(s, dep, par, r):
        # heapq is a min-heap: negate the score; depth, parent index and rank ascend.
        heapq.heappush(heap, (-float(s), dep, par, r, s))

    if B > 0:
        push(np.float32(score[0] + vals[0][0]), 1, 0, 0)
    while len(tok) <= B:
        _, dep, par, r, s = heapq.heappop(heap)
        idx = len(tok)
        tok.append(int(ids[dep - 1][r]))
        parent.append(par)
        depth.append(dep)
        score.append(s)
        rank.append(r)
        if dep < D:
            push(np.float32(s + vals[dep][0]), dep + 1, idx, 0)
        if r + 1 < K:
            push(np.float32(score[par] + vals[dep - 1][r + 1]), dep, par, r + 1)
    return dict(tok=np.array(tok, np.int32), parent=np.array(parent, np.int32),
                depth=np.array(depth, np.int32), score=np.array(score, np.float32),
                rank=np.array(rank, np.int32))


def build_chain(lp: np.ndarray):
    """Vanilla DFlash draft: the most likely token at every position, as one chain.

    [DDTree] section "실험 결과": DDTree is measured against plain DFlash at the same block
    size, which verifies the drafter's block as it stands, one token per position.
    [DFlash] section "DFlash의 핵심 아이디어" (3): one drafter pass fills the block.
    Readings: the most likely token is the lowest id among exactly equal log-probs (the
    same rule as the greedy target); the chain uses the tree's arrays (root = index 0,
    node i at depth i with parent i - 1, fp32 score summed root first).
    """
    lp = np.asarray(lp, dtype=np.float32)
    if np.isnan(lp).any():
        raise TreeError("NaN log-probability")
    D, V = lp.shape
    tok, parent, depth, score = [-1], [-1], [0], [np.float32(0.0)]
    for d in range(D):
        i = int(np.argmax(lp[d]))  # first occurrence of the maximum = lowest id
        tok.append(i)
        parent.append(d)
        depth.append(d + 1)
        score.append(np.float32(score[-1] + lp[d, i]))
    return dict(tok=np.array(tok, np.int32), parent=np.array(parent, np.int32),
                depth=np.array(depth, np.int32), score=np.array(score, np.float32))


def ancestor_mask(parent: np.ndarray) -> np.ndarray:
    """Bit j of row i is set iff node j is node i or one of its ancestors.

    [DDTree] section "방법론 자세히 보기": each flattened tree token may attend only to
    tokens on its own ancestor path.  Packed as uint32 words, little-endian bits.
    """
    n = len(parent)
    words = (n + 31) // 32
    out = np.zeros((n, words), dtype=np.uint32)
    for i in range(n):
        j = i
        while j >= 0:
            out[i, j // 32] |= np.uint32(1 << (j % 32))
            j = int(parent[j])
    return out


def expected_acceptance(score: np.ndarray) -> float:
    """Sum of the non-root nodes' prefix probabilities (expected accepted drafted tokens)."""
    return float(np.sum(np.exp(np.asarray(score[1:], dtype=np.float64))))


# ----------------------------------------------------------------------------- brute force
def _sorted_lists(lp):
    out = []
    for d in range(lp.shape[0]):
        # stable sort of negated log-probs keeps ids ascending among equal values
        order = np.argsort(-lp[d].astype(np.float64), kind="stable")
        out.append((order.astype(np.int32), lp[d][order]))
    return out


def brute_force_tree(lp: np.ndarray, B: int):
    """Enumerate every prefix, sort by the total order, keep the first B (tiny V, D only)."""
    lp = np.asarray(lp, dtype=np.float32)
    D, V = lp.shape
    lists = _sorted_lists(lp)
    scores = {}
    prefixes = []
    for k in range(1, D + 1):
        for ranks in itertools.product(range(V), repeat=k):
            parent_s = scores[ranks[:-1]] if k > 1 else np.float32(0.0)
            scores[ranks] = np.float32(parent_s + lists[k - 1][1][ranks[-1]])
            prefixes.append(ranks)

    def cmp(p, q):
        sp, sq = scores[p], scores[q]
        if sp != sq:
            return -1 if sp > sq else 1
        if len(p) != len(q):
            return -1 if len(p) < len(q) else 1
        if len(p) > 1 and p[:-1] != q[:-1]:
            return cmp(p[:-1], q[:-1])
        return (p[-1] > q[-1]) - (p[-1] < q[-1])

    chosen = sorted(prefixes, key=functools.cmp_to_key(cmp))[:B]
    index = {(): 0}
    tok, parent, depth, score, rank = [-1], [-1], [0], [np.float32(0)], [-1]
    for p in chosen:
        index[p] = len(tok)
        tok.append(int(lists[len(p) - 1][0][p[-1]]))
        parent.append(index[p[:-1]])
        depth.append(len(p))
        score.append(scores[p])
        rank.append(p[-1])
    return dict(tok=np.array(tok, np.int32), parent=np.array(parent, np.int32),
                depth=np.array(depth, np.int32), score=np.array(score, np.float32),
                rank=np.array(rank, np.int32))


def best_closed_subset_value(lp: np.ndarray, B: int) -> float:
    """Max over all prefix-closed sets of exactly B prefixes of the sum of prefix probabilities.

    Exhaustive search over token prefixes (not ranks), for tiny V and D only.
    """
    lp = np.asarray(lp, dtype=np.float64)
    D, V = lp.shape
    best = -np.inf

    def rec(frontier, chosen_val, count):
        nonlocal best
        if count == B:
            best = max(best, chosen_val)
            return
        # choose the next prefix from the frontier in canonical (index) order to avoid repeats
        for i, (pref, s) in enumerate(frontier):
            rest = frontier[i + 1:]
            kids = []
            if len(pref) < D:
                kids = [(pref + (v,), s + lp[len(pref), v]) for v in range(V)]
            rec(rest + kids, chosen_val + np.exp(s), count + 1)

    rec([((v,), lp[0, v]) for v in range(V)], 0.0, 0)
    return float(best)
