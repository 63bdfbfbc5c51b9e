"""Tree verification: ancestor-only attention, greedy longest-path acceptance, KV compaction.

[DDTree] section "핵심 아이디어" and "방법론 자세히 보기": the tree is flattened and
fed to the target in one forward pass under an ancestor-only attention mask; the
verifier walks the tree along the target's own outputs, accepts the longest path that
matches, and compacts the KV cache so that rejected branches are dropped.

Readings:
  * tree node i (index 0 = root = bonus token) is written to cache slot N + i and
    rotated at position N + depth(i); after acceptance, the node at depth j is moved
    to slot N + j, whose position is then equal to its slot.
  * the target's greedy choice is the lowest token id among equal maxima.
  * the accepted count a excludes the root; the step commits a drafted tokens plus
    one new bonus token (the target's choice after the last accepted node).
"""
from __future__ import annotations

import numpy as np

from . import model


def ancestors(parent, i):
    """Ancestor-or-self indices of node i in increasing order (root first)."""
    out = []
    while i >= 0:
        out.append(i)
        i = int(parent[i])
    return out[::-1]


def tree_attention(shape, q, k_cache, v_cache, N, parent):
    """Ancestor-only attention for every tree row.

    q: [T, Hq, hd]; k_cache, v_cache: [cap, Hkv, hd] with tree node j at slot N + j.
    Row i sees cache slots [0, N) and tree slots N + j for j ancestor-or-self of i,
    in increasing slot order.  Returns [T, Hq*hd].
    """
    def keys(i):
        idx = list(range(N)) + [N + j for j in ancestors(parent, i)]
        return k_cache[idx], v_cache[idx]
    return model.attention_rows(shape, q, keys)


def greedy_walk(target_choice, tok, parent):
    """Longest path from the root whose every edge token equals the target's choice at its parent.

    Returns (path node indices in depth order, new bonus token).  Children of one node
    carry distinct tokens, so at most one child can match.
    """
    T = len(tok)
    cur, path = 0, []
    while True:
        want = int(target_choice[cur])
        nxt = [c for c in range(1, T) if int(parent[c]) == cur and int(tok[c]) == want]
        if not nxt:
            break
        cur = nxt[0]
        path.append(cur)
    return path, int(target_choice[cur])


def compact(cache, N, path):
    """Move accepted nodes' K/V to consecutive slots: new[N + j] = old[N + path[j-1]].

    cache: array [..., cap, ...] indexed by slot on axis 0 (a copy is taken first, so the
    definition holds whatever the overlap between sources and destinations).
    """
    old = cache.copy()
    for j, idx in enumerate(path, start=1):
        cache[N + j] = old[N + idx]
    return N + 1 + len(path)
