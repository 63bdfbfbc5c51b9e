"""Pins for the oracle's DDTree builder, log-softmax and top-K (CPU only).

Each check ties the oracle to something other than itself: brute-force enumeration of
every prefix, an exhaustive search over prefix-closed trees, Monte-Carlo sampling of the
factorized distribution, a library sort, or a closed form.
"""
import heapq
import itertools

import numpy as np
import pytest
import scipy.special

from oracle import ddtree
import synth


def _rand_lp(seed, D, V, ties=False, neginf=False):
    g = np.random.default_rng(seed)
    x = g.normal(0, 2.0, size=(D, V))
    if ties:
        x = np.round(x)  # many equal logits -> equal log-probs within a row
    lp = ddtree.log_softmax(x)
    if neginf:
        lp[g.random(lp.shape) < 0.2] = -np.inf
    return lp


def _same_tree(a, b):
    for k in ("tok", "parent", "depth", "rank"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(a["score"].view(np.uint32), b["score"].view(np.uint32))


@pytest.mark.parametrize("V,D", [(2, 1), (2, 4), (3, 3), (4, 2), (5, 3), (6, 2)])
@pytest.mark.parametrize("mode", ["plain", "ties", "neginf"])
def test_heap_equals_brute_force(V, D, mode):
    total = ddtree.n_prefixes(V, D)
    for seed in range(4):
        lp = _rand_lp(100 * V + 10 * D + seed, D, V, ties=(mode == "ties"), neginf=(mode == "neginf"))
        for B in sorted({b for b in (0, 1, 2, 3, 7, 16) if b <= total} | {total}):
            _same_tree(ddtree.build_tree(lp, B), ddtree.brute_force_tree(lp, B))


def test_heap_equals_brute_force_sum_ties():
    # log-probs on a coarse dyadic grid so that different prefixes reach equal float32 sums
    for seed in range(6):
        g = np.random.default_rng(seed)
        lp = (-g.integers(0, 4, size=(3, 4)) * 0.5).astype(np.float32)
        for B in (5, 11, 30, ddtree.n_prefixes(4, 3)):
            _same_tree(ddtree.build_tree(lp, B), ddtree.brute_force_tree(lp, B))


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 6])
def test_top_b_is_optimal_over_prefix_closed_trees(B):
    for seed in range(3):
        lp = _rand_lp(7 + seed, 3, 3)
        tree = ddtree.build_tree(lp, B)
        best = ddtree.best_closed_subset_value(lp, B)
        assert ddtree.expected_acceptance(tree["score"]) == pytest.approx(best, rel=1e-6)


def test_expected_acceptance_matches_monte_carlo():
    # E[accepted drafted tokens] = sum of prefix probabilities (DDTree page, method section)
    D, V, B = 3, 5, 12
    lp = _rand_lp(42, D, V)
    tree = ddtree.build_tree(lp, B)
    n = 1_000_000
    g = np.random.default_rng(123)
    p = np.exp(lp.astype(np.float64))
    p /= p.sum(axis=1, keepdims=True)
    draws = np.stack([g.choice(V, size=n, p=p[d]) for d in range(D)], axis=1)
    child = -np.ones((B + 1, V), dtype=np.int64)
    for i in range(1, B + 1):
        child[tree["parent"][i], tree["tok"][i]] = i
    cur = np.zeros(n, dtype=np.int64)
    acc = np.zeros(n, dtype=np.int64)
    alive = np.ones(n, dtype=bool)
    for d in range(D):
        nxt = child[cur, draws[:, d]]
        alive &= nxt >= 0
        acc += alive
        cur = np.where(alive, nxt, 0)
    mean, sd = acc.mean(), acc.std()
    expect = ddtree.expected_acceptance(tree["score"])
    assert abs(mean - expect) < 4 * sd / np.sqrt(n) + 1e-6


def test_topk_matches_heapq():
    g = np.random.default_rng(5)
    row = np.round(g.normal(size=2000), 1).astype(np.float32)  # heavy ties
    for K in (1, 7, 64, 500, 2000):
        ids, vals = ddtree.topk_sorted(row, K)
        ref = heapq.nlargest(K, range(len(row)), key=lambda i: (float(row[i]), -i))
        np.testing.assert_array_equal(ids, ref)
        np.testing.assert_array_equal(vals, row[ref])


def test_log_softmax_closed_forms():
    x = np.random.default_rng(1).normal(0, 3, size=(4, 1000))
    lp = ddtree.log_softmax(x)
    np.testing.assert_allclose(np.exp(lp.astype(np.float64)).sum(-1), 1.0, atol=1e-5)
    np.testing.assert_array_equal(ddtree.log_softmax(x + 123.0), lp)
    np.testing.assert_allclose(lp, scipy.special.log_softmax(x, axis=-1), atol=2e-6, rtol=1e-6)


def test_ancestor_mask_special_cases():
    chain = np.array([-1, 0, 1, 2, 3])
    m = ddtree.ancestor_mask(chain)
    dense = np.array([[(m[i, j // 32] >> (j % 32)) & 1 for j in range(5)] for i in range(5)])
    np.testing.assert_array_equal(dense, np.tril(np.ones((5, 5), dtype=int)))
    star = np.array([-1] + [0] * 40)
    m = ddtree.ancestor_mask(star)
    assert m.shape == (41, 2)
    for i in range(41):
        bits = {j for j in range(41) if (m[i, j // 32] >> (j % 32)) & 1}
        assert bits == ({0, i} if i else {0})


def test_chain_special_case():
    # one dominant token per position and B = D: the tree is the argmax chain (vanilla DFlash)
    D, V = 6, 50
    g = np.random.default_rng(9)
    x = g.normal(0, 1, size=(D, V))
    hot = g.integers(0, V, size=D)
    x[np.arange(D), hot] += 30.0
    tree = ddtree.build_tree(ddtree.log_softmax(x), D)
    np.testing.assert_array_equal(tree["tok"][1:], hot)
    np.testing.assert_array_equal(tree["parent"], np.arange(-1, D))
    np.testing.assert_array_equal(tree["depth"], np.arange(D + 1))


def test_budget_and_nan_errors():
    lp = _rand_lp(0, 2, 3)
    with pytest.raises(ddtree.TreeError):
        ddtree.build_tree(lp, ddtree.n_prefixes(3, 2) + 1)
    lp[1, 2] = np.nan
    with pytest.raises(ddtree.TreeError):
        ddtree.build_tree(lp, 4)


def test_parents_precede_children_at_config_scale():
    lp = ddtree.log_softmax(synth.ddtree_logits(1002, 1, 15, 151936)[0])
    t = ddtree.build_tree(lp, 256)
    assert np.all(t["parent"][1:] < np.arange(1, 257))
    assert np.all(t["depth"][1:] == t["depth"][t["parent"][1:]] + 1)
    s = t["score"][1:].astype(np.float64)
    assert np.all(np.diff(s) <= 0)  # pop order is by score


@pytest.mark.parametrize("V,D", [(2, 4), (3, 3), (5, 2), (4, 4)])
@pytest.mark.parametrize("mode", ["plain", "ties", "neginf"])
def test_chain_is_best_sequence_by_exhaustive_search(V, D, mode):
    # the DFlash chain: over all V^D token sequences, the one whose fp32 root-first sum is
    # largest, and among those the lexicographically lowest ids
    g = np.random.default_rng(V * 10 + D)
    x = g.normal(0, 2, size=(D, V))
    if mode == "ties":
        x = np.round(x)
    lp = ddtree.log_softmax(x)
    if mode == "neginf":
        lp[g.random(lp.shape) < 0.3] = -np.inf
    best, best_seq = None, None
    for seq in itertools.product(range(V), repeat=D):   # lexicographic order
        s = np.float32(0.0)
        for d, t in enumerate(seq):
            s = np.float32(s + lp[d, t])
        if best is None or s > best:
            best, best_seq = s, seq
    c = ddtree.build_chain(lp)
    np.testing.assert_array_equal(c["tok"][1:], best_seq)
    assert c["score"][-1].view(np.uint32) == np.float32(best).view(np.uint32)
    np.testing.assert_array_equal(c["parent"], np.arange(-1, D))
    np.testing.assert_array_equal(c["depth"], np.arange(D + 1))
    # every prefix score is the fp32 running sum, root first
    run = np.float32(0.0)
    for d in range(D):
        run = np.float32(run + lp[d, c["tok"][d + 1]])
        assert c["score"][d + 1].view(np.uint32) == run.view(np.uint32)


def test_chain_equals_tree_of_budget_d_with_dominant_tokens():
    D, V = 7, 300
    g = np.random.default_rng(21)
    x = g.normal(0, 1, size=(D, V))
    x[np.arange(D), g.integers(0, V, size=D)] += 25.0
    lp = ddtree.log_softmax(x)
    c, t = ddtree.build_chain(lp), ddtree.build_tree(lp, D)
    for k in ("tok", "parent", "depth"):
        np.testing.assert_array_equal(c[k], t[k])
    np.testing.assert_array_equal(c["score"].view(np.uint32), t["score"].view(np.uint32))


def test_chain_nan_rejected():
    lp = _rand_lp(1, 3, 5)
    lp[2, 1] = np.nan
    with pytest.raises(ddtree.TreeError):
        ddtree.build_chain(lp)
