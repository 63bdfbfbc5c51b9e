"""Pins for the oracle's mixture-of-experts feed-forward (CPU).

The pages name a mixture-of-experts target (Qwen3-Coder-30B-A3B) but print no layer
equations; the layer is read as the Qwen3-MoE one (router softmax, top-k experts with
renormalised weights, SwiGLU experts).  Pinned here by: the reduction to the dense layer
with one expert, brute force over all expert subsets for the routing (with planted ties),
invariance under relabelling the experts, a formulation with torch library routines, and
tree rows equal to sequential decoding along their root paths.
"""
import dataclasses
import itertools

import numpy as np
import pytest

import synth
from oracle import ddtree, model, step

SHAPE = synth.ModelShape(2, 64, 4, 2, 16, 0, 97, feat_layers=(1, 2), n_experts=6, top_k=2, d_expert=40)


def _rows(seed, n, d):
    return synth.normal(seed, "moe.h", (n, d)).astype(np.float64)


def test_single_expert_reduces_to_dense_layer():
    shape = dataclasses.replace(SHAPE, n_experts=1, top_k=1)
    lw = synth.layer_weights(shape, 5, "moe1")
    dense = dataclasses.replace(lw, w_gate_up=lw.w_experts_gate_up[0], w_down=lw.w_experts_down[0])
    h = _rows(5, 7, shape.d_model)
    dense_shape = dataclasses.replace(shape, d_ff=shape.d_expert, n_experts=0, top_k=0)
    np.testing.assert_array_equal(model.moe_block(lw, shape, h), model.mlp_block(dense, dense_shape, h))


@pytest.mark.parametrize("k", [1, 2, 3])
def test_routing_equals_best_subset_by_brute_force(k):
    shape = dataclasses.replace(SHAPE, top_k=k)
    lw = synth.layer_weights(shape, 6, "moer")
    # planted exact ties: experts 1 and 4 share router weights, as do 2 and 5
    lw.w_router[4] = lw.w_router[1]
    lw.w_router[5] = lw.w_router[2]
    x = _rows(6, 40, shape.d_model)
    ids, w, logits = model.moe_route(lw, shape, x)
    p = np.exp(logits - logits.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    for i in range(len(x)):
        best, best_set = None, None
        for sub in itertools.combinations(range(shape.n_experts), k):  # lexicographic order
            v = sum(p[i, e] for e in sub)
            if best is None or v > best + 1e-15:
                best, best_set = v, sub
        assert tuple(sorted(ids[i])) == best_set, (i, ids[i], best_set)
        # listed by probability, lower id first among equals; weights renormalised
        assert all(p[i, ids[i][j]] >= p[i, ids[i][j + 1]] for j in range(k - 1))
        np.testing.assert_allclose(w[i].sum(), 1.0, rtol=0, atol=1e-15)
        np.testing.assert_allclose(w[i] / w[i][0], p[i, ids[i]] / p[i, ids[i][0]], rtol=1e-13)


def test_expert_relabelling_invariance():
    lw = synth.layer_weights(SHAPE, 7, "moep")
    perm = np.array([3, 0, 5, 1, 4, 2])
    lp = dataclasses.replace(lw, w_router=lw.w_router[perm], w_experts_gate_up=lw.w_experts_gate_up[perm],
                             w_experts_down=lw.w_experts_down[perm])
    h = _rows(7, 9, SHAPE.d_model)
    np.testing.assert_allclose(model.moe_block(lp, SHAPE, h), model.moe_block(lw, SHAPE, h), rtol=1e-13, atol=1e-15)


def test_moe_block_matches_torch_library_formulation():
    import torch
    import torch.nn.functional as F
    lw = synth.layer_weights(SHAPE, 8, "moet")
    h = _rows(8, 11, SHAPE.d_model)
    T = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    x = F.rms_norm(T(h), (SHAPE.d_model,), T(lw.mlp_norm), eps=SHAPE.rms_eps)
    probs = F.softmax(x @ T(lw.w_router).T, dim=-1)
    topv, topi = torch.topk(probs, SHAPE.top_k, dim=-1)
    wt = topv / topv.sum(-1, keepdim=True)
    Fe = SHAPE.d_expert
    gu = torch.einsum("nkfd,nd->nkf", T(lw.w_experts_gate_up)[topi], x)
    act = F.silu(gu[..., :Fe]) * gu[..., Fe:]
    out = torch.einsum("nkdf,nkf->nkd", T(lw.w_experts_down)[topi], act)
    ref = T(h) + (wt[..., None] * out).sum(1)
    np.testing.assert_allclose(model.moe_block(lw, SHAPE, h), ref.numpy(), rtol=1e-10, atol=1e-12)


def test_moe_target_tree_rows_equal_sequential_decode():
    tw = synth.target_weights(SHAPE, 9)
    lp = ddtree.log_softmax(np.random.default_rng(9).normal(0, 2, size=(3, SHAPE.vocab)))
    tree = ddtree.build_tree(lp, 6)
    tok = tree["tok"].copy()
    tok[0] = 5
    N, cap = 4, 32
    prompt = synth.uniform_ints(9, "moe.prompt", (N,), 0, SHAPE.vocab)
    base = step.KVCache.empty(SHAPE, cap)
    step.target_tree_forward(tw, prompt, np.arange(-1, N - 1), np.arange(N), base, 0)
    cache = step.KVCache([k.copy() for k in base.k], [v.copy() for v in base.v])
    _, feats, logits = step.target_tree_forward(tw, tok, tree["parent"], tree["depth"], cache, N)
    for i in range(len(tok)):
        path = []
        j = i
        while j >= 0:
            path.append(j)
            j = int(tree["parent"][j])
        path = path[::-1]
        c = step.KVCache([k.copy() for k in base.k], [v.copy() for v in base.v])
        _, f2, l2 = step.target_tree_forward(tw, tok[path], np.arange(-1, len(path) - 1), np.arange(len(path)), c, N)
        np.testing.assert_allclose(feats[i], f2[-1], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(logits[i], l2[-1], rtol=1e-11, atol=1e-12)
