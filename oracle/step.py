"""One speculative step and the two generation loops (speculative and plain greedy), one sequence.

[DFlash] section "왜 기존 speculative decoding도 한계가 있었나": a drafter proposes,
the target checks the proposal in one pass, accepted tokens are kept and generation
resumes from the first mismatch.
[DFlash] section "DFlash의 핵심 아이디어" (3): the drafter fills every masked position
of a short block in one forward pass.
[DDTree] section "핵심 아이디어": the drafter input is the masked block after the bonus
token; its per-position distributions drive the tree (see ddtree.py), which the target
verifies in one pass (see verify.py).

Readings:
  * block of L rows: row 0 is the bonus token, rows 1..L-1 the mask token; the drafter's
    rows 1..L-1 give D = L-1 draft depths.
  * context fusion: c = RMSNorm(W_fc . concat(hidden states of the feature layers));
    in every drafter layer, c is projected by that layer's own W_k / W_v (then k-norm and
    rotation at the context position) and appended to that layer's context K/V, which
    the block rows attend to together with the block's own keys, with no mask.
  * the target's feature rows are the residual outputs of the listed (1-indexed) layers.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import ddtree, model, verify


@dataclass
class KVCache:
    """Per layer K and V, [cap, Hkv, hd] float64, indexed by slot."""
    k: list
    v: list

    @staticmethod
    def empty(shape, cap):
        z = lambda: np.zeros((cap, shape.n_kv_heads, shape.head_dim))
        return KVCache([z() for _ in range(shape.n_layers)], [z() for _ in range(shape.n_layers)])


def target_tree_forward(tw, tok, parent, depth, cache: KVCache, N, choose=None):
    """Target forward over a flattened tree (or one token, or a chain).

    Writes node i's K/V to slot N + i of every layer, attends ancestor-only, and returns
    (choice per node, feature rows [T, n_feat*d], logits [T, V]).  The choice is the greedy
    one (argmax, lowest id on ties), or choose(logits, positions) with the absolute
    position N + depth + 1 of the token each node predicts (sampling, see sample.py).
    """
    shape = tw.shape
    tok = np.asarray(tok)
    T = len(tok)
    pos = N + np.asarray(depth)
    h = np.asarray(tw.embed, np.float64)[tok]
    feats = []
    for li, layer in enumerate(tw.layers):
        x = model.rms_norm(h, layer.attn_norm, shape.rms_eps)
        q, k, v = model.qkv_rows(layer, shape, x)
        q, k = model.qk_finish(layer, shape, q, k, pos)
        cache.k[li][N:N + T] = k
        cache.v[li][N:N + T] = v
        o = verify.tree_attention(shape, q, cache.k[li], cache.v[li], N, parent)
        h = h + model.linear(o, layer.w_o)
        h = model.ffn_block(layer, shape, h)
        if li + 1 in shape.feat_layers:
            feats.append(h.copy())
    logits = model.lm_head(tw, h)
    choice = model.argmax_lowest(logits) if choose is None else choose(logits, pos + 1)
    return choice, np.concatenate(feats, axis=-1), logits


def fuse_context(dw, feat):
    """c = RMSNorm(W_fc f) for each new context row f (concatenated target hidden states)."""
    return model.rms_norm(model.linear(feat, dw.fc), dw.fc_norm, dw.shape.rms_eps)


def draft_block(dw, feat, ctx: KVCache, ctx_len, bonus):
    """One drafter forward: append the new context rows, then fill the block in one pass.

    feat: [n_new, n_feat*d] target features of the newly committed positions
    (positions ctx_len .. ctx_len+n_new-1).  Returns (log-probs float32 [D, V],
    new ctx_len, drafter logits [D, V]).
    """
    shape = dw.shape
    L = shape.block_size
    n_new = feat.shape[0]
    if n_new:
        c = fuse_context(dw, feat)
        pos_c = ctx_len + np.arange(n_new)
        for li, layer in enumerate(dw.layers):
            _, kc, vc = model.qkv_rows(layer, shape, c)
            kc = model.rope(model.rms_norm(kc, layer.k_norm, shape.rms_eps), pos_c[:, None], shape.rope_theta)
            ctx.k[li][ctx_len:ctx_len + n_new] = kc
            ctx.v[li][ctx_len:ctx_len + n_new] = vc
    ctx_len += n_new
    block = np.array([bonus] + [shape.mask_token] * (L - 1))
    pos = ctx_len + np.arange(L)
    h = np.asarray(dw.embed, np.float64)[block]
    for li, layer in enumerate(dw.layers):
        x = model.rms_norm(h, layer.attn_norm, shape.rms_eps)
        q, k, v = model.qkv_rows(layer, shape, x)
        q, k = model.qk_finish(layer, shape, q, k, pos)
        K = np.concatenate([ctx.k[li][:ctx_len], k])
        V = np.concatenate([ctx.v[li][:ctx_len], v])
        o = model.attention_rows(shape, q, lambda i: (K, V))
        h = h + model.linear(o, layer.w_o)
        h = model.mlp_block(layer, shape, h)
    logits = model.lm_head(dw, h[1:])
    return ddtree.log_softmax(logits), ctx_len, logits


@dataclass
class SeqState:
    cache: KVCache
    N: int
    ctx: KVCache
    ctx_len: int
    bonus: int
    feat: np.ndarray            # pending feature rows for the drafter's context
    out: list = field(default_factory=list)


def prefill(tw, dw, prompt, cap, choose=None):
    """Causal prompt pass, one token at a time; yields the first bonus token and the features."""
    cache = KVCache.empty(tw.shape, cap)
    feats = []
    choice = None
    for i, t in enumerate(prompt):
        ch, f, _ = target_tree_forward(tw, [t], [-1], [0], cache, i, choose)
        feats.append(f[0])
        choice = int(ch[0])
    ctx = KVCache.empty(dw.shape, cap) if dw is not None else None
    return SeqState(cache, len(prompt), ctx, 0, choice, np.array(feats), [choice])


def spec_step(tw, dw, st: SeqState, B, plant=None, choose=None):
    """Draft -> DDTree -> verify -> accept -> compact.  Returns (tree, path).

    plant(st, logits) -> logits may bias the drafter's logits before the log-softmax
    (test harness only: random-init drafters rarely agree with random-init targets).
    choose: the target's choice per node (greedy when None; see target_tree_forward).
    """
    lp, st.ctx_len, logits = draft_block(dw, st.feat, st.ctx, st.ctx_len, st.bonus)
    if plant is not None:
        lp = ddtree.log_softmax(plant(st, logits))
    tree = ddtree.build_tree(lp, B)
    tok = tree["tok"].copy()
    tok[0] = st.bonus
    choice, feats, _ = target_tree_forward(tw, tok, tree["parent"], tree["depth"], st.cache, st.N, choose)
    path, new_bonus = verify.greedy_walk(choice, tok, tree["parent"])
    for li in range(tw.shape.n_layers):
        verify.compact(st.cache.k[li], st.N, path)
        verify.compact(st.cache.v[li], st.N, path)
    st.N += 1 + len(path)
    st.feat = feats[[0] + path]
    st.out.extend([int(tok[p]) for p in path] + [new_bonus])
    st.bonus = new_bonus
    return tree, path


def spec_generate(tw, dw, prompt, n_new, B, cap, plant=None, choose=None):
    st = prefill(tw, dw, prompt, cap, choose)
    steps = []
    while len(st.out) < n_new:
        _, path = spec_step(tw, dw, st, B, plant, choose)
        steps.append(len(path))
    return st.out[:n_new], steps


def greedy_generate(tw, prompt, n_new, cap, choose=None):
    """Plain decoding, one target forward per token (greedy, or drawing with choose)."""
    st = prefill(tw, None, prompt, cap, choose)
    while len(st.out) < n_new:
        ch, _, _ = target_tree_forward(tw, [st.bonus], [-1], [0], st.cache, st.N, choose)
        st.N += 1
        st.bonus = int(ch[0])
        st.out.append(st.bonus)
    return st.out[:n_new]
