"""Pins for the oracle's layer arithmetic, tree attention and the whole speculative loop (CPU)."""
import math
import os

import numpy as np
import pytest
import scipy.special

import synth
from oracle import ddtree, model, step, verify

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_num(tok):
    if tok.startswith("ln"):
        return math.log(float(tok[2:]))
    if "/" in tok:
        a, b = tok.split("/")
        return float(a) / float(b)
    return float(tok)


def test_attend_golden_3x5():
    rows = {"q": [], "k": [], "v": [], "out": []}
    for line in open(os.path.join(GOLDEN, "attention_3x5.txt")):
        if line.startswith("#") or not line.strip():
            continue
        tag, *vals = line.split()
        rows[tag].append([_parse_num(t) for t in vals])
    out = model.attend(np.array(rows["q"][0]), np.array(rows["k"]), np.array(rows["v"]), 1.0)
    np.testing.assert_allclose(out, rows["out"][0], rtol=1e-14)


def test_rms_norm_closed_form():
    x = np.random.default_rng(0).normal(0, 5, size=(3, 64))
    y = model.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-12)
    w = np.linspace(0.5, 2, 64)
    np.testing.assert_allclose(model.rms_norm(x, w, 0.0), y * w, rtol=1e-12)


def test_rope_closed_forms():
    g = np.random.default_rng(1)
    hd, theta = 16, 1e4
    q, k = g.normal(size=hd), g.normal(size=hd)
    np.testing.assert_allclose(model.rope(q, 0, theta), q)
    for m in (1, 7, 300):
        r = model.rope(q, m, theta)
        assert np.linalg.norm(r) == pytest.approx(np.linalg.norm(q), rel=1e-12)
        # pair i as a complex number (x_i + i x_{i+hd/2}) times exp(i m theta^{-2i/hd})
        z = (q[:hd // 2] + 1j * q[hd // 2:]) * np.exp(1j * m * theta ** (-np.arange(hd // 2) * 2 / hd))
        np.testing.assert_allclose(r, np.concatenate([z.real, z.imag]), atol=1e-12)
    # relative-position property of the score
    a = model.rope(q, 10, theta) @ model.rope(k, 4, theta)
    b = model.rope(q, 106, theta) @ model.rope(k, 100, theta)
    assert a == pytest.approx(b, rel=1e-9)


def _dense_causal(q, K, V, scale):
    """Textbook dense masked attention over one sequence, softmax from scipy."""
    s = (q @ K.T) * scale
    mask = np.tril(np.ones(s.shape, dtype=bool), k=K.shape[0] - q.shape[0])
    s = np.where(mask, s, -np.inf)
    return scipy.special.softmax(s, axis=-1) @ V


def test_tree_attention_equals_causal_over_root_path():
    shape = synth.ModelShape(1, 64, 4, 2, 16, 64, 32)
    g = np.random.default_rng(3)
    D, V, B, N = 4, 6, 14, 9
    tree = ddtree.build_tree(ddtree.log_softmax(g.normal(size=(D, V))), B)
    T = B + 1
    q = g.normal(size=(T, 4, 16))
    kc = g.normal(size=(N + T + 3, 2, 16))
    vc = g.normal(size=(N + T + 3, 2, 16))
    out = verify.tree_attention(shape, q, kc, vc, N, tree["parent"]).reshape(T, 4, 16)
    for i in range(T):
        path = verify.ancestors(tree["parent"], i)
        idx = list(range(N)) + [N + j for j in path]
        for h in range(4):
            ref = _dense_causal(q[i, h][None], kc[idx, h // 2], vc[idx, h // 2], 0.25)[0]
            np.testing.assert_allclose(out[i, h], ref, rtol=1e-12, atol=1e-12)


def test_greedy_walk_and_compact_hand_built():
    # root -> {1:a=5, 2:b=7}; 1 -> {3:c=9, 4:d=2}; 3 -> {5:e=4}; 2 -> {6:f=9}
    tok = np.array([-1, 5, 7, 9, 2, 4, 9])
    parent = np.array([-1, 0, 0, 1, 1, 3, 2])
    choice = np.array([5, 9, 0, 4, 0, 8, 0])  # target agrees along 1, 3, 5 then says 8
    path, bonus = verify.greedy_walk(choice, tok, parent)
    assert path == [1, 3, 5] and bonus == 8
    path, bonus = verify.greedy_walk(np.array([3, 0, 0, 0, 0, 0, 0]), tok, parent)
    assert path == [] and bonus == 3
    path, bonus = verify.greedy_walk(np.array([7, 0, 9, 0, 0, 0, 1]), tok, parent)
    assert path == [2, 6] and bonus == 1
    cache = np.arange(30 * 2).reshape(30, 2).astype(float)
    old = cache.copy()
    n_after = verify.compact(cache, 10, [1, 3, 5])
    assert n_after == 14
    np.testing.assert_array_equal(cache[11], old[11])
    np.testing.assert_array_equal(cache[12], old[13])
    np.testing.assert_array_equal(cache[13], old[15])
    np.testing.assert_array_equal(cache[:11], old[:11])


def _toy_models(seed=1001):
    tw = synth.target_weights(synth.TOY_TARGET, seed)
    dw = synth.drafter_weights(synth.TOY_DRAFTER, tw, synth.TOY_TARGET.n_feat, seed)
    return tw, dw


@pytest.mark.slow
def test_speculative_output_equals_plain_greedy():
    """Losslessness: DFlash+DDTree greedy output is the target's own greedy output."""
    tw, dw = _toy_models()
    prompt = synth.uniform_ints(1001, "prompt", (64,), 0, 512)
    n_new, B, cap = 48, 8, 64 + 48 + 16 + 8
    ref = step.greedy_generate(tw, prompt, n_new + 8, cap)
    g = np.random.default_rng(77)

    def plant(st, logits):
        k = len(st.out)
        out = logits.copy()
        for d in range(logits.shape[0]):
            if k - 1 + d + 1 < len(ref) and g.random() < 0.8:
                out[d, ref[k + d]] += 12.0
        return out

    got, steps = step.spec_generate(tw, dw, prompt, n_new, B, cap, plant)
    assert got == ref[:n_new]
    assert sum(steps) > n_new // 3, steps  # the tree was actually used
    assert max(steps) >= 2


def test_drafter_block_is_bidirectional_and_context_conditioned():
    tw, dw = _toy_models()
    feat = synth.normal(5, "feat", (5, 2 * 128))
    ctx = step.KVCache.empty(dw.shape, 32)
    lp1, n1, _ = step.draft_block(dw, feat, ctx, 0, 17)
    assert n1 == 5 and lp1.shape == (3, 512)
    np.testing.assert_allclose(np.exp(lp1.astype(np.float64)).sum(-1), 1, atol=1e-5)
    # a different bonus token changes every position (rows see each other)
    ctx2 = step.KVCache.empty(dw.shape, 32)
    lp2, _, _ = step.draft_block(dw, feat, ctx2, 0, 18)
    assert np.all(np.abs(lp1 - lp2).max(-1) > 1e-6)
    # different context features change the drafts too
    ctx3 = step.KVCache.empty(dw.shape, 32)
    lp3, _, _ = step.draft_block(dw, feat[::-1].copy(), ctx3, 0, 17)
    assert np.all(np.abs(lp1 - lp3).max(-1) > 1e-6)


def _torch_reference_forward(tw, tok, n_ctx_keys=0):
    """Same network from torch library routines: F.rms_norm, complex-valued rotation,
    F.scaled_dot_product_attention (causal, grouped-query).  float64, CPU."""
    import torch
    import torch.nn.functional as F
    sh = tw.shape
    T, d, hd, Hq, Hkv = len(tok), sh.d_model, sh.head_dim, sh.n_q_heads, sh.n_kv_heads
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    h = t(tw.embed)[torch.as_tensor(tok)]
    half = hd // 2
    freq = sh.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2 / hd)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64), torch.arange(T, dtype=torch.float64)[:, None] * freq)

    def rotate(x):  # x [T, H, hd]
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    feats = []
    for li, L in enumerate(tw.layers):
        x = F.rms_norm(h, (d,), t(L.attn_norm), sh.rms_eps)
        y = x @ t(L.w_qkv).T
        q = y[:, :Hq * hd].view(T, Hq, hd)
        k = y[:, Hq * hd:(Hq + Hkv) * hd].view(T, Hkv, hd)
        v = y[:, (Hq + Hkv) * hd:].view(T, Hkv, hd)
        q = rotate(F.rms_norm(q, (hd,), t(L.q_norm), sh.rms_eps))
        k = rotate(F.rms_norm(k, (hd,), t(L.k_norm), sh.rms_eps))
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                           is_causal=True, enable_gqa=True)
        h = h + o.transpose(0, 1).reshape(T, Hq * hd) @ t(L.w_o).T
        x = F.rms_norm(h, (d,), t(L.mlp_norm), sh.rms_eps)
        gu = x @ t(L.w_gate_up).T
        h = h + (F.silu(gu[:, :sh.d_ff]) * gu[:, sh.d_ff:]) @ t(L.w_down).T
        if li + 1 in sh.feat_layers:
            feats.append(h)
    logits = F.rms_norm(h, (d,), t(tw.final_norm), sh.rms_eps) @ t(tw.embed).T
    return torch.cat(feats, -1).numpy(), logits.numpy()


def test_target_forward_matches_torch_library_formulation():
    shape = synth.ModelShape(2, 64, 4, 2, 16, 96, 80, feat_layers=(1, 2))
    tw = synth.target_weights(shape, 55)
    tok = synth.uniform_ints(55, "tok", (7,), 0, 80)
    T = len(tok)
    # a chain tree at N = 0 is a causal prompt pass
    cache = step.KVCache.empty(shape, 16)
    ch, feats, logits = step.target_tree_forward(tw, tok, np.arange(-1, T - 1), np.arange(T), cache, 0)
    rf, rl = _torch_reference_forward(tw, tok)
    np.testing.assert_allclose(feats, rf, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(logits, rl, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(ch, np.argmax(rl, -1))


def _torch_reference_draft(dw, feat, bonus):
    """The drafter block from torch library routines, all context rows at once (positions
    0 .. n-1, block rows n .. n+L-1): F.rms_norm, complex-valued rotation at explicit
    positions, F.scaled_dot_product_attention without a mask over [context ++ block] keys
    (grouped-query), F.log_softmax.  float64, CPU."""
    import torch
    import torch.nn.functional as F
    sh = dw.shape
    d, hd, Hq, Hkv, L = sh.d_model, sh.head_dim, sh.n_q_heads, sh.n_kv_heads, sh.block_size
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    half = hd // 2
    freq = sh.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2 / hd)

    def rotate(x, pos):  # x [T, H, hd], pos [T]
        rot = torch.polar(torch.ones(len(pos), half, dtype=torch.float64), pos[:, None].double() * freq)
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    n = feat.shape[0]
    c = F.rms_norm(t(feat) @ t(dw.fc).T, (d,), t(dw.fc_norm), sh.rms_eps)
    pos_c, pos_b = torch.arange(n), torch.arange(n, n + L)
    block = torch.as_tensor([bonus] + [sh.mask_token] * (L - 1))
    h = t(dw.embed)[block]
    for ly in dw.layers:
        Wq, Wk, Wv = (t(ly.w_qkv)[:Hq * hd], t(ly.w_qkv)[Hq * hd:(Hq + Hkv) * hd], t(ly.w_qkv)[(Hq + Hkv) * hd:])
        kc = rotate(F.rms_norm((c @ Wk.T).view(n, Hkv, hd), (hd,), t(ly.k_norm), sh.rms_eps), pos_c)
        vc = (c @ Wv.T).view(n, Hkv, hd)
        x = F.rms_norm(h, (d,), t(ly.attn_norm), sh.rms_eps)
        q = rotate(F.rms_norm((x @ Wq.T).view(L, Hq, hd), (hd,), t(ly.q_norm), sh.rms_eps), pos_b)
        kb = rotate(F.rms_norm((x @ Wk.T).view(L, Hkv, hd), (hd,), t(ly.k_norm), sh.rms_eps), pos_b)
        vb = (x @ Wv.T).view(L, Hkv, hd)
        K, V = torch.cat([kc, kb]), torch.cat([vc, vb])
        o = F.scaled_dot_product_attention(q.transpose(0, 1), K.transpose(0, 1), V.transpose(0, 1), enable_gqa=True)
        h = h + o.transpose(0, 1).reshape(L, Hq * hd) @ t(ly.w_o).T
        x = F.rms_norm(h, (d,), t(ly.mlp_norm), sh.rms_eps)
        gu = x @ t(ly.w_gate_up).T
        h = h + (F.silu(gu[:, :sh.d_ff]) * gu[:, sh.d_ff:]) @ t(ly.w_down).T
    logits = F.rms_norm(h[1:], (d,), t(dw.final_norm), sh.rms_eps) @ t(dw.embed).T
    return F.log_softmax(logits, -1).numpy(), logits.numpy()


def test_drafter_block_matches_torch_library_formulation():
    # context fusion, per-layer K/V injection at the context positions, and the block's
    # unmasked attention over context ++ block, against an independent formulation
    tw, dw = _toy_models()
    n_feat = synth.TOY_TARGET.n_feat
    feat = synth.normal(6, "feat", (5, n_feat * dw.shape.d_model))
    ctx = step.KVCache.empty(dw.shape, 32)
    lp, n, logits = step.draft_block(dw, feat, ctx, 0, 23)
    rlp, rlogits = _torch_reference_draft(dw, feat, 23)
    assert n == 5
    np.testing.assert_allclose(logits, rlogits, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lp, rlp, rtol=1e-6, atol=1e-6)  # oracle log-probs are stored as fp32
    # the same context committed in two calls (3 rows, then 2) gives the same block
    ctx2 = step.KVCache.empty(dw.shape, 32)
    _, n2, _ = step.draft_block(dw, feat[:3], ctx2, 0, 7)
    lp2, n2, logits2 = step.draft_block(dw, feat[3:], ctx2, n2, 23)
    assert n2 == 5
    np.testing.assert_allclose(logits2, rlogits, rtol=1e-10, atol=1e-12)


def _first_max_by_scan(row):
    """Lowest index of the row's maximum: one pass, a later index replaces the running best
    only when strictly larger."""
    best = 0
    for i in range(1, len(row)):
        if row[i] > row[best]:
            best = i
    return best


def test_argmax_lowest_resolves_planted_ties_to_lowest_id():
    # rows whose maximum occurs at several positions (exact float64 ties), placed before,
    # around and after the other entries; the greedy choice is the lowest of those ids
    g = np.random.default_rng(17)
    V = 97
    logits = g.normal(0, 1, size=(40, V))
    expect = []
    for r in range(logits.shape[0]):
        k = 2 + r % 4
        pos = np.sort(g.choice(V, size=k, replace=False))
        logits[r, pos] = logits[r].max() + 1.0 + (r % 3)
        expect.append(int(pos[0]))
    logits[0, :] = 0.25                     # every entry ties: id 0
    expect[0] = 0
    logits[1, :] = -np.inf                  # all -inf: still id 0
    logits[1, 50] = -np.inf
    expect[1] = 0
    logits[2, V - 1] = logits[2].max() + 5  # a single maximum at the last id
    expect[2] = V - 1
    got = model.argmax_lowest(logits)
    assert got.dtype == np.int32
    np.testing.assert_array_equal(got, expect)
    np.testing.assert_array_equal(got, [_first_max_by_scan(row) for row in logits])
