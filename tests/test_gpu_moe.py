"""The mixture-of-experts target on the GPU vs the oracle: the target tree forward with
router, top-k routing, expert-ordered grouped expert products and the weighted combine.

Routing is a discrete decision on slightly different inputs (bf16 activations on the GPU,
float64 in the oracle), so with a random router rows are compared where the oracle's k-th
and (k+1)-th router logits are clear of that noise; elsewhere the GPU may have picked the
other expert.  An all-zero router makes every probability equal, so the lower-id rule sends
every token to experts 0 .. k-1 with weight 1/k on both sides: every row is compared, the
routed experts hold all rows (several token tiles, a ragged last one) and the rest are empty.
"""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib, engine
from oracle import ddtree, model, step, verify

from gpu_util import bf16_dev, cache_to_oracle, rel_close, to_np

pytestmark = pytest.mark.gpu

N_CTX, CAP = 37, 512


def _shape(E, k):
    return synth.ModelShape(1, 512, 8, 2, 128, 0, 4000, feat_layers=(1,), block_size=8, n_experts=E, top_k=k,
                            d_expert=128)


def _tree(shape, B, seed):
    rng = np.random.default_rng(seed)
    t = ddtree.build_tree(ddtree.log_softmax(rng.normal(0, 2, size=(5, shape.vocab))), B)
    t["tok"][0] = 9
    return t


def _cache(shape, seed):
    kc = synth.normal(seed, "mk", (1, 1, shape.n_kv_heads, CAP, 128))
    vc = synth.normal(seed, "mv", (1, 1, shape.n_kv_heads, CAP, 128))
    kc[..., N_CTX:, :] = 0
    vc[..., N_CTX:, :] = 0
    return kc, vc


def _oracle_cache(kc, vc):
    return cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), 0)


def _gpu_forward(tw, t, kc, vc):
    shape = tw.shape
    tm = engine.DeviceModel.from_host(tw)
    T = len(t["tok"])
    k_t = bf16_dev(kc)
    v_t = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(t[key][None].astype(np.int32)).cuda()
    anc = torch.from_numpy(ddtree.ancestor_mask(t["parent"])[None].view(np.int32)).cuda()
    clen = torch.tensor([N_CTX], dtype=torch.int32, device="cuda")
    choice = torch.zeros(1, T, dtype=torch.int32, device="cuda")
    feat = torch.zeros(1, T, shape.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, 1, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k_t, v_t, clen, choice, feat, ws)
    counts = torch.full((shape.n_layers, shape.n_experts), -1, dtype=torch.int32, device="cuda")
    _lib.target_expert_counts(tm.cfg, 1, T, ws, counts)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return choice[0].cpu().numpy(), to_np(feat[0]), counts.cpu().numpy()


def _router_margin(tw, t, kc, vc):
    """Per tree row, the gap between the oracle's k-th and (k+1)-th router logits."""
    shape, L = tw.shape, tw.layers[0]
    pos = N_CTX + t["depth"]
    h = np.asarray(tw.embed, np.float64)[t["tok"]]
    q, k, v = model.qkv_rows(L, shape, model.rms_norm(h, L.attn_norm, shape.rms_eps))
    q, k = model.qk_finish(L, shape, q, k, pos)
    c = _oracle_cache(kc, vc)
    c.k[0][N_CTX:N_CTX + len(pos)] = k
    c.v[0][N_CTX:N_CTX + len(pos)] = v
    h = h + model.linear(verify.tree_attention(shape, q, c.k[0], c.v[0], N_CTX, t["parent"]), L.w_o)
    lg = np.sort(model.linear(model.rms_norm(h, L.mlp_norm, shape.rms_eps), L.w_router), axis=-1)[:, ::-1]
    return lg[:, shape.top_k - 1] - lg[:, shape.top_k]


def _check(tw, t, kc, vc, rows):
    choice, feat, counts = _gpu_forward(tw, t, kc, vc)
    # every row goes to top_k distinct experts
    assert counts.min() >= 0 and np.all(counts.sum(axis=1) == len(t["tok"]) * tw.shape.top_k)
    assert counts.max() <= len(t["tok"])
    och, ofeat, ologits = step.target_tree_forward(tw, t["tok"], t["parent"], t["depth"], _oracle_cache(kc, vc), N_CTX)
    rel_close(feat[rows], ofeat[rows])
    top2 = np.sort(ologits, axis=-1)[:, -2:]
    sure = rows & ((top2[:, 1] - top2[:, 0]) > 0.02 * np.abs(ologits).max())
    assert sure.mean() > 0.3
    np.testing.assert_array_equal(choice[sure], och[sure])
    return counts


@pytest.mark.parametrize("E,k,B", [(32, 4, 64), (32, 8, 300), (64, 2, 40), (128, 8, 256)])
def test_moe_target_tree_forward_matches_oracle(E, k, B):
    tw = synth.target_weights(_shape(E, k), 5000 + E + B)
    t = _tree(tw.shape, B, E + B)
    kc, vc = _cache(tw.shape, E + B)
    clear = _router_margin(tw, t, kc, vc) > 0.02
    assert clear.mean() > 0.4
    _check(tw, t, kc, vc, clear)


@pytest.mark.parametrize("k,B", [(8, 300), (1, 130)])
def test_moe_all_tokens_to_the_lowest_experts(k, B):
    tw = synth.target_weights(_shape(32, k), 6000 + B)
    tw.layers[0].w_router[:] = 0
    t = _tree(tw.shape, B, B)
    kc, vc = _cache(tw.shape, B)
    ids, w, _ = model.moe_route(tw.layers[0], tw.shape, np.ones((1, tw.shape.d_model)))
    assert ids[0].tolist() == list(range(k)) and np.all(w == 1.0 / k)
    counts = _check(tw, t, kc, vc, np.ones(B + 1, bool))
    np.testing.assert_array_equal(counts[0], [B + 1] * k + [0] * (32 - k))


def test_moe_target_two_sequences_share_the_experts():
    # b = 2 with different cache lengths: the rows of both sequences are routed together
    # (an expert's chunk may hold rows of both); each sequence is compared with the oracle.
    # One layer, so a row's result depends on its own routing only (attention comes first).
    shape = synth.ModelShape(1, 512, 8, 2, 128, 0, 4000, feat_layers=(1,), block_size=8, n_experts=32, top_k=4,
                             d_expert=128)
    tw = synth.target_weights(shape, 7001)
    tm = engine.DeviceModel.from_host(tw)
    b, B, Ns, cap = 2, 90, [37, 200], 512
    T = B + 1
    rng = np.random.default_rng(7)
    kc = synth.normal(7001, "mk2", (1, b, 2, cap, 128))
    vc = synth.normal(7001, "mv2", (1, b, 2, cap, 128))
    trees = []
    for s in range(b):
        kc[:, s, :, Ns[s]:] = 0
        vc[:, s, :, Ns[s]:] = 0
        t = ddtree.build_tree(ddtree.log_softmax(rng.normal(0, 2, size=(7, shape.vocab))), B)
        t["tok"][0] = 100 + s
        trees.append(t)
    k_t = bf16_dev(kc)
    v_t = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(np.stack([t[key] for t in trees]).astype(np.int32)).cuda()
    anc = torch.from_numpy(np.stack([ddtree.ancestor_mask(t["parent"]) for t in trees]).view(np.int32)).cuda()
    clen = torch.tensor(Ns, dtype=torch.int32, device="cuda")
    choice = torch.zeros(b, T, dtype=torch.int32, device="cuda")
    feat = torch.zeros(b, T, shape.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, b, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k_t, v_t, clen, choice, feat, ws)
    counts = torch.zeros(1, 32, dtype=torch.int32, device="cuda")
    _lib.target_expert_counts(tm.cfg, b, T, ws, counts)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert np.all(counts.cpu().numpy().sum(axis=1) == b * T * 4)
    n_clear = 0
    for s in range(b):
        cache = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), s)
        och, ofeat, ologits = step.target_tree_forward(tw, trees[s]["tok"], trees[s]["parent"], trees[s]["depth"],
                                                       cache, Ns[s])
        # rows whose routing is clear in both layers (oracle margins), as in the one-sequence test
        clear = np.ones(T, bool)
        h = np.asarray(tw.embed, np.float64)[trees[s]["tok"]]
        c2 = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), s)
        for li, L in enumerate(tw.layers):
            pos = Ns[s] + trees[s]["depth"]
            q, k_, v_ = model.qkv_rows(L, shape, model.rms_norm(h, L.attn_norm, shape.rms_eps))
            q, k_ = model.qk_finish(L, shape, q, k_, pos)
            c2.k[li][Ns[s]:Ns[s] + T] = k_
            c2.v[li][Ns[s]:Ns[s] + T] = v_
            h = h + model.linear(verify.tree_attention(shape, q, c2.k[li], c2.v[li], Ns[s], trees[s]["parent"]),
                                 L.w_o)
            lg = np.sort(model.linear(model.rms_norm(h, L.mlp_norm, shape.rms_eps), L.w_router), axis=-1)[:, ::-1]
            clear &= (lg[:, shape.top_k - 1] - lg[:, shape.top_k]) > 0.02
            h = model.moe_block(L, shape, h)
        n_clear += clear.sum()
        rel_close(to_np(feat[s])[clear], ofeat[clear])
        top2 = np.sort(ologits, axis=-1)[:, -2:]
        sure = clear & ((top2[:, 1] - top2[:, 0]) > 0.02 * np.abs(ologits).max())
        np.testing.assert_array_equal(choice[s].cpu().numpy()[sure], och[sure])
    assert n_clear > 0.4 * b * T


def test_moe_layer_at_qwen3_30b_a3b_width():
    # One layer at the benchmarked width (d 2048, 32/4 heads, experts of width 768, 8 per row;
    # 32 experts instead of 128 to keep the host weights small) over a 257-row tree: the
    # grouped GEMM runs the step's k-steps (32 for gate/up, 12 for down) and feature tiles
    # (12 and 16).  Sampled rows with clear routing are checked against the oracle.
    shape = synth.ModelShape(1, 2048, 32, 4, 128, 0, 4000, feat_layers=(1,), block_size=16, n_experts=32, top_k=8,
                             d_expert=768)
    tw = synth.target_weights(shape, 8001)
    tm = engine.DeviceModel.from_host(tw)
    N, B, cap = 300, 256, 640
    T = B + 1
    t = ddtree.build_tree(ddtree.log_softmax(np.random.default_rng(8).normal(0, 2, size=(15, shape.vocab))), B)
    t["tok"][0] = 42
    kc = synth.normal(8001, "wk", (1, 1, 4, cap, 128))
    vc = synth.normal(8001, "wv", (1, 1, 4, cap, 128))
    kc[..., N:, :] = 0
    vc[..., N:, :] = 0
    k_t = bf16_dev(kc)
    v_t = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(t[key][None].astype(np.int32)).cuda()
    anc = torch.from_numpy(ddtree.ancestor_mask(t["parent"])[None].view(np.int32)).cuda()
    clen = torch.tensor([N], dtype=torch.int32, device="cuda")
    choice = torch.zeros(1, T, dtype=torch.int32, device="cuda")
    feat = torch.zeros(1, T, shape.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, 1, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k_t, v_t, clen, choice, feat, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    # oracle: attention for every row (the tree's K/V), then the feed-forward of sampled rows
    L = tw.layers[0]
    h = np.asarray(tw.embed, np.float64)[t["tok"]]
    q, k_, v_ = model.qkv_rows(L, shape, model.rms_norm(h, L.attn_norm, shape.rms_eps))
    q, k_ = model.qk_finish(L, shape, q, k_, N + t["depth"])
    c = _oracle_cache(kc, vc)
    c.k[0][N:N + T] = k_
    c.v[0][N:N + T] = v_
    rows = np.random.default_rng(9).choice(T, 40, replace=False)
    rows.sort()
    qs = q[rows]
    o = model.attention_rows(shape, qs, lambda i: (np.concatenate([c.k[0][:N], c.k[0][N + np.array(
        verify.ancestors(t["parent"], int(rows[i])))]]), np.concatenate([c.v[0][:N], c.v[0][N + np.array(
        verify.ancestors(t["parent"], int(rows[i])))]])))
    hs = h[rows] + model.linear(o, L.w_o)
    lg = np.sort(model.linear(model.rms_norm(hs, L.mlp_norm, shape.rms_eps), L.w_router), axis=-1)[:, ::-1]
    clear = (lg[:, 7] - lg[:, 8]) > 0.02
    assert clear.sum() >= 10
    want = model.moe_block(L, shape, hs[clear])
    rel_close(to_np(feat[0])[rows[clear]], want)


def test_moe_prompt_pass_1024_rows():
    # the prompt pass with a mixture-of-experts target: 1024 rows as one causal chain (the
    # library masks the chain itself), 4096 routed rows, so the experts hold up to ~1000 rows
    # each and the dispatch picks chunks; rows with clear routing against the oracle
    shape = _shape(32, 4)
    tw = synth.target_weights(shape, 9001)
    tm = engine.DeviceModel.from_host(tw)
    P, cap = 1024, 1088
    prompt = synth.uniform_ints(9001, "moe.prompt", (1, P), 0, shape.vocab).astype(np.int32)
    k_t = torch.zeros(1, 1, 2, cap, 128, dtype=torch.bfloat16, device="cuda")
    v_t = torch.zeros(1, 1, 2, 128, cap, dtype=torch.bfloat16, device="cuda")
    clen = torch.zeros(1, dtype=torch.int32, device="cuda")
    choice = torch.zeros(1, P, dtype=torch.int32, device="cuda")
    feat = torch.zeros(1, P, shape.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, 1, P))
    _lib.target_tree_forward(tm.cfg, tm.weights, torch.from_numpy(prompt).cuda(), None, None, k_t, v_t, clen, choice,
                             feat, ws)
    counts = torch.zeros(1, 32, dtype=torch.int32, device="cuda")
    _lib.target_expert_counts(tm.cfg, 1, P, ws, counts)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert counts.cpu().numpy().sum() == P * 4
    parent, depth = np.arange(-1, P - 1), np.arange(P)
    L = tw.layers[0]
    h = np.asarray(tw.embed, np.float64)[prompt[0]]
    q, k_, v_ = model.qkv_rows(L, shape, model.rms_norm(h, L.attn_norm, shape.rms_eps))
    q, k_ = model.qk_finish(L, shape, q, k_, depth)
    c = step.KVCache.empty(shape, cap)
    c.k[0][:P] = k_
    c.v[0][:P] = v_
    h = h + model.linear(verify.tree_attention(shape, q, c.k[0], c.v[0], 0, parent), L.w_o)
    lg = np.sort(model.linear(model.rms_norm(h, L.mlp_norm, shape.rms_eps), L.w_router), axis=-1)[:, ::-1]
    clear = (lg[:, 3] - lg[:, 4]) > 0.02
    assert clear.mean() > 0.4
    want = model.moe_block(L, shape, h[clear])
    rel_close(to_np(feat[0])[clear], want)
