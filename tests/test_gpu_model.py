"""dflash_target_tree_forward and dflash_draft_block vs the oracle, and the whole
speculative loop on the GPU against the target's own greedy decoding."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib, engine
from oracle import ddtree, model, step

from gpu_util import bf16_dev, cache_to_oracle, rel_close, to_np

pytestmark = pytest.mark.gpu

TS, DS = synth.SMALL_TARGET, synth.SMALL_DRAFTER


@pytest.fixture(scope="module")
def models():
    tw = synth.target_weights(TS, 2001)
    dw = synth.drafter_weights(DS, tw, TS.n_feat, 2001)
    tm = engine.DeviceModel.from_host(tw)
    dm = engine.DeviceModel.from_host(dw, embed=tm.embed, n_feat=TS.n_feat)
    return tw, dw, tm, dm


def _clear_choice(gpu_choice, o_choice, o_logits, frac=0.02):
    """Greedy choices must match wherever the oracle's top-2 margin is clear of bf16 noise."""
    top2 = np.sort(o_logits, axis=-1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > frac * np.abs(o_logits).max()
    np.testing.assert_array_equal(gpu_choice[clear], o_choice[clear])
    assert clear.mean() > 0.3  # the comparison is not vacuous
    # where it is not clear, the GPU's choice is still (nearly) a maximum under the oracle
    sel = o_logits[np.arange(len(gpu_choice)), gpu_choice]
    assert np.all(o_logits.max(-1) - sel <= frac * np.abs(o_logits).max())


@pytest.mark.parametrize("b,B,Ns", [(2, 20, [37, 150]), (1, 64, [300]), (3, 0, [5, 0, 77]),
                                    (1, 256, [200]), (2, 131, [37, 350]), (2, 134, [60, 300])])
def test_target_tree_forward_matches_oracle(models, b, B, Ns):
    tw, _, tm, _ = models
    T, cap = B + 1, 512
    rng = np.random.default_rng(B)
    kc = synth.normal(B, "tk", (TS.n_layers, b, TS.n_kv_heads, cap, 128))
    vc = synth.normal(B, "tv", (TS.n_layers, b, TS.n_kv_heads, cap, 128))
    trees = []
    for s in range(b):
        kc[:, s, :, Ns[s]:] = 0
        vc[:, s, :, Ns[s]:] = 0
        t = ddtree.build_tree(ddtree.log_softmax(rng.normal(0, 2, size=(7, TS.vocab))), B)
        t["tok"][0] = int(rng.integers(0, TS.vocab))
        trees.append(t)
    k = bf16_dev(kc)
    v = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(np.stack([t[key] for t in trees]).astype(np.int32)).cuda()
    anc = torch.from_numpy(np.stack([ddtree.ancestor_mask(t["parent"]) for t in trees]).view(np.int32)).cuda()
    clen = torch.tensor(Ns, dtype=torch.int32, device="cuda")
    choice = torch.zeros(b, T, dtype=torch.int32, device="cuda")
    feat = torch.zeros(b, T, TS.n_feat * TS.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, b, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k, v, clen, choice, feat, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert clen.cpu().tolist() == Ns  # not modified
    for s in range(b):
        cache = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), s)
        och, ofeat, ologits = step.target_tree_forward(tw, trees[s]["tok"], trees[s]["parent"], trees[s]["depth"],
                                                       cache, Ns[s])
        rel_close(to_np(feat[s]), ofeat)
        _clear_choice(choice[s].cpu().numpy(), och, ologits)
        # tree K/V written to slots N .. N+T-1 of every layer (V transposed)
        gk = to_np(k[:, s, :, Ns[s]:Ns[s] + T])          # [L][Hkv][T][hd]
        gv = to_np(v[:, s, :, :, Ns[s]:Ns[s] + T])       # [L][Hkv][hd][T]
        for l in range(TS.n_layers):
            rel_close(gk[l], cache.k[l][Ns[s]:Ns[s] + T].transpose(1, 0, 2))
            rel_close(gv[l], cache.v[l][Ns[s]:Ns[s] + T].transpose(1, 2, 0))


@pytest.mark.parametrize("b,ctx0,n_new", [(2, [0, 40], [5, 8]), (1, [123], [1]), (2, [9, 0], [0, 3])])
def test_draft_block_matches_oracle(models, b, ctx0, n_new):
    _, dw, _, dm = models
    cap, max_new, L = 256, 8, DS.block_size
    feat = synth.normal(31, "df", (b, max_new, TS.n_feat * TS.d_model))
    kc = synth.normal(31, "dk", (DS.n_layers, b, DS.n_kv_heads, cap, 128))
    vc = synth.normal(31, "dv", (DS.n_layers, b, DS.n_kv_heads, cap, 128))
    for s in range(b):
        kc[:, s, :, ctx0[s]:] = 0
        vc[:, s, :, ctx0[s]:] = 0
    bonus = [17 + 5 * s for s in range(b)]
    k = bf16_dev(kc)
    v = bf16_dev(vc).transpose(-1, -2).contiguous()
    ctx_len = torch.tensor(ctx0, dtype=torch.int32, device="cuda")
    lp = torch.zeros(b, L - 1, DS.vocab, dtype=torch.float32, device="cuda")
    ws = _lib.Workspace(_lib.draft_block_workspace_size(dm.cfg, b, max_new))
    _lib.draft_block(dm.cfg, dm.weights, bf16_dev(feat), torch.tensor(n_new, dtype=torch.int32, device="cuda"),
                     k, v, ctx_len, torch.tensor(bonus, dtype=torch.int32, device="cuda"), lp, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert ctx_len.cpu().tolist() == [c + n for c, n in zip(ctx0, n_new)]
    g_lp = lp.cpu().numpy()
    for s in range(b):
        ctx = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), s)
        olp, n1, ologits = step.draft_block(dw, feat[s, :n_new[s]].astype(np.float64), ctx, ctx0[s], bonus[s])
        assert n1 == ctx0[s] + n_new[s]
        rel_close(g_lp[s], olp)
        np.testing.assert_allclose(np.exp(g_lp[s].astype(np.float64)).sum(-1), 1.0, atol=1e-3)
        # injected context rows
        gk = to_np(k[:, s, :, ctx0[s]:n1])
        gv = to_np(v[:, s, :, :, ctx0[s]:n1])
        for l in range(DS.n_layers):
            if n_new[s]:
                rel_close(gk[l], ctx.k[l][ctx0[s]:n1].transpose(1, 0, 2))
                rel_close(gv[l], ctx.v[l][ctx0[s]:n1].transpose(1, 2, 0))


@pytest.mark.parametrize("mode,B", [("tree", 16), ("chain", 0)])  # DDTree, and vanilla DFlash (argmax chain)
def test_speculative_loop_is_lossless(models, mode, B):
    """Spec output equals the target's greedy choice at every position whose margin is clear."""
    tw, dw, tm, dm = models
    b, P, n_gen, cap = 2, 40, 48, 512
    prompt = synth.uniform_ints(2001, "prompt", (b, P), 0, TS.vocab)
    ref = [step.greedy_generate(tw, prompt[s], n_gen + 16, cap) for s in range(b)]
    dec = engine.SpecDecoder(tm, dm, b, B, cap, prompt_len=P, mode=mode)
    dec.prefill(torch.from_numpy(prompt).cuda())
    outs = [[int(x)] for x in dec.bonus.cpu().tolist()]
    rng = np.random.default_rng(5)

    def plant(d):
        # harness: bias the drafter's log-probs towards the oracle's greedy continuation
        lp = d.logprobs
        for s in range(b):
            k = len(outs[s])
            for j in range(d.D):
                if k + j < len(ref[s]) and rng.random() < 0.8:
                    lp[s, j, ref[s][k + j]] += 12.0
    dec.plant = plant
    n_acc_total = 0
    while min(len(o) for o in outs) < n_gen:
        dec.step()
        torch.cuda.synchronize()
        assert dec.status() == 0
        acc = dec.acc["acc_tok"].cpu().numpy()
        na = dec.acc["n_acc"].cpu().numpy()
        n_acc_total += int(na.sum())
        for s in range(b):
            outs[s].extend(int(t) for t in acc[s, :na[s] + 1])
    assert n_acc_total > n_gen // 2, n_acc_total
    # teacher-forced oracle pass over prompt + spec output: margins and greedy choices
    for s in range(b):
        seq = list(prompt[s]) + outs[s][:n_gen]
        cache = step.KVCache.empty(tw.shape, len(seq) + 8)
        T = len(seq)
        och, _, ologits = step.target_tree_forward(tw, seq, np.arange(-1, T - 1), np.arange(T), cache, 0)
        pred = och[P - 1:T - 1]           # oracle's choice for each generated position
        got = np.array(outs[s][:n_gen])
        top2 = np.sort(ologits[P - 1:T - 1], axis=-1)[:, -2:]
        clear = (top2[:, 1] - top2[:, 0]) > 0.02 * np.abs(ologits).max()
        bad = np.nonzero(clear & (pred != got))[0]
        assert len(bad) == 0, (s, bad, pred[bad], got[bad])


def test_target_tree_forward_wide_rows():
    # d = 2048: the residual + RMSNorm consumer runs two float4 per thread (the d = 4096 layout)
    shape = synth.ModelShape(1, 2048, 16, 4, 128, 2048, 1024, feat_layers=(1,), block_size=4)
    tw = synth.target_weights(shape, 2003)
    tm = engine.DeviceModel.from_host(tw)
    b, B, N, cap = 1, 12, [45], 128
    rng = np.random.default_rng(3)
    kc = synth.normal(7, "wk", (1, b, 4, cap, 128))
    vc = synth.normal(7, "wv", (1, b, 4, cap, 128))
    kc[:, 0, :, N[0]:] = 0
    vc[:, 0, :, N[0]:] = 0
    t = ddtree.build_tree(ddtree.log_softmax(rng.normal(0, 2, size=(3, shape.vocab))), B)
    t["tok"][0] = 5
    T = B + 1
    k = bf16_dev(kc)
    v = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(t[key][None].astype(np.int32)).cuda()
    anc = torch.from_numpy(ddtree.ancestor_mask(t["parent"])[None].view(np.int32)).cuda()
    clen = torch.tensor(N, dtype=torch.int32, device="cuda")
    choice = torch.zeros(b, T, dtype=torch.int32, device="cuda")
    feat = torch.zeros(b, T, shape.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, b, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k, v, clen, choice, feat, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    cache = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), 0)
    och, ofeat, ologits = step.target_tree_forward(tw, t["tok"], t["parent"], t["depth"], cache, N[0])
    rel_close(to_np(feat[0]), ofeat)
    _clear_choice(choice[0].cpu().numpy(), och, ologits)


def test_target_tree_forward_qwen3_width():
    # One target layer at Qwen3-8B width over a 256-node tree: the four projection GEMMs run
    # at exactly the shapes and launch configuration of the benchmarked step (257 rows;
    # N x K = 6144 x 4096, 4096 x 4096, 24576 x 4096, 4096 x 12288; one CTA per SM,
    # stream-K partial tiles), and their consumers sum those partials.  Small vocabulary and
    # context keep the oracle to seconds.
    shape = synth.ModelShape(1, 4096, 32, 8, 128, 12288, 2048, feat_layers=(1,), block_size=16)
    tw = synth.target_weights(shape, 2005)
    tm = engine.DeviceModel.from_host(tw)
    b, B, N, cap = 1, 256, [64], 384
    rng = np.random.default_rng(5)
    t = ddtree.build_tree(ddtree.log_softmax(rng.normal(0, 2, size=(shape.block_size - 1, shape.vocab))), B)
    t["tok"][0] = 5
    T = B + 1
    kc = synth.normal(7, "fk", (1, b, shape.n_kv_heads, cap, 128))
    vc = synth.normal(7, "fv", (1, b, shape.n_kv_heads, cap, 128))
    kc[:, 0, :, N[0]:] = 0
    vc[:, 0, :, N[0]:] = 0
    k = bf16_dev(kc)
    v = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(t[key][None].astype(np.int32)).cuda()
    anc = torch.from_numpy(ddtree.ancestor_mask(t["parent"])[None].view(np.int32)).cuda()
    clen = torch.tensor(N, dtype=torch.int32, device="cuda")
    choice = torch.zeros(b, T, dtype=torch.int32, device="cuda")
    feat = torch.zeros(b, T, shape.d_model, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, b, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k, v, clen, choice, feat, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    cache = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), 0)
    och, ofeat, ologits = step.target_tree_forward(tw, t["tok"], t["parent"], t["depth"], cache, N[0])
    rel_close(to_np(feat[0]), ofeat)
    _clear_choice(choice[0].cpu().numpy(), och, ologits)
    # the tree rows' K/V went to slots N .. N + B of the cache
    ok = to_np(k)[0, 0][:, N[0]:N[0] + T].transpose(1, 0, 2)
    rel_close(ok, cache.k[0][N[0]:N[0] + T])


def test_prefill_and_first_context_match_oracle(models):
    # prompt scale: 2 x 1024 prompt rows, so the target's GEMMs run several token tiles of 256
    # (M = 2048) and the attention a causal tail of 1024 keys (no ancestor bitmask: the library
    # masks the chain itself); then the drafter fuses all 1024 feature rows into its context
    tw, dw, tm, dm = models
    b, P = 2, 1024
    cap = P + 64
    prompt = synth.uniform_ints(2002, "long_prompt", (b, P), 0, TS.vocab)
    dec = engine.SpecDecoder(tm, dm, b, 16, cap, prompt_len=P)
    choice = dec.prefill(torch.from_numpy(prompt).cuda())
    dec.draft()
    torch.cuda.synchronize()
    assert dec.ws_prefill.status() == 0 and dec.ws_draft0.status() == 0
    assert dec.ctx_len.cpu().tolist() == [P] * b
    g_choice = choice.cpu().numpy()
    g_feat = to_np(dec.prompt_feat)
    g_lp = dec.logprobs.cpu().numpy()
    bonus = dec.bonus.cpu().numpy()
    for s in range(b):
        cache = step.KVCache.empty(TS, cap)
        och, ofeat, ologits = step.target_tree_forward(tw, prompt[s], np.arange(-1, P - 1), np.arange(P), cache, 0)
        rel_close(g_feat[s], ofeat)
        _clear_choice(g_choice[s], och, ologits)
        gk = to_np(dec.k_cache[:, s, :, :P])            # [L][Hkv][P][hd]
        gv = to_np(dec.v_cache[:, s, :, :, :P])         # [L][Hkv][hd][P]
        for l in range(TS.n_layers):
            rel_close(gk[l], cache.k[l][:P].transpose(1, 0, 2))
            rel_close(gv[l], cache.v[l][:P].transpose(1, 2, 0))
        # the first drafter call on the GPU's own feature rows and bonus token
        ctx = step.KVCache.empty(DS, cap)
        olp, n1, _ = step.draft_block(dw, g_feat[s].astype(np.float64), ctx, 0, int(bonus[s]))
        assert n1 == P
        rel_close(g_lp[s], olp)
        np.testing.assert_allclose(np.exp(g_lp[s].astype(np.float64)).sum(-1), 1.0, atol=1e-3)
        ck = to_np(dec.ctx_k[:, s, :, :P])
        cv = to_np(dec.ctx_v[:, s, :, :, :P])
        for l in range(DS.n_layers):
            rel_close(ck[l], ctx.k[l][:P].transpose(1, 0, 2))
            rel_close(cv[l], ctx.v[l][:P].transpose(1, 2, 0))


def test_draft_block_qwen3_width():
    # One drafter layer at Qwen3-8B width (d 4096, 32/8 heads, F 12288) fed 5 target feature
    # layers (context fusion 20480 -> 4096): the drafter's GEMMs run at the benchmarked shapes
    # and launch configuration (16 block rows, 16 + 16 rows for q/k/v, 16 context rows for the
    # fusion), over 512 cached context keys.  Small vocabulary keeps the oracle to seconds.
    V, nf, ctx0, n_new = 2048, 5, 512, 16
    tshape = synth.ModelShape(0, 4096, 32, 8, 128, 12288, V, feat_layers=(), block_size=16)
    tw = synth.target_weights(tshape, 2007)
    ds = synth.ModelShape(1, 4096, 32, 8, 128, 12288, V, block_size=16)
    dw = synth.drafter_weights(ds, tw, nf, 2007)
    tm_embed = bf16_dev(tw.embed)
    dm = engine.DeviceModel.from_host(dw, embed=tm_embed, n_feat=nf)
    cap, L = 640, ds.block_size
    feat = synth.normal(33, "dfq", (1, n_new, nf * ds.d_model))
    kc = synth.normal(33, "dkq", (1, 1, ds.n_kv_heads, cap, 128))
    vc = synth.normal(33, "dvq", (1, 1, ds.n_kv_heads, cap, 128))
    kc[:, :, :, ctx0:] = 0
    vc[:, :, :, ctx0:] = 0
    k = bf16_dev(kc)
    v = bf16_dev(vc).transpose(-1, -2).contiguous()
    ctx_len = torch.tensor([ctx0], dtype=torch.int32, device="cuda")
    lp = torch.zeros(1, L - 1, V, dtype=torch.float32, device="cuda")
    ws = _lib.Workspace(_lib.draft_block_workspace_size(dm.cfg, 1, n_new))
    _lib.draft_block(dm.cfg, dm.weights, bf16_dev(feat), torch.tensor([n_new], dtype=torch.int32, device="cuda"),
                     k, v, ctx_len, torch.tensor([77], dtype=torch.int32, device="cuda"), lp, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0 and ctx_len.item() == ctx0 + n_new
    ctx = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), 0)
    olp, n1, _ = step.draft_block(dw, feat[0].astype(np.float64), ctx, ctx0, 77)
    rel_close(lp[0].cpu().numpy(), olp)
    rel_close(to_np(k[0, 0, :, ctx0:n1]), ctx.k[0][ctx0:n1].transpose(1, 0, 2))
    rel_close(to_np(v[0, 0, :, :, ctx0:n1]), ctx.v[0][ctx0:n1].transpose(1, 2, 0))
