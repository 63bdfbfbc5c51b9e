"""Temperature draws of the target's token on the GPU against the oracle's (oracle/sample.py):
the LM head at the full vocabulary, the target tree forward, and the speculative loop at
temperature 1 against plain sampling from the target.

Both sides take the draw in fp32 (logit * (1/T) + Gumbel noise from the same counter-based
keys), but their logits differ by the accumulation order and their logarithms by an ulp, so
draws are compared where the two largest noisy values are clearly apart."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib, engine
from oracle import ddtree, model, sample, step

from gpu_util import bf16_dev, cache_to_oracle

pytestmark = pytest.mark.gpu

V, K = 151936, 4096
TS, DS = synth.SMALL_TARGET, synth.SMALL_DRAFTER
DF_ERR_ARG = -1


def _logits64(X, W_host, rows=8192):
    X64 = X.astype(np.float64)
    out = np.empty((X.shape[0], W_host.shape[0]))
    for c in range(0, W_host.shape[0], rows):
        out[:, c:c + rows] = X64 @ W_host[c:c + rows].astype(np.float64).T
    return out


@pytest.fixture(scope="module")
def embed():
    W = synth.device_normal((V, K), 0.02, 3101, "sample.embed")
    return W, W.float().cpu().numpy()


@pytest.mark.parametrize("M,temperature", [(16, 1.0), (257, 1.0), (257, 0.6)])
def test_linear_sample_full_vocab(embed, M, temperature):
    W, W_host = embed
    X = synth.normal(3102, f"sample.X{M}", (M, K))
    seq = synth.uniform_ints(3103, f"sample.seq{M}", (M,), 0, 8)
    pos = synth.uniform_ints(3104, f"sample.pos{M}", (M,), 0, 1 << 20)
    seed = 0x1234_5678_9ABC_DEF0
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.from_numpy(a.astype(np.int32)).cuda()
    ws = _lib.linear_sample(bf16_dev(X), W, temperature, seed, dev(seq), dev(pos), out)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = out.cpu().numpy()
    logits = _logits64(X, W_host)
    ref = np.array([sample.draw(logits[t], temperature, seed, int(seq[t]), int(pos[t])) for t in range(M)])
    gap = np.array([sample.noisy_top2_gap(logits[t], temperature, seed, int(seq[t]), int(pos[t])) for t in range(M)])
    clear = gap > 1e-3
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(got[clear], ref[clear])
    # the draws are not the argmax (temperature 1 over 151936 tokens of near-equal logits)
    assert np.mean(got != model.argmax_lowest(logits)) > 0.5
    # another seed, other draws
    out2 = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    _lib.linear_sample(bf16_dev(X), W, temperature, seed + 1, dev(seq), dev(pos), out2)
    torch.cuda.synchronize()
    assert np.mean(out2.cpu().numpy() != got) > 0.5


def test_linear_sample_small_temperature_is_the_argmax(embed):
    W, W_host = embed
    M = 64
    X = synth.normal(3105, "sample.Xcold", (M, K))
    z = torch.zeros(M, dtype=torch.int32, device="cuda")
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    _lib.linear_sample(bf16_dev(X), W, 1e-4, 99, z, torch.arange(M, dtype=torch.int32, device="cuda"), out)
    torch.cuda.synchronize()
    logits = _logits64(X, W_host)
    top2 = np.sort(logits, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 2e-3
    assert clear.mean() > 0.8
    np.testing.assert_array_equal(out.cpu().numpy()[clear], model.argmax_lowest(logits)[clear])


def test_sampled_entries_reject_bad_temperatures(embed):
    W, _ = embed
    X = bf16_dev(synth.normal(3106, "sample.Xbad", (4, K)))
    z = torch.zeros(4, dtype=torch.int32, device="cuda")
    for t in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(_lib.StatusError) as e:
            _lib.linear_sample(X, W, t, 1, z, z, z)
        assert e.value.code == DF_ERR_ARG


@pytest.fixture(scope="module")
def models():
    tw = synth.target_weights(TS, 2101)
    dw = synth.drafter_weights(DS, tw, TS.n_feat, 2101)
    tm = engine.DeviceModel.from_host(tw)
    dm = engine.DeviceModel.from_host(dw, embed=tm.embed, n_feat=TS.n_feat)
    return tw, dw, tm, dm


def _gaps(logits, temperature, seed, s, positions):
    return np.array([sample.noisy_top2_gap(logits[i], temperature, seed, s, int(positions[i]))
                     for i in range(len(positions))])


@pytest.mark.parametrize("b,B,Ns", [(2, 20, [37, 150]), (1, 256, [200])])
def test_target_tree_forward_sampled_matches_oracle(models, b, B, Ns):
    tw, _, tm, _ = models
    T, cap, temperature, seed = B + 1, 512, 1.0, 777
    rng = np.random.default_rng(B + 1)
    kc = synth.normal(B + 1, "stk", (TS.n_layers, b, TS.n_kv_heads, cap, 128))
    vc = synth.normal(B + 1, "stv", (TS.n_layers, b, TS.n_kv_heads, cap, 128))
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
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, b, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k, v, clen, choice, None, ws,
                             temperature, seed)
    torch.cuda.synchronize()
    assert ws.status() == 0
    n_clear = 0
    for s in range(b):
        cache = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), s)
        och, _, ologits = step.target_tree_forward(tw, trees[s]["tok"], trees[s]["parent"], trees[s]["depth"], cache,
                                                   Ns[s], sample.sampler(temperature, seed, s))
        gap = _gaps(ologits, temperature, seed, s, Ns[s] + trees[s]["depth"] + 1)
        clear = gap > 0.02 * np.abs(ologits).max()
        n_clear += int(clear.sum())
        np.testing.assert_array_equal(choice[s].cpu().numpy()[clear], och[clear])
    assert n_clear > 0.5 * b * T


@pytest.mark.parametrize("mode,B", [("tree", 16), ("chain", 0)])  # DDTree, and vanilla DFlash
def test_speculative_sampling_loop_matches_plain_sampling(models, mode, B):
    """At temperature 1 the emitted tokens are the target's own draws: teacher-forced, the
    oracle draws each generated token from the GPU's prefix, wherever the draw is clear."""
    tw, dw, tm, dm = models
    b, P, n_gen, cap, temperature, seed = 2, 40, 48, 512, 1.0, 4242
    prompt = synth.uniform_ints(2102, "prompt", (b, P), 0, TS.vocab)
    ref = [step.greedy_generate(tw, prompt[s], n_gen + 16, cap, sample.sampler(temperature, seed, s))
           for s in range(b)]
    dec = engine.SpecDecoder(tm, dm, b, B, cap, prompt_len=P, mode=mode, temperature=temperature, seed=seed)
    dec.prefill(torch.from_numpy(prompt).cuda())
    outs = [[int(x)] for x in dec.bonus.cpu().tolist()]
    rng = np.random.default_rng(6)

    def plant(d):
        # harness: bias the drafter towards the oracle's sampled continuation
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
    for s in range(b):
        seq = list(prompt[s]) + outs[s][:n_gen]
        Tn = len(seq)
        cache = step.KVCache.empty(tw.shape, Tn + 8)
        och, _, ologits = step.target_tree_forward(tw, seq, np.arange(-1, Tn - 1), np.arange(Tn), cache, 0,
                                                   sample.sampler(temperature, seed, s))
        pred = och[P - 1:Tn - 1]            # the oracle's draw at every generated position
        got = np.array(outs[s][:n_gen])
        gap = _gaps(ologits[P - 1:Tn - 1], temperature, seed, s, np.arange(P, Tn))
        clear = gap > 0.02 * np.abs(ologits).max()
        assert clear.mean() > 0.5
        bad = np.nonzero(clear & (pred != got))[0]
        assert len(bad) == 0, (s, bad, pred[bad], got[bad])
        # and the run is not the greedy one
        assert np.mean(got != model.argmax_lowest(ologits[P - 1:Tn - 1])) > 0.1


def test_moe_target_tree_forward_sampled_matches_oracle():
    """The sampled head after a mixture-of-experts target (an all-zero router: every row to
    experts 0 .. k-1 on both sides, so the routing is exact): draws against the oracle's."""
    shape = synth.ModelShape(1, 512, 8, 2, 128, 0, 4000, feat_layers=(1,), block_size=8, n_experts=32, top_k=4,
                             d_expert=128)
    tw = synth.target_weights(shape, 2103)
    tw.layers[0].w_router[:] = 0
    tm = engine.DeviceModel.from_host(tw)
    B, N, cap, temperature, seed = 60, 37, 256, 1.0, 31337
    T = B + 1
    rng = np.random.default_rng(2103)
    t = ddtree.build_tree(ddtree.log_softmax(rng.normal(0, 2, size=(5, shape.vocab))), B)
    t["tok"][0] = 9
    kc = synth.normal(2103, "smk", (1, 1, shape.n_kv_heads, cap, 128))
    vc = synth.normal(2103, "smv", (1, 1, shape.n_kv_heads, cap, 128))
    kc[..., N:, :] = 0
    vc[..., N:, :] = 0
    k = bf16_dev(kc)
    v = bf16_dev(vc).transpose(-1, -2).contiguous()
    st = lambda key: torch.from_numpy(t[key][None].astype(np.int32)).cuda()
    anc = torch.from_numpy(ddtree.ancestor_mask(t["parent"])[None].view(np.int32)).cuda()
    clen = torch.tensor([N], dtype=torch.int32, device="cuda")
    choice = torch.zeros(1, T, dtype=torch.int32, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, 1, T))
    _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k, v, clen, choice, None, ws,
                             temperature, seed)
    torch.cuda.synchronize()
    assert ws.status() == 0
    cache = cache_to_oracle(torch.from_numpy(kc).to(torch.bfloat16), torch.from_numpy(vc).transpose(-1, -2), 0)
    och, _, ologits = step.target_tree_forward(tw, t["tok"], t["parent"], t["depth"], cache, N,
                                               sample.sampler(temperature, seed, 0))
    gap = _gaps(ologits, temperature, seed, 0, N + t["depth"] + 1)
    clear = gap > 0.02 * np.abs(ologits).max()
    assert clear.mean() > 0.5
    np.testing.assert_array_equal(choice[0].cpu().numpy()[clear], och[clear])
