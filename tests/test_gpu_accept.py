"""accept_and_compact vs the oracle's greedy walk and compaction: bit-exact."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib
from oracle import ddtree, verify

pytestmark = pytest.mark.gpu


def _planted_choice(tree, rng, follow=0.7, V=1000):
    """Per node: with prob `follow` the token of its best child, else a token no child has."""
    T = len(tree["tok"])
    choice = np.zeros(T, dtype=np.int32)
    kids = [[] for _ in range(T)]
    for c in range(1, T):
        kids[tree["parent"][c]].append(c)
    for i in range(T):
        toks = {int(tree["tok"][c]) for c in kids[i]}
        if kids[i] and rng.random() < follow:
            choice[i] = tree["tok"][kids[i][0]]
        else:
            t = int(rng.integers(0, V))
            while t in toks:
                t = int(rng.integers(0, V))
            choice[i] = t
    return choice


@pytest.mark.parametrize("b,B,D,n_layers,Hkv,cap", [(3, 40, 7, 2, 2, 256), (2, 256, 15, 3, 8, 4608),
                                                    (1, 1, 15, 1, 1, 64)])
def test_accept_and_compact_matches_oracle(b, B, D, n_layers, Hkv, cap):
    rng = np.random.default_rng(B)
    T = B + 1
    trees, choices = [], []
    for s in range(b):
        lp = ddtree.log_softmax(rng.normal(0, 3, size=(D, 1000)))
        t = ddtree.build_tree(lp, B)
        t["tok"][0] = 7 + s
        trees.append(t)
        choices.append(_planted_choice(t, rng, follow=0.8))
    N = np.array([int(rng.integers(0, cap - T - 1)) for _ in range(b)], dtype=np.int32)
    kc = synth.normal(B, "kc", (n_layers, b, Hkv, cap, 128))
    vc = synth.normal(B, "vc", (n_layers, b, Hkv, cap, 128))
    F = 64
    feat = synth.normal(B, "feat", (b, T, F))
    max_new = D + 1
    dev = "cuda"
    k_t = torch.from_numpy(kc).to(dev, torch.bfloat16)
    v_t = torch.from_numpy(vc).to(dev, torch.bfloat16).transpose(-1, -2).contiguous()
    clen = torch.from_numpy(N).to(dev)
    new_feat = torch.zeros(b, max_new, F, dtype=torch.bfloat16, device=dev)
    out = {k: torch.zeros(b, *(() if k in ("n_new", "n_acc", "new_bonus") else (max_new,)), dtype=torch.int32,
                          device=dev) for k in ("n_new", "acc_tok", "n_acc", "new_bonus", "src_slot")}
    i32 = lambda key: torch.from_numpy(np.stack([t[key] for t in trees])).to(dev)
    ws = _lib.Workspace(_lib.accept_and_compact_workspace_size(b, T))
    _lib.accept_and_compact(torch.from_numpy(np.stack(choices)).to(dev), i32("tok"), i32("parent"), k_t, v_t, clen,
                            torch.from_numpy(feat).to(dev, torch.bfloat16), new_feat, out, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    k_g = k_t.float().cpu().numpy()
    v_g = v_t.transpose(-1, -2).float().cpu().numpy()
    for s in range(b):
        path, bonus = verify.greedy_walk(choices[s], trees[s]["tok"], trees[s]["parent"])
        a = len(path)
        assert out["n_acc"][s].item() == a and out["n_new"][s].item() == a + 1
        assert out["new_bonus"][s].item() == bonus
        acc = out["acc_tok"][s].cpu().numpy()
        np.testing.assert_array_equal(acc[:a], trees[s]["tok"][path])
        assert acc[a] == bonus
        src = out["src_slot"][s].cpu().numpy()
        np.testing.assert_array_equal(src[:a], N[s] + np.array(path, dtype=np.int64))
        assert clen[s].item() == N[s] + 1 + a
        for l in range(n_layers):
            ko = kc[l, s].transpose(1, 0, 2).copy()   # [cap][Hkv][hd]
            vo = vc[l, s].transpose(1, 0, 2).copy()
            verify.compact(ko, int(N[s]), path)
            verify.compact(vo, int(N[s]), path)
            np.testing.assert_array_equal(k_g[l, s].transpose(1, 0, 2), ko)
            np.testing.assert_array_equal(v_g[l, s].transpose(1, 0, 2), vo)
        nf = new_feat[s].float().cpu().numpy()
        np.testing.assert_array_equal(nf[:a + 1], feat[s][[0] + path])
    assert sum(out["n_acc"].cpu().numpy()) > 0


def _splitmix64(x):
    # published definition (Steele, Lea, Flood 2014), on Python ints mod 2^64
    M = (1 << 64) - 1
    x = (x + 0x9E3779B97F4A7C15) & M
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & M
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & M
    return x ^ (x >> 31)


@pytest.mark.parametrize("miss_bias", [0.0, 14.5])
def test_plant_logprobs_harness(miss_bias):
    # the benchmark's acceptance plant: the planted rows are a renormalised bias at the
    # reference token, drawn per (seed, sequence, position, depth); the others are unchanged,
    # or near misses (the bias on a decoy, the miss bias on the reference)
    b, D, V, n_pos, rate, bias, seed = 3, 15, 5000, 400, 0.6, 16.0, 77
    lp = ddtree.log_softmax(np.random.default_rng(0).normal(0, 1.3, size=(b, D, V)))
    ref = np.random.default_rng(1).integers(0, V, size=(b, n_pos, D)).astype(np.int32)
    pos = np.array([10, 200, 250], dtype=np.int32)
    ref[2, 250, 3:9] = -1                                     # no reference at these depths
    lp_t = torch.from_numpy(lp).cuda()
    _lib.plant_logprobs(lp_t, torch.from_numpy(ref).cuda(), torch.from_numpy(pos).cuda(), rate, bias, seed,
                        miss_bias=miss_bias)
    got = lp_t.cpu().numpy().astype(np.float64)
    n_planted = 0
    for s in range(b):
        for d in range(1, D + 1):
            h = _splitmix64(seed ^ _splitmix64((s << 40) ^ (int(pos[s]) << 8) ^ d))
            r = int(ref[s, pos[s], d - 1])
            planted = r >= 0 and (h >> 11) / 2.0 ** 53 < rate
            row = lp[s, d - 1].astype(np.float64)
            if r < 0 or (not planted and miss_bias == 0.0):
                np.testing.assert_array_equal(got[s, d - 1], row)
                continue
            n_planted += planted
            x = row.copy()
            if planted:
                x[r] += bias
            else:
                decoy = (r + 1 + _splitmix64(h) % (V - 1)) % V
                assert decoy != r
                x[decoy] += bias
                x[r] += miss_bias
            expect = x - np.log(np.sum(np.exp(x)))    # log-softmax of the biased logits
            np.testing.assert_allclose(got[s, d - 1], expect, atol=2e-5)
            order = np.argsort(-got[s, d - 1])
            if planted:
                assert order[0] == r
            else:  # the decoy and the reference lead (in either order, by their own logits)
                assert set(order[:2].tolist()) == {decoy, r}
    assert 10 < n_planted < 3 * D
