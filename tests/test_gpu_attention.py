"""tree_verify_attention vs the oracle's ancestor-only attention."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib
from oracle import ddtree, verify

from gpu_util import bf16_dev, rel_close, to_np

pytestmark = pytest.mark.gpu


def _case(seed, b, T, N, Hq, Hkv, cap, D=6, V=50):
    q = synth.normal(seed, "q", (b, T, Hq, 128))
    k = synth.normal(seed, "k", (b, Hkv, cap, 128))
    v = synth.normal(seed, "v", (b, Hkv, cap, 128))
    trees = []
    for s in range(b):
        lp = ddtree.log_softmax(synth.normal(seed, f"lp{s}", (D, V), std=2.0, bf16=False))
        trees.append(ddtree.build_tree(lp, T - 1))
    anc = np.stack([ddtree.ancestor_mask(t["parent"]) for t in trees])
    return q, k, v, trees, anc


def _run_gpu(q, k, v, N, anc):
    b, T, Hq, _ = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    out = torch.zeros(b, T, Hq, 128, dtype=torch.bfloat16, device="cuda")
    ws = _lib.Workspace(_lib.tree_verify_attention_workspace_size(b, T, Hq, Hkv, 128, cap))
    vt = bf16_dev(v).transpose(-1, -2).contiguous()
    _lib.tree_verify_attention(bf16_dev(q), bf16_dev(k), vt, torch.tensor(N, dtype=torch.int32, device="cuda"),
                               torch.from_numpy(anc.view(np.int32)).cuda(), 1 / np.sqrt(128), out, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return to_np(out)


def _oracle(q, k, v, N, tree, s, rows):
    G = q.shape[2] // k.shape[1]
    kc = k[s].transpose(1, 0, 2).astype(np.float64)
    vc = v[s].transpose(1, 0, 2).astype(np.float64)
    from oracle import model
    out = np.zeros((len(rows), q.shape[2], 128))
    for r, i in enumerate(rows):
        idx = list(range(N[s])) + [N[s] + j for j in verify.ancestors(tree["parent"], i)]
        for h in range(q.shape[2]):
            out[r, h] = model.attend(q[s, i, h], kc[idx, h // G], vc[idx, h // G], 1 / np.sqrt(128))
    return out


@pytest.mark.parametrize("b,T,N,Hq,Hkv,cap", [
    (2, 37, [100, 333], 8, 2, 512),      # ragged cache lengths, ragged tree tail
    (1, 257, [1000], 32, 8, 1280),       # B = 256 tree, GQA 4
    (3, 5, [0, 7, 129], 4, 4, 256),      # empty cache, no GQA
    (1, 130, [64], 16, 2, 256),          # GQA 8
])
def test_tree_attention_small(b, T, N, Hq, Hkv, cap):
    q, k, v, trees, anc = _case(7, b, T, N, Hq, Hkv, cap)
    got = _run_gpu(q, k, v, N, anc)
    for s in range(b):
        ref = _oracle(q, k, v, N, trees[s], s, list(range(T)))
        rel_close(got[s], ref)


@pytest.mark.parametrize("T,N", [(257, 4096), (513, 8192)])
def test_tree_attention_full_shape_sampled(T, N):
    # Qwen3-8B attention shape: 32 q heads, 8 kv heads, head_dim 128; sampled rows
    q, k, v, trees, anc = _case(11, 1, T, [N], 32, 8, N + T + 7 & ~7, D=15, V=2000)
    got = _run_gpu(q, k, v, [N], anc)
    rows = sorted(set(np.random.default_rng(0).choice(T, 24, replace=False).tolist()) | {0, T - 1})
    ref = _oracle(q, k, v, [N], trees[0], 0, rows)
    rel_close(got[0, rows], ref)


def test_chain_tree_equals_causal_block():
    # a chain (B = D) makes the ancestor mask causal: compare with plain causal attention
    b, T, N, Hq, Hkv, cap = 1, 16, 40, 8, 2, 128
    q = synth.normal(3, "cq", (b, T, Hq, 128))
    k = synth.normal(3, "ck", (b, Hkv, cap, 128))
    v = synth.normal(3, "cv", (b, Hkv, cap, 128))
    parent = np.arange(-1, T - 1)
    anc = ddtree.ancestor_mask(parent)[None]
    got = _run_gpu(q, k, v, [N], anc)
    from oracle import model
    for i in range(T):
        for h in range(Hq):
            ref = model.attend(q[0, i, h], k[0, h // 4, :N + i + 1].astype(np.float64),
                               v[0, h // 4, :N + i + 1].astype(np.float64), 1 / np.sqrt(128))
            assert np.abs(got[0, i, h] - ref).max() <= 2e-2 * np.abs(ref).max()


@pytest.mark.parametrize("b", [16])
def test_tree_attention_many_waves(b):
    # b*Hkv*ceil(T/32) = 1152 CTAs: several waves of CTAs per SM, no split of the key range
    T, Hq, Hkv, cap = 257, 32, 8, 2048
    N = [900 + 37 * s for s in range(b)]
    q, k, v, trees, anc = _case(13, b, T, N, Hq, Hkv, cap, D=15, V=200)
    got = _run_gpu(q, k, v, N, anc)
    for s in (0, b // 2, b - 1):
        rows = [0, 1, 128, 200, T - 1]
        rel_close(got[s, rows], _oracle(q, k, v, N, trees[s], s, rows))
