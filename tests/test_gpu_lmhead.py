"""The two LM-head paths at the full vocabulary (151936 rows, K = 4096), against float64.

At this size every CTA of the GEMM folds several 128-row weight tiles (1187 tiles over one
CTA per SM): the target's fused argmax keeps per-warp running maxima across them, and the
drafter's log-softmax writes per-tile softmax partials that a second pass reduces.

  dflash_linear_argmax      the target LM head of dflash_target_tree_forward: greedy
                            choice, lowest token id among exactly equal maxima
  dflash_linear_logsoftmax  the drafter LM head of dflash_draft_block: log-probs, checked
                            element by element within 1e-3 absolute of the float64
                            log-softmax of the same bf16 products
"""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib
from oracle import ddtree, model

from gpu_util import bf16_dev

pytestmark = pytest.mark.gpu

V, K = 151936, 4096


@pytest.fixture(scope="module")
def embed():
    """Tied embedding of Qwen3-8B shape, N(0, 0.02^2) bf16, on the device and on the host."""
    W = synth.device_normal((V, K), 0.02, 3001, "lmhead.embed")
    return W, W.float().cpu().numpy()


def _logits64(X, W_host, rows=8192):
    """Float64 X W^T, in row chunks of W (the bf16 products are exact in float64)."""
    X64 = X.astype(np.float64)
    out = np.empty((X.shape[0], W_host.shape[0]))
    for c in range(0, W_host.shape[0], rows):
        out[:, c:c + rows] = X64 @ W_host[c:c + rows].astype(np.float64).T
    return out


def _plant_rows(X, W, W_host, picks, scale=0.004):
    """Row r of W := bf16(scale * X[t]) for each (t, r): a clear maximum for token t."""
    for t, r in picks:
        row = synth.bf16_round(X[t] * scale)
        W_host[r] = row
        W[r] = torch.from_numpy(row).to(W.device, torch.bfloat16)


@pytest.mark.parametrize("M", [16, 257, 300])
def test_argmax_full_vocab(embed, M):
    W0, Wh0 = embed
    W, W_host = W0.clone(), Wh0.copy()
    g = np.random.default_rng(M)
    X = synth.normal(3002, f"lmhead.X{M}", (M, K))
    # exact ties: for a third of the tokens, two rows a < b (anywhere in the vocabulary, so in
    # different weight tiles and mostly different CTAs) get the same planted weights
    tokens = g.choice(M, size=M // 3, replace=False)
    rows = g.choice(V, size=2 * len(tokens), replace=False)
    for i, t in enumerate(tokens):
        a, b = sorted(int(x) for x in rows[2 * i:2 * i + 2])
        _plant_rows(X, W, W_host, [(t, a), (t, b)])
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    ws = _lib.linear_argmax(bf16_dev(X), W, out)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = out.cpu().numpy()
    logits = _logits64(X, W_host)
    best = model.argmax_lowest(logits)
    # compare wherever the best value's margin over the next distinct value is clear of the
    # fp32 accumulation error (the planted pairs tie exactly, in both computations)
    top3 = -np.partition(-logits, 2, axis=1)[:, :3]
    top3.sort(axis=1)
    v0 = top3[:, 2]
    v1 = np.where(top3[:, 1] < v0, top3[:, 1], top3[:, 0])
    clear = (v0 - v1) > 1e-4 * np.abs(logits).max(axis=1)
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(got[clear], best[clear])
    for i, t in enumerate(tokens):
        a = min(int(x) for x in rows[2 * i:2 * i + 2])
        assert best[t] == a and got[t] == a, (t, got[t], a)  # the planted pair wins at its lower index
    # elsewhere the choice is still a maximum up to the accumulation error
    sel = logits[np.arange(M), got]
    assert np.all(logits.max(axis=1) - sel <= 1e-4 * np.abs(logits).max(axis=1))


@pytest.mark.parametrize("M", [15, 240])
def test_logsoftmax_full_vocab_within_1e3(embed, M):
    W0, Wh0 = embed
    W, W_host = W0.clone(), Wh0.copy()
    X = synth.normal(3003, f"lmhead.lsX{M}", (M, K))
    # a few rows with a dominant token (peaked distributions) beside flat ones
    _plant_rows(X, W, W_host, [(t, (1000 + 7919 * t) % V) for t in range(0, M, 3)])
    out = torch.full((M, V), np.nan, dtype=torch.float32, device="cuda")
    ws = _lib.linear_logsoftmax(bf16_dev(X), W, out)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = out.cpu().numpy().astype(np.float64)
    ref = ddtree.log_softmax(_logits64(X, W_host)).astype(np.float64)
    err = np.abs(got - ref).max()
    assert err <= 1e-3, err
    np.testing.assert_allclose(np.exp(got).sum(-1), 1.0, atol=1e-3)
