"""dflash_linear (the tcgen05 weight-streaming GEMM behind every projection) vs float64."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib

from gpu_util import bf16_dev, rel_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (16, 256, 512), (33, 200, 192), (257, 1000, 1024), (260, 256, 64), (264, 520, 320), (265, 300, 128),
                                   (300, 384, 4096), (600, 130, 256), (1028, 512, 128), (16, 4096, 4096)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_linear_matches_float64(M, N, K, accumulate):
    X = synth.normal(5, f"X{M}", (M, K))
    W = synth.normal(5, f"W{N}x{K}", (N, K), std=0.05)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    out = torch.full((M, N), 0.5 if accumulate else np.nan, dtype=torch.float32, device="cuda")
    ws = _lib.linear(bf16_dev(X), bf16_dev(W), out, accumulate=accumulate)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = out.cpu().numpy().astype(np.float64) - (0.5 if accumulate else 0.0)
    # fp32 accumulation of exact bf16 products: tight bound
    rel_close(got, ref, tol=1e-4)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (33, 1000, 192), (257, 4000, 256), (600, 2000, 128), (1028, 640, 64)])
def test_linear_argmax(M, N, K):
    # the fused-argmax epilogue (target LM head): per token the lowest index among equal maxima
    g = np.random.default_rng(M + N)
    X = synth.normal(9, f"AX{M}", (M, K))
    W = synth.normal(9, f"AW{N}x{K}", (N, K), std=0.05)
    # planted exact ties: for some tokens t, rows a_t < b_t equal and strongly aligned with X[t]
    planted = {}
    for t in g.choice(M, size=min(M, N // 4), replace=False):
        a, b = sorted(g.choice(N, size=2, replace=False))
        if a in planted.values() or b in planted.values():
            continue
        row = synth.bf16_round(X[t] * 0.5)
        W[a] = row
        W[b] = row
        planted[int(t)] = int(a)
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    ws = _lib.linear_argmax(bf16_dev(X), bf16_dev(W), out)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = out.cpu().numpy()
    logits = X.astype(np.float64) @ W.astype(np.float64).T
    # rows with identical weights give bit-identical logits: group them, and expect the lowest
    # index of the winning group wherever its margin over the next group is clear of the fp32
    # accumulation error (bf16 products are exact in fp32; the sums carry ~K ulp)
    rep_of = np.arange(N)
    for t, a in planted.items():
        dup = np.where((W == W[a]).all(axis=1))[0]
        rep_of[dup] = dup.min()
    reps = np.unique(rep_of)
    lg = logits[:, reps]  # one column per group, its lowest index
    order = np.argsort(-lg, axis=1, kind="stable")
    best = reps[order[:, 0]]
    margin = lg[np.arange(M), order[:, 0]] - lg[np.arange(M), order[:, 1]]
    clear = margin > 1e-4 * np.abs(logits).max(axis=1)
    np.testing.assert_array_equal(got[clear], best[clear])
    assert clear.mean() > 0.8
    for t, a in planted.items():
        if clear[t] and best[t] == a:
            assert got[t] == a  # an exact tie resolved to the lower index
    assert np.all((got >= 0) & (got < N))
