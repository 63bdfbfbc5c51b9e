"""Failure detection on the device, in forms that fault and hang nothing.

  * a full cache: a tree forward whose slots run past the cache capacity records
    DF_ERR_CAPACITY in the workspace status word (the rows that do not fit are not written)
  * an exhausted wait: a workspace whose hold word is set makes the GEMM's MMA issuer wait
    for a flag that nothing clears; with a short wait limit the call reports DF_ERR_TIMEOUT,
    having issued no tensor-core work (its loads are drained), and the same workspace then
    serves a normal call
"""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib, engine
from oracle import ddtree

from gpu_util import bf16_dev, rel_close

pytestmark = pytest.mark.gpu


def test_cache_capacity_overflow_is_reported():
    shape = synth.SMALL_TARGET
    tw = synth.target_weights(shape, 4001)
    tm = engine.DeviceModel.from_host(tw)
    b, B, cap = 1, 7, 64
    T = B + 1
    t = ddtree.build_tree(ddtree.log_softmax(np.random.default_rng(1).normal(0, 2, size=(3, shape.vocab))), B)
    t["tok"][0] = 3
    k = torch.zeros(shape.n_layers, b, shape.n_kv_heads, cap, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(shape.n_layers, b, shape.n_kv_heads, 128, cap, dtype=torch.bfloat16, device="cuda")
    st = lambda key: torch.from_numpy(t[key][None].astype(np.int32)).cuda()
    anc = torch.from_numpy(ddtree.ancestor_mask(t["parent"])[None].view(np.int32)).cuda()
    choice = torch.zeros(b, T, dtype=torch.int32, device="cuda")
    ws = _lib.Workspace(_lib.target_tree_forward_workspace_size(tm.cfg, b, T))
    for n, expect in ((cap - T, 0), (cap - T + 3, -4)):  # fits exactly; 3 slots past the end
        clen = torch.tensor([n], dtype=torch.int32, device="cuda")
        _lib.target_tree_forward(tm.cfg, tm.weights, st("tok"), st("depth"), anc, k, v, clen, choice, None, ws)
        torch.cuda.synchronize()
        assert ws.status() == expect, n


def test_exhausted_wait_reports_timeout_and_workspace_recovers():
    M, N, K = 16, 256, 512
    X = synth.normal(4002, "X", (M, K))
    W = synth.normal(4002, "W", (N, K), std=0.05)
    ws = _lib.Workspace(_lib.load().dflash_linear_workspace_size())
    out = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    ws.configure(wait_limit_ns=20_000_000, hold=True)   # 20 ms; the hold word is never cleared
    _lib.linear(bf16_dev(X), bf16_dev(W), out, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == -7
    ws.configure(wait_limit_ns=0, hold=False)
    _lib.linear(bf16_dev(X), bf16_dev(W), out, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rel_close(out.cpu().numpy(), X.astype(np.float64) @ W.astype(np.float64).T, tol=1e-4)
