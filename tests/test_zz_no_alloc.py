"""ddtree_build_static: the tree builder for callers that cannot allocate device memory
or pass a workspace (its scratch is a fixed array inside the library).  Collected last.

Checks, through the C ABI, that two calls in a row give exactly the oracle's tree and
exactly what ddtree_build gives with a caller-provided workspace (tree topology is compared
bit for bit, as everywhere), also at the largest size the fixed scratch holds.
"""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib
from oracle import ddtree

from gpu_util import tree_out

pytestmark = pytest.mark.gpu

STATIC_TOPK_ENTRIES = 1 << 18  # b * D * min(B, V) limit stated in dflash.h


def _host(out):
    r = {k: v.cpu().numpy() for k, v in out.items()}
    r["score"] = r["score"].view(np.uint32)
    r["anc"] = r["anc"].view(np.uint32)
    return r


def _check_oracle(g, lp, B, root):
    for s in range(lp.shape[0]):
        o = ddtree.build_tree(lp[s], B)
        assert g["tok"][s][0] == root[s]
        np.testing.assert_array_equal(g["tok"][s][1:], o["tok"][1:])
        np.testing.assert_array_equal(g["parent"][s], o["parent"])
        np.testing.assert_array_equal(g["depth"][s], o["depth"])
        np.testing.assert_array_equal(g["score"][s], o["score"].view(np.uint32))
        np.testing.assert_array_equal(g["anc"][s], ddtree.ancestor_mask(o["parent"]))


def _both(lp_np, B, root):
    b, D, V = lp_np.shape
    lp = torch.from_numpy(lp_np).cuda()
    root_t = torch.tensor(root, dtype=torch.int32, device="cuda")
    ref = tree_out(b, B + 1)
    ws = _lib.Workspace(_lib.ddtree_build_workspace_size(b, D, V, B))
    _lib.ddtree_build(lp, B, ref, ws, root_tok=root_t)
    got = tree_out(b, B + 1)
    _lib.ddtree_build_static(lp, B, got, root_tok=root_t)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return _host(ref), _host(got)


def test_static_scratch_matches_oracle_and_workspace_version_twice():
    b, D, V = 4, 15, 151936
    root = [1, 2, 3, 4]
    for seed, B in ((1002, 256), (1003, 1024)):   # the second call reuses (and must clear) the scratch
        lp = ddtree.log_softmax(synth.ddtree_logits(seed, b, D, V))
        r, g = _both(lp, B, root)
        for k in r:
            np.testing.assert_array_equal(g[k], r[k], err_msg=k)
        _check_oracle(g, lp, B, root)


def test_static_scratch_at_its_exact_limit():
    # b * D * min(B, V) == the limit: the last top-K lists end exactly at the scratch's end
    b, D, B, V = 16, 16, 1024, 1500
    assert b * D * min(B, V) == STATIC_TOPK_ENTRIES
    lp = ddtree.log_softmax(synth.ddtree_logits(1004, b, D, V))
    root = list(range(b))
    r, g = _both(lp, B, root)
    for k in r:
        np.testing.assert_array_equal(g[k], r[k], err_msg=k)
    _check_oracle(g, lp, B, root)


def test_static_scratch_rejects_oversized_call():
    lp = torch.zeros(32, 15, 2048, device="cuda")   # 32 * 15 * 1024 > 262144 top-K entries
    with pytest.raises(_lib.StatusError) as e:
        _lib.ddtree_build_static(lp, 1024, tree_out(32, 1025))
    assert e.value.code == -9
