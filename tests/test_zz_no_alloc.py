"""ddtree_build_static: the tree builder for callers that cannot allocate device memory
or pass a workspace (its scratch is a fixed array inside the library).  Collected last.

Checks, through the C ABI, that two calls in a row give exactly what ddtree_build gives
with a caller-provided workspace (tree topology is compared bit for bit, as everywhere).
"""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib
from oracle import ddtree

from gpu_util import tree_out

pytestmark = pytest.mark.gpu


def _host(out):
    r = {k: v.cpu().numpy() for k, v in out.items()}
    r["score"] = r["score"].view(np.uint32)
    return r


def test_static_scratch_matches_workspace_version_twice():
    b, D, V = 4, 15, 151936
    lp1 = torch.from_numpy(ddtree.log_softmax(synth.ddtree_logits(1002, b, D, V))).cuda()
    lp2 = torch.from_numpy(ddtree.log_softmax(synth.ddtree_logits(1003, b, D, V))).cuda()
    root = torch.tensor([1, 2, 3, 4], dtype=torch.int32, device="cuda")
    for lp, B in ((lp1, 256), (lp2, 1024)):   # second call reuses (and must clear) the scratch
        ref = tree_out(b, B + 1)
        ws = _lib.Workspace(_lib.ddtree_build_workspace_size(b, D, V, B))
        _lib.ddtree_build(lp, B, ref, ws, root_tok=root)
        got = tree_out(b, B + 1)
        _lib.ddtree_build_static(lp, B, got, root_tok=root)
        torch.cuda.synchronize()
        assert ws.status() == 0
        r, g = _host(ref), _host(got)
        for k in r:
            np.testing.assert_array_equal(g[k], r[k], err_msg=k)


def test_static_scratch_rejects_oversized_call():
    lp = torch.zeros(32, 15, 2048, device="cuda")   # 32 * 15 * 1024 > 262144 top-K entries
    with pytest.raises(_lib.StatusError) as e:
        _lib.ddtree_build_static(lp, 1024, tree_out(32, 1025))
    assert e.value.code == -9
