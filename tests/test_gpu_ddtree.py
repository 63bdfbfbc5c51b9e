"""ddtree_build (top-K + best-first heap + ancestor bitsets) vs the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import synth
from block_diffusion_draft_dflash_gb300 import _lib
from oracle import ddtree

from gpu_util import gpu_ddtree

pytestmark = pytest.mark.gpu


def _check_same(g, lp, B, root=None):
    b = lp.shape[0]
    for s in range(b):
        o = ddtree.build_tree(lp[s], B)
        tok = g["tok"][s]
        assert tok[0] == (-1 if root is None else root[s])
        np.testing.assert_array_equal(tok[1:], o["tok"][1:], err_msg=f"tok seq {s}")
        np.testing.assert_array_equal(g["parent"][s], o["parent"], err_msg=f"parent seq {s}")
        np.testing.assert_array_equal(g["depth"][s], o["depth"], err_msg=f"depth seq {s}")
        np.testing.assert_array_equal(g["score"][s].view(np.uint32), o["score"].view(np.uint32))
        np.testing.assert_array_equal(g["anc"][s], ddtree.ancestor_mask(o["parent"]))


@pytest.mark.parametrize("V,D", [(2, 3), (3, 3), (5, 2), (6, 4), (7, 1)])
@pytest.mark.parametrize("mode", ["plain", "ties", "neginf"])
def test_tiny_vocab_bit_exact(V, D, mode):
    g = np.random.default_rng(V * 100 + D)
    x = g.normal(0, 2, size=(3, D, V))
    if mode == "ties":
        x = np.round(x)
    lp = ddtree.log_softmax(x)
    if mode == "neginf":
        lp[g.random(lp.shape) < 0.25] = -np.inf
    total = ddtree.n_prefixes(V, D)
    for B in sorted({0, 1, 2, 5, min(17, total), total}):
        out, st = gpu_ddtree(lp, B, root=[3, 4, 5])
        assert st == 0
        _check_same(out, lp, B, root=[3, 4, 5])
        # the brute-force enumeration agrees too (independent of the heap)
        for s in range(3):
            bf = ddtree.brute_force_tree(lp[s], B)
            np.testing.assert_array_equal(out["parent"][s], bf["parent"])


@pytest.mark.parametrize("B", [16, 64, 256, 512, 1024])
def test_config_shape_budget_sweep(B):
    # DDTree build in isolation: block 16 (15 draft depths), vocab 151936, N(0, 3^2) logits
    # plus a +8 spike per position; 4 sequences per budget here, the full batch below.
    lp = ddtree.log_softmax(synth.ddtree_logits(1002, 4, 15, 151936))
    out, st = gpu_ddtree(lp, B)
    assert st == 0
    _check_same(out, lp, B)


def test_config_full_batch_b64():
    lp = ddtree.log_softmax(synth.ddtree_logits(1002, 64, 15, 151936))
    out, st = gpu_ddtree(lp, 256)
    assert st == 0
    _check_same(out, lp, 256)


def test_ragged_vocab_and_equal_rows():
    # V not a multiple of 4 (scalar path), and rows of all-equal log-probs (every key ties)
    lp = ddtree.log_softmax(np.random.default_rng(1).normal(0, 1, size=(2, 5, 1001)))
    lp[1, 2, :] = np.float32(-np.log(1001.0))
    out, st = gpu_ddtree(lp, 300)
    assert st == 0
    _check_same(out, lp, 300)


@pytest.mark.parametrize("D,B", [(15, 2048), (31, 64)])
def test_max_budget_and_depth(D, B):
    lp = ddtree.log_softmax(np.random.default_rng(2).normal(0, 1, size=(1, D, 4096)))
    out, st = gpu_ddtree(lp, B)
    assert st == 0
    _check_same(out, lp, B)


def test_nan_is_reported():
    lp = ddtree.log_softmax(np.random.default_rng(3).normal(size=(2, 3, 500)))
    lp[1, 1, 17] = np.nan
    _, st = gpu_ddtree(lp, 10)
    assert st == -6


def test_budget_over_prefix_count_rejected():
    lp = torch.zeros(1, 2, 3, device="cuda")
    with pytest.raises(_lib.StatusError) as e:
        _lib.ddtree_build(lp, 13, {k: torch.zeros(1, 14, dtype=torch.int32, device="cuda")
                                   for k in ("tok", "parent", "depth", "anc")} |
                          {"score": torch.zeros(1, 14, device="cuda")}, _lib.Workspace(4096))
    assert e.value.code == -1


def _gpu_chain(lp, root=None):
    from gpu_util import tree_out
    b, D, V = lp.shape
    lp_t = torch.from_numpy(np.ascontiguousarray(lp, dtype=np.float32)).cuda()
    out = tree_out(b, D + 1)
    ws = _lib.Workspace(_lib.chain_build_workspace_size(b, D))
    root_t = None if root is None else torch.as_tensor(root, dtype=torch.int32, device="cuda")
    _lib.chain_build(lp_t, out, ws, root_tok=root_t)
    torch.cuda.synchronize()
    st = ws.status()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["anc"] = res["anc"].view(np.uint32)
    return res, st


@pytest.mark.parametrize("b,D,V,mode", [(64, 15, 151936, "plain"), (3, 15, 151936, "ties"), (2, 31, 1001, "neginf"),
                                        (4, 1, 7, "ties")])
def test_chain_build_bit_exact(b, D, V, mode):
    # vanilla DFlash: the per-position argmax chain, bit-exact against the oracle
    x = synth.ddtree_logits(1002, b, D, V)
    if mode == "ties":
        x = np.round(x)          # many exactly equal log-probs, the maximum among them
    lp = ddtree.log_softmax(x)
    if mode == "neginf":
        lp[np.random.default_rng(0).random(lp.shape) < 0.5] = -np.inf
        lp[0, 0, :] = -np.inf    # a whole row of -inf: the chain takes id 0
    root = list(range(100, 100 + b))
    g, st = _gpu_chain(lp, root)
    assert st == 0
    for s in range(b):
        o = ddtree.build_chain(lp[s])
        assert g["tok"][s][0] == root[s]
        np.testing.assert_array_equal(g["tok"][s][1:], o["tok"][1:])
        np.testing.assert_array_equal(g["parent"][s], o["parent"])
        np.testing.assert_array_equal(g["depth"][s], o["depth"])
        np.testing.assert_array_equal(g["score"][s].view(np.uint32), o["score"].view(np.uint32))
        np.testing.assert_array_equal(g["anc"][s], ddtree.ancestor_mask(o["parent"]))


def test_chain_nan_is_reported():
    lp = ddtree.log_softmax(np.random.default_rng(3).normal(size=(2, 3, 500)))
    lp[1, 2, 499] = np.nan
    _, st = _gpu_chain(lp)
    assert st == -6


@pytest.mark.parametrize("mode", ["ties", "equal_rows", "neginf"])
def test_sampled_topk_paths_bit_exact(mode):
    # vocabularies of 32768 and more use the sampled-threshold top-K; rows where the sampled
    # threshold cannot hold (all keys equal, heavy ties, -inf mass) must still be exact
    g = np.random.default_rng(11)
    b, D, V, B = 2, 4, 40000, 300
    x = g.normal(0, 3, size=(b, D, V))
    if mode == "ties":
        x = np.round(x)                       # large groups of exactly equal keys at the threshold
    lp = ddtree.log_softmax(x)
    if mode == "equal_rows":
        lp[0, 1, :] = np.float32(-np.log(float(V)))   # every key equal: more candidates than the cap
        lp[1, 3, :V // 2] = np.float32(-30.0)
    if mode == "neginf":
        lp[g.random(lp.shape) < 0.7] = -np.inf
        lp[1, 2, :] = -np.inf                 # a row with no finite key
    out, st = gpu_ddtree(lp, B)
    assert st == 0
    _check_same(out, lp, B)


def test_sampled_topk_nan_is_reported():
    lp = ddtree.log_softmax(np.random.default_rng(4).normal(size=(2, 3, 40000)))
    lp[1, 2, 39999] = np.nan
    _, st = gpu_ddtree(lp, 64)
    assert st == -6
