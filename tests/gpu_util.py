"""Helpers shared by the GPU parity tests (host-side conversions only)."""
import numpy as np
import torch

from block_diffusion_draft_dflash_gb300 import _lib

DEV = "cuda"


def bf16_dev(x):
    return torch.as_tensor(np.ascontiguousarray(x, dtype=np.float32)).to(DEV, torch.bfloat16).contiguous()


def to_np(t):
    return t.detach().float().cpu().numpy() if t.dtype in (torch.bfloat16, torch.float16) else t.cpu().numpy()


def rel_close(gpu, ref, tol=2e-2):
    """max |g - o| <= tol * max |o| over the tensor (the bf16-storage / fp32-accumulate bound)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref).max()
    scale = np.abs(ref).max()
    assert err <= tol * scale, f"max|d| = {err:.4g} > {tol} * {scale:.4g}"
    return err / max(scale, 1e-30)


def tree_out(b, T, dev=DEV):
    W = (T + 31) // 32
    z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device=dev)
    return dict(tok=z(b, T), parent=z(b, T), depth=z(b, T), score=z(b, T, dt=torch.float32), anc=z(b, T, W))


def gpu_ddtree(lp, B, root=None):
    lp_t = torch.from_numpy(np.ascontiguousarray(lp, dtype=np.float32)).to(DEV)
    b, D, V = lp.shape
    out = tree_out(b, B + 1)
    ws = _lib.Workspace(_lib.ddtree_build_workspace_size(b, D, V, B))
    root_t = None if root is None else torch.as_tensor(root, dtype=torch.int32, device=DEV)
    _lib.ddtree_build(lp_t, B, out, ws, root_tok=root_t)
    torch.cuda.synchronize()
    st = ws.status()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["anc"] = res["anc"].view(np.uint32)
    return res, st


def cache_to_oracle(k_planes, v_planes_t, s):
    """Device-layout caches [L][b][Hkv][cap][hd] and [L][b][Hkv][hd][cap] -> oracle KVCache of sequence s."""
    from oracle import step
    k = to_np(k_planes[:, s]).astype(np.float64)           # [L][Hkv][cap][hd]
    v = to_np(v_planes_t[:, s]).astype(np.float64)         # [L][Hkv][hd][cap]
    return step.KVCache([k[l].transpose(1, 0, 2).copy() for l in range(k.shape[0])],
                        [v[l].transpose(2, 0, 1).copy() for l in range(v.shape[0])])
