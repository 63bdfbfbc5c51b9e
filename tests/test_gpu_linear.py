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
