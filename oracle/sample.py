"""Drawing the target's next token at temperature T (test infrastructure; never product code).

[DFlash] section "실험 결과" and [DDTree] section "실험 결과" evaluate decoding at
temperature 1.0 as well as greedily, but neither page states how a drafted token is
accepted when the target samples.

Reading (the plainest lossless rule the pages' verification allows): the verifier follows
the target's own outputs down the tree ([DDTree] "방법론 자세히 보기"), so at temperature T
each node's output is a token the target draws from softmax(logits / T) instead of its
argmax, and the walk continues while that token is one of the node's children.  Every
emitted token is then the target's own draw, so the output is distributed exactly as plain
sampling from the target; the tree only decides how many draws one forward pass verifies.

The draw is Gumbel-max: argmax_v (logit_v / T + g_v) with g_v = -log(-log u_v) and u_v
uniform in (0, 1) from a counter-based generator keyed to (seed, sequence, position of the
drawn token, v).  Keying the noise to the absolute position, not to the step or the tree
node, makes speculative decoding reproduce plain sampling token for token under the same
seed.  The generator is the 32-bit finalizer of MurmurHash3 (fmix32, A. Appleby, public
domain) applied in a fixed chain; the GPU implements the same chain from the same
definition.  The decision (the argmax) is taken in fp32, as the kernel takes it.
"""
from __future__ import annotations

import numpy as np

M32 = np.uint32(0xFFFFFFFF)
GOLD = 0x9E3779B9     # mixing constants of the chain (any fixed odd numbers would do)
C_POS = 0xC2B2AE35
C_TOK = 0x27D4EB2F


def fmix32(h):
    """MurmurHash3's 32-bit finalizer, on uint32 scalars or arrays."""
    h = np.asarray(h, dtype=np.uint64) & 0xFFFFFFFF
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h.astype(np.uint32)


def row_seed(seed: int, s: int, n: int) -> np.uint32:
    """Key of the draw for sequence s at absolute position n (the position of the drawn token)."""
    lo, hi = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
    a = fmix32(lo ^ ((GOLD * (s + 1)) & 0xFFFFFFFF))
    a = fmix32(int(a) ^ hi)
    return fmix32((int(a) + C_POS * n) & 0xFFFFFFFF)


def uniforms(seed: int, s: int, n: int, V: int) -> np.ndarray:
    """u_v for v < V, float32: (23 random bits + 1/2) / 2^23, exact in float32 and inside
    [2^-24, 1 - 2^-24], so neither logarithm of the Gumbel transform meets 0 or 1."""
    r = np.uint64(row_seed(seed, s, n))
    v = np.arange(V, dtype=np.uint64)
    h = fmix32(r ^ ((v * C_TOK) & 0xFFFFFFFF))
    return ((h >> 9).astype(np.float32) + np.float32(0.5)) * np.float32(1.0 / 8388608.0)


def gumbel(seed: int, s: int, n: int, V: int) -> np.ndarray:
    u = uniforms(seed, s, n, V)
    return -np.log(-np.log(u))


def draw(logits_row: np.ndarray, temperature: float, seed: int, s: int, n: int) -> int:
    """The token drawn at (s, n): argmax of fp32(logit) * fp32(1/T) + g, lowest id on ties."""
    x = np.asarray(logits_row, np.float64).astype(np.float32) * np.float32(1.0 / temperature)
    x = x + gumbel(seed, s, n, x.shape[-1])
    return int(np.argmax(x))


def noisy_top2_gap(logits_row, temperature, seed, s, n) -> float:
    """Gap between the two largest noisy values (how far the draw is from a tie)."""
    x = np.asarray(logits_row, np.float64).astype(np.float32) * np.float32(1.0 / temperature)
    x = np.sort((x + gumbel(seed, s, n, x.shape[-1])).astype(np.float64))
    return float(x[-1] - x[-2])


def sampler(temperature: float, seed: int, s: int = 0):
    """A chooser for oracle.step: (logits [T, V], positions [T]) -> drawn tokens [T]."""
    def choose(logits, positions):
        return np.array([draw(logits[i], temperature, seed, s, int(positions[i])) for i in range(len(positions))],
                        dtype=np.int64)
    return choose
