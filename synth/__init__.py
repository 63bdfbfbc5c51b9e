"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module only draws random numbers and names shapes.  It holds none of the
method's arithmetic (no normalisation, attention, softmax, tree logic): both the
oracle and the CUDA library receive what it produces as plain inputs.

Random numbers come from numpy's counter-based Philox generator, keyed by a seed
and a tensor name, so every tensor is reproducible on its own and identical on
x86 and Arm hosts.  Values that the CUDA path stores in bf16 are rounded to bf16
here (round-to-nearest-even via torch's CPU cast), so both sides see the very same
numbers.  Large full-size tensors (the 8B-parameter shapes) are drawn directly on
the GPU with torch's seeded CUDA generator; those never feed the oracle whole, only
sampled slices copied back to the host.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field, replace

import numpy as np
import torch


# ----------------------------------------------------------------------------- shapes
@dataclass(frozen=True)
class ModelShape:
    """Shape of one decoder-only transformer (Qwen3 family layout).

    feat_layers: 1-indexed target layers whose residual outputs are concatenated
    into the drafter's context feature row (target models only).
    block_size: L, the drafter block (row 0 = bonus token, rows 1..L-1 = mask).
    """
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    feat_layers: tuple = ()
    block_size: int = 16
    mask_id: int = -1  # -1 means vocab-1
    # mixture-of-experts feed-forward (n_experts > 0): n_experts SwiGLU experts of width
    # d_expert, top_k of them per token; d_ff is then unused
    n_experts: int = 0
    top_k: int = 0
    d_expert: int = 0

    @property
    def q_dim(self):
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim

    @property
    def mask_token(self):
        return self.vocab - 1 if self.mask_id < 0 else self.mask_id

    @property
    def n_feat(self):
        return len(self.feat_layers)


# Toy speculative step (oracle-sized): 2-layer target, 1-layer drafter, head_dim 32.
TOY_TARGET = ModelShape(2, 128, 4, 4, 32, 512, 512, feat_layers=(1, 2), block_size=4)
TOY_DRAFTER = ModelShape(1, 128, 4, 4, 32, 512, 512, block_size=4)

# Qwen3-8B-shaped target and the 5-layer DFlash drafter.
QWEN3_8B_TARGET = ModelShape(36, 4096, 32, 8, 128, 12288, 151936,
                             feat_layers=(2, 10, 18, 26, 34), block_size=16)
DFLASH_QWEN3_8B_DRAFTER = ModelShape(5, 4096, 32, 8, 128, 12288, 151936, block_size=16)

# Qwen3-Coder-30B-A3B-shaped target (mixture of experts): 48 layers, d 2048, 32 q / 4 kv heads
# x 128, 128 experts of width 768, 8 per token.
QWEN3_30B_A3B_TARGET = ModelShape(48, 2048, 32, 4, 128, 768, 151936, feat_layers=(2, 14, 26, 38, 46),
                                  block_size=16, n_experts=128, top_k=8, d_expert=768)
DFLASH_QWEN3_30B_A3B_DRAFTER = ModelShape(5, 2048, 32, 4, 128, 6144, 151936, block_size=16)

# Small head_dim-128 shapes for GPU parity: several tiles in every GEMM dimension,
# ragged vocab tail, GQA group 4, two feature layers.
SMALL_TARGET = ModelShape(3, 512, 8, 2, 128, 1536, 4000, feat_layers=(1, 3), block_size=8)
SMALL_DRAFTER = ModelShape(2, 512, 8, 2, 128, 1536, 4000, block_size=8)


# ----------------------------------------------------------------------------- rng
def _key(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:16], "little")


def gen(seed: int, name: str) -> np.random.Generator:
    """Counter-based generator for one named tensor."""
    return np.random.Generator(np.random.Philox(key=_key(seed, name)))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32/fp64 values to the nearest bf16 and return them as float32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def normal(seed, name, shape, std=1.0, mean=0.0, bf16=True):
    x = gen(seed, name).standard_normal(shape, dtype=np.float32) * np.float32(std) + np.float32(mean)
    return bf16_round(x) if bf16 else x


def uniform_ints(seed, name, shape, low, high):
    return gen(seed, name).integers(low, high, size=shape, dtype=np.int64).astype(np.int32)


# ----------------------------------------------------------------------------- weights
@dataclass
class LayerWeights:
    attn_norm: np.ndarray   # [d]
    w_qkv: np.ndarray       # [(Hq+2Hkv)*hd, d]  rows: q heads, k heads, v heads
    q_norm: np.ndarray      # [hd]
    k_norm: np.ndarray      # [hd]
    w_o: np.ndarray         # [d, Hq*hd]
    mlp_norm: np.ndarray    # [d]
    w_gate_up: np.ndarray   # [2F, d]  rows 0..F-1 gate, F..2F-1 up (dense layers)
    w_down: np.ndarray      # [d, F]
    w_router: np.ndarray = None        # mixture of experts: [E, d]
    w_experts_gate_up: np.ndarray = None  # [E, 2 Fe, d]  per expert: gate rows, then up rows
    w_experts_down: np.ndarray = None     # [E, d, Fe]


@dataclass
class ModelWeights:
    shape: ModelShape
    layers: list
    final_norm: np.ndarray  # [d]
    embed: np.ndarray       # [V, d]  token embedding, also the (tied) LM head
    fc: np.ndarray = None   # drafter only: [d, n_feat*d] context fusion
    fc_norm: np.ndarray = None  # drafter only: [d]


def _norm_w(seed, name, n):
    # norm gains near 1 but not equal to 1, so a dropped gain shows up in parity.
    return normal(seed, name, (n,), std=0.1, mean=1.0)


def layer_weights(shape: ModelShape, seed: int, prefix: str, std=0.02) -> LayerWeights:
    d, hd, F = shape.d_model, shape.head_dim, shape.d_ff
    nqkv = (shape.n_q_heads + 2 * shape.n_kv_heads) * hd
    moe = shape.n_experts > 0
    E, Fe = shape.n_experts, shape.d_expert
    return LayerWeights(
        attn_norm=_norm_w(seed, prefix + ".attn_norm", d),
        w_qkv=normal(seed, prefix + ".w_qkv", (nqkv, d), std),
        q_norm=_norm_w(seed, prefix + ".q_norm", hd),
        k_norm=_norm_w(seed, prefix + ".k_norm", hd),
        w_o=normal(seed, prefix + ".w_o", (d, shape.q_dim), std),
        mlp_norm=_norm_w(seed, prefix + ".mlp_norm", d),
        w_gate_up=None if moe else normal(seed, prefix + ".w_gate_up", (2 * F, d), std),
        w_down=None if moe else normal(seed, prefix + ".w_down", (d, F), std),
        w_router=normal(seed, prefix + ".w_router", (E, d), std) if moe else None,
        w_experts_gate_up=normal(seed, prefix + ".w_experts_gate_up", (E, 2 * Fe, d), std) if moe else None,
        w_experts_down=normal(seed, prefix + ".w_experts_down", (E, d, Fe), std) if moe else None,
    )


def target_weights(shape: ModelShape, seed: int, std=0.02) -> ModelWeights:
    layers = [layer_weights(shape, seed, f"target.{i}", std) for i in range(shape.n_layers)]
    return ModelWeights(shape, layers, _norm_w(seed, "target.final_norm", shape.d_model),
                        normal(seed, "embed", (shape.vocab, shape.d_model), std))


def drafter_weights(shape: ModelShape, target: ModelWeights, n_feat: int, seed: int, std=0.02) -> ModelWeights:
    """Drafter layers are its own; the embedding / LM head is the target's (shared, frozen)."""
    layers = [layer_weights(shape, seed, f"drafter.{i}", std) for i in range(shape.n_layers)]
    d = shape.d_model
    return ModelWeights(shape, layers, _norm_w(seed, "drafter.final_norm", d), target.embed,
                        fc=normal(seed, "drafter.fc", (d, n_feat * d), std),
                        fc_norm=_norm_w(seed, "drafter.fc_norm", d))


# ----------------------------------------------------------------------------- DDTree inputs
def ddtree_logits(seed: int, b: int, D: int, V: int, std=3.0, spike=8.0) -> np.ndarray:
    """Per-position logits: i.i.d. N(0, std^2) plus +spike at one uniform token per position.

    Returned as float64; callers turn them into fp32 log-probs with the oracle's
    log-softmax (host side) so that both implementations see identical fp32 inputs.
    """
    g = gen(seed, f"ddtree_logits:{b}x{D}x{V}")
    x = g.standard_normal((b, D, V)) * std
    hot = g.integers(0, V, size=(b, D))
    np.put_along_axis(x, hot[..., None], np.take_along_axis(x, hot[..., None], -1) + spike, -1)
    return x


# ----------------------------------------------------------------------------- device-side draws
def device_normal(shape, std, seed, name, device="cuda", dtype=torch.bfloat16, mean=0.0):
    """Seeded N(mean, std^2) drawn on the GPU (used for full-size weights and caches)."""
    g = torch.Generator(device=device)
    g.manual_seed(_key(seed, name) & ((1 << 63) - 1))
    t = torch.empty(shape, device=device, dtype=torch.float32)
    t.normal_(mean=mean, std=std, generator=g)
    return t.to(dtype)
