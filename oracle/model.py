"""Decoder-layer arithmetic for the target and the drafter, float64, one row at a time.

The pages describe the models only structurally:
  [DFlash] section "DFlash의 핵심 아이디어" (1, 2): hidden states of several target
  layers are fused into one compressed context signal, and that signal is fed to every
  drafter layer as memory it attends to (not only at the input).
  [DFlash] section "학습 방식도 추론 시나리오에 맞춰 바꿨다": positions inside one
  block see each other; the drafter shares the target's token embedding and LM head.
  [DFlash-news] section "DFlash 핵심 기술 구조": the target's features reach the
  drafter as keys and values of its attention layers ("KV injection").

Readings taken here (Qwen3 family, the target the pages evaluate):
  pre-norm residual layers; RMSNorm with eps; per-head RMSNorm on q and k; rotary
  embedding in rotate-half form with base theta; grouped-query attention (q head h uses
  kv head h // (Hq/Hkv)); softmax scale 1/sqrt(head_dim); SwiGLU MLP
  down(silu(gate) * up); a final RMSNorm before the tied LM head.
  The pages also evaluate Qwen3-Coder-30B-A3B-Instruct ([DFlash] SGLang results; [DDTree]
  "실험 결과"), a mixture-of-experts target; its feed-forward is read as the Qwen3-MoE one:
  a router softmax over the experts, the top-k experts per token with weights renormalised
  to sum 1, each expert a SwiGLU feed-forward, no shared expert.

Rows never interact except through attention, and every row is computed with the same
routine in the same order, so a tree row and the same token decoded alone give bitwise
equal float64 results.  Attention sums only over the keys a row may see, in increasing
slot order; masked keys are skipped rather than added with weight zero.
"""
from __future__ import annotations

import numpy as np


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of the last axis (head_dim) at integer position(s) pos.

    Pair i of the vector is (x[i], x[i + hd/2]) rotated by angle pos * theta^(-2i/hd).
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / hd)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T, computed row by row so that each row's result does not depend on the batch."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    W = np.asarray(W, dtype=np.float64)
    return np.stack([W @ row for row in x])


def silu(x):
    return x / (1.0 + np.exp(-x))


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * K q) weighted sum of V rows, for one query vector."""
    s = (np.asarray(K, np.float64) @ np.asarray(q, np.float64)) * scale
    m = np.max(s)
    p = np.exp(s - m)
    return (p @ np.asarray(V, np.float64)) / np.sum(p)


def qkv_rows(layer, shape, x_normed):
    """Project normed rows to per-head q, k, v (before q/k norm and rotation)."""
    hd, Hq, Hkv = shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    y = linear(x_normed, layer.w_qkv)
    q = y[:, :Hq * hd].reshape(-1, Hq, hd)
    k = y[:, Hq * hd:(Hq + Hkv) * hd].reshape(-1, Hkv, hd)
    v = y[:, (Hq + Hkv) * hd:].reshape(-1, Hkv, hd)
    return q, k, v


def qk_finish(layer, shape, q, k, pos):
    """Per-head RMSNorm of q and k, then rotary embedding at each row's position."""
    pos = np.asarray(pos)
    qn = rms_norm(q, layer.q_norm, shape.rms_eps)
    kn = rms_norm(k, layer.k_norm, shape.rms_eps)
    return rope(qn, pos[:, None], shape.rope_theta), rope(kn, pos[:, None], shape.rope_theta)


def attention_rows(shape, q, keys_of_row):
    """q: [n, Hq, hd]; keys_of_row(i) -> (K [m, Hkv, hd], V [m, Hkv, hd]) visible to row i."""
    Hq, Hkv, hd = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    group = Hq // Hkv
    scale = 1.0 / np.sqrt(hd)
    out = np.zeros((q.shape[0], Hq, hd))
    for i in range(q.shape[0]):
        K, V = keys_of_row(i)
        for h in range(Hq):
            out[i, h] = attend(q[i, h], K[:, h // group], V[:, h // group], scale)
    return out.reshape(q.shape[0], Hq * hd)


def mlp_block(layer, shape, h):
    """h + down(silu(gate) * up) of the post-attention-normed rows."""
    F = shape.d_ff
    x = rms_norm(h, layer.mlp_norm, shape.rms_eps)
    gu = linear(x, layer.w_gate_up)
    act = silu(gu[:, :F]) * gu[:, F:]
    return h + linear(act, layer.w_down)


def moe_route(layer, shape, x):
    """Router of a mixture-of-experts layer: a softmax over the experts' logits, the top_k
    experts by probability (lower expert id first among equal probabilities), their weights
    renormalised to sum to 1.  Returns (ids [n, k], weights [n, k], logits [n, E])."""
    logits = linear(x, layer.w_router)
    E, k = logits.shape[1], shape.top_k
    p = np.exp(logits - logits.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    ids = np.zeros((len(p), k), dtype=np.int64)
    w = np.zeros((len(p), k))
    for i in range(len(p)):
        order = np.lexsort((np.arange(E), -p[i]))[:k]
        ids[i] = order
        w[i] = p[i][order] / np.sum(p[i][order])
    return ids, w, logits


def expert_ffn(layer, e, x_row):
    """Expert e's SwiGLU feed-forward of one normed row: down(silu(gate x) * up x)."""
    Fe = layer.w_experts_down.shape[2]
    gu = np.asarray(layer.w_experts_gate_up[e], np.float64) @ np.asarray(x_row, np.float64)
    return np.asarray(layer.w_experts_down[e], np.float64) @ (silu(gu[:Fe]) * gu[Fe:])


def moe_block(layer, shape, h):
    """h + sum over the chosen experts of weight * expert(x), x the post-attention-normed rows."""
    x = rms_norm(h, layer.mlp_norm, shape.rms_eps)
    ids, w, _ = moe_route(layer, shape, x)
    y = np.zeros_like(x)
    for i in range(len(x)):
        for j in range(shape.top_k):
            y[i] += w[i, j] * expert_ffn(layer, int(ids[i, j]), x[i])
    return h + y


def ffn_block(layer, shape, h):
    """The layer's feed-forward half: dense SwiGLU or mixture of experts."""
    return moe_block(layer, shape, h) if shape.n_experts else mlp_block(layer, shape, h)


def lm_head(weights, h):
    """Final RMSNorm then logits against the (tied) embedding matrix."""
    x = rms_norm(h, weights.final_norm, weights.shape.rms_eps)
    return linear(x, weights.embed)


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Row argmax; ties go to the lowest token id (np.argmax returns the first maximum)."""
    return np.argmax(np.asarray(logits), axis=-1).astype(np.int32)
