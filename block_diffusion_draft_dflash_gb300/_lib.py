"""ctypes binding of libdflash.so (include/dflash.h).

Argument marshalling only: every function takes torch tensors that already live on the
GPU, checks dtype / device / contiguity, and passes raw pointers plus the current CUDA
stream to the C ABI.  Nothing here computes any part of the speculative step, and there
is no fallback: if the library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

c_i32p = C.POINTER(C.c_int32)


class StatusError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({status_string(code)})")
        self.code = code


class ModelCfg(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("d_ff", C.c_int32), ("vocab", C.c_int32),
                ("n_feat_layers", C.c_int32), ("feat_layers", C.c_int32 * 8), ("block_size", C.c_int32),
                ("mask_id", C.c_int32), ("rms_eps", C.c_float), ("rope_theta", C.c_float),
                ("n_experts", C.c_int32), ("top_k", C.c_int32), ("d_expert", C.c_int32)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("attn_norm", "w_qkv", "q_norm", "k_norm", "w_o", "mlp_norm",
                                          "w_gate_up", "w_down", "w_router", "w_experts_gate_up",
                                          "w_experts_down")]


class ModelWeights(C.Structure):
    _fields_ = [("layers", C.POINTER(LayerWeights)), ("final_norm", C.c_void_p), ("embed", C.c_void_p),
                ("fc", C.c_void_p), ("fc_norm", C.c_void_p)]


_lib = None

_SIGS = {
    "dflash_status_string": (C.c_char_p, [C.c_int]),
    "dflash_check_device": (C.c_int, []),
    "dflash_workspace_status": (C.c_int, [C.c_void_p, C.c_void_p]),
    "dflash_trace_enable": (C.c_int, [C.c_int]),
    "dflash_trace_read": (C.c_int, [C.c_int, C.c_char_p, C.POINTER(C.c_double), C.POINTER(C.c_int)]),
    "ddtree_build_workspace_size": (C.c_size_t, [C.c_int] * 4),
    "ddtree_build": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int] + [C.c_void_p] * 7 +
                     [C.c_size_t, C.c_void_p]),
    "ddtree_build_static": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int] + [C.c_void_p] * 7),
    "dflash_chain_build_workspace_size": (C.c_size_t, [C.c_int, C.c_int]),
    "dflash_chain_build": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int] + [C.c_void_p] * 7 +
                           [C.c_size_t, C.c_void_p]),
    "tree_verify_attention_workspace_size": (C.c_size_t, [C.c_int] * 6),
    "tree_verify_attention": (C.c_int, [C.c_int] * 5 + [C.c_void_p] * 3 + [C.c_int, C.c_void_p, C.c_void_p,
                              C.c_float, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "accept_and_compact_workspace_size": (C.c_size_t, [C.c_int, C.c_int]),
    "accept_and_compact": (C.c_int, [C.c_int, C.c_int] + [C.c_void_p] * 5 + [C.c_int] * 4 + [C.c_void_p] * 2 +
                           [C.c_int, C.c_void_p, C.c_int] + [C.c_void_p] * 6 + [C.c_size_t, C.c_void_p]),
    "dflash_target_tree_forward_workspace_size": (C.c_size_t, [C.c_void_p, C.c_int, C.c_int]),
    "dflash_target_tree_forward": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int] + [C.c_void_p] * 5 +
                                   [C.c_int] + [C.c_void_p] * 4 + [C.c_size_t, C.c_void_p]),
    "dflash_target_tree_forward_sampled": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int] + [C.c_void_p] * 5 +
                                           [C.c_int, C.c_void_p, C.c_float, C.c_ulonglong] + [C.c_void_p] * 3 +
                                           [C.c_size_t, C.c_void_p]),
    "dflash_target_expert_counts": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_size_t, C.c_void_p,
                                              C.c_void_p]),
    "dflash_linear_workspace_size": (C.c_size_t, []),
    "dflash_linear_argmax_workspace_size": (C.c_size_t, [C.c_int]),
    "dflash_linear_argmax": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                       C.c_void_p, C.c_size_t, C.c_void_p]),
    "dflash_linear_sample_workspace_size": (C.c_size_t, [C.c_int]),
    "dflash_linear_sample": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_float, C.c_ulonglong,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "dflash_linear": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int,
                      C.c_void_p, C.c_size_t, C.c_void_p]),
    "dflash_linear_logsoftmax_workspace_size": (C.c_size_t, [C.c_int, C.c_int]),
    "dflash_linear_logsoftmax": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                           C.c_void_p, C.c_size_t, C.c_void_p]),
    "dflash_workspace_configure": (C.c_int, [C.c_void_p, C.c_ulonglong, C.c_int, C.c_void_p]),
    "dflash_plant_logprobs": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p,
                                        C.c_float, C.c_float, C.c_float, C.c_ulonglong, C.c_void_p]),
    "dflash_draft_block_workspace_size": (C.c_size_t, [C.c_void_p, C.c_int, C.c_int]),
    "dflash_draft_block": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_int] + [C.c_void_p] * 4 +
                           [C.c_int] + [C.c_void_p] * 3 + [C.c_size_t, C.c_void_p]),
}


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libdflash.so (building it first if needed) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libdflash.so not built at {_build.LIB}")
    lib = C.CDLL(_build.LIB)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().dflash_status_string(code).decode()


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise StatusError(fn, rc)


def _dev(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Workspace:
    """A device scratch buffer for one of the calls (256-byte aligned via torch)."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = int(nbytes)
        self.buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return C.c_void_p(self.buf.data_ptr())

    def status(self) -> int:
        return load().dflash_workspace_status(self.ptr, _stream())

    def configure(self, wait_limit_ns: int = 0, hold: bool = False):
        """Failure-path settings (see dflash_workspace_configure)."""
        _check("dflash_workspace_configure",
               load().dflash_workspace_configure(self.ptr, int(wait_limit_ns), int(hold), _stream()))


# ----------------------------------------------------------------------------- calls
def ddtree_build_workspace_size(b, D, V, B):
    return load().ddtree_build_workspace_size(b, D, V, B)


def ddtree_build(logprobs, B, out, ws: Workspace, root_tok=None):
    """logprobs [b][D][V] fp32 -> out dict of tok/parent/depth/score/anc tensors (preallocated)."""
    b, D, V = logprobs.shape
    _dev(logprobs, torch.float32, "logprobs")
    for k in ("tok", "parent", "depth"):
        _dev(out[k], torch.int32, k)
    _dev(out["score"], torch.float32, "score")
    _dev(out["anc"], torch.int32, "anc")
    _dev(root_tok, torch.int32, "root_tok")
    _check("ddtree_build", load().ddtree_build(
        _p(logprobs), b, D, V, B, _p(root_tok), _p(out["tok"]), _p(out["parent"]), _p(out["depth"]),
        _p(out["score"]), _p(out["anc"]), ws.ptr, ws.nbytes, _stream()))


def ddtree_build_static(logprobs, B, out, root_tok=None):
    """ddtree_build without a workspace (the library's fixed device scratch; see dflash.h)."""
    b, D, V = logprobs.shape
    _dev(logprobs, torch.float32, "logprobs")
    for k in ("tok", "parent", "depth"):
        _dev(out[k], torch.int32, k)
    _dev(out["score"], torch.float32, "score")
    _dev(out["anc"], torch.int32, "anc")
    _dev(root_tok, torch.int32, "root_tok")
    _check("ddtree_build_static", load().ddtree_build_static(
        _p(logprobs), b, D, V, B, _p(root_tok), _p(out["tok"]), _p(out["parent"]), _p(out["depth"]),
        _p(out["score"]), _p(out["anc"]), _stream()))


def chain_build_workspace_size(b, D):
    return load().dflash_chain_build_workspace_size(b, D)


def chain_build(logprobs, out, ws: Workspace, root_tok=None):
    """logprobs [b][D][V] fp32 -> the argmax chain in out (tok/parent/depth/score/anc, D+1 nodes)."""
    b, D, V = logprobs.shape
    _dev(logprobs, torch.float32, "logprobs")
    for k in ("tok", "parent", "depth"):
        _dev(out[k], torch.int32, k)
    _dev(out["score"], torch.float32, "score")
    _dev(out["anc"], torch.int32, "anc")
    _dev(root_tok, torch.int32, "root_tok")
    _check("dflash_chain_build", load().dflash_chain_build(
        _p(logprobs), b, D, V, _p(root_tok), _p(out["tok"]), _p(out["parent"]), _p(out["depth"]),
        _p(out["score"]), _p(out["anc"]), ws.ptr, ws.nbytes, _stream()))


def tree_verify_attention_workspace_size(b, n_tree, Hq, Hkv, hd, cap):
    return load().tree_verify_attention_workspace_size(b, n_tree, Hq, Hkv, hd, cap)


def tree_verify_attention(q, k_cache, v_cache, cache_len, anc, scale, out, ws: Workspace):
    b, T, Hq, hd = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _dev(t, torch.bfloat16, n)
    _dev(cache_len, torch.int32, "cache_len")
    _dev(anc, torch.int32, "anc")
    _check("tree_verify_attention", load().tree_verify_attention(
        b, T, Hq, Hkv, hd, _p(q), _p(k_cache), _p(v_cache), cap, _p(cache_len), _p(anc), float(scale), _p(out),
        ws.ptr, ws.nbytes, _stream()))


def accept_and_compact_workspace_size(b, n_tree):
    return load().accept_and_compact_workspace_size(b, n_tree)


def accept_and_compact(choice, tok, parent, k_cache, v_cache, cache_len, tree_feat, new_feat, out, ws: Workspace):
    """k_cache [L][b][Hkv][cap][hd], v_cache [L][b][Hkv][hd][cap]; out: n_new, acc_tok, n_acc, new_bonus, src_slot."""
    b, T = choice.shape
    nl, Hkv, cap, hd = (k_cache.shape[0], k_cache.shape[2], k_cache.shape[3], k_cache.shape[4]) \
        if k_cache is not None else (0, 1, 1, 128)
    max_new = out["acc_tok"].shape[1]
    feat_dim = tree_feat.shape[-1] if tree_feat is not None else 0
    _check("accept_and_compact", load().accept_and_compact(
        b, T, _p(choice), _p(tok), _p(parent), _p(k_cache), _p(v_cache), nl, Hkv, hd, cap, _p(cache_len),
        _p(tree_feat), feat_dim, _p(new_feat), max_new, _p(out["n_new"]), _p(out["acc_tok"]), _p(out["n_acc"]),
        _p(out["new_bonus"]), _p(out["src_slot"]), ws.ptr, ws.nbytes, _stream()))


def target_tree_forward_workspace_size(cfg: ModelCfg, b, n_tree):
    return load().dflash_target_tree_forward_workspace_size(C.byref(cfg), b, n_tree)


def target_tree_forward(cfg: ModelCfg, weights: ModelWeights, tok, depth, anc, k_cache, v_cache, cache_len, choice,
                        tree_feat, ws: Workspace, temperature: float = 0.0, seed: int = 0):
    """temperature 0: the greedy choice per node; > 0: the target's temperature draw per node
    (dflash_target_tree_forward_sampled, keyed to seed, sequence and position)."""
    b, T = tok.shape
    cap = k_cache.shape[3]
    if temperature > 0:
        _check("dflash_target_tree_forward_sampled", load().dflash_target_tree_forward_sampled(
            C.byref(cfg), C.byref(weights), b, T, _p(tok), _p(depth), _p(anc), _p(k_cache), _p(v_cache), cap,
            _p(cache_len), float(temperature), seed & 0xFFFFFFFFFFFFFFFF, _p(choice), _p(tree_feat), ws.ptr,
            ws.nbytes, _stream()))
        return
    _check("dflash_target_tree_forward", load().dflash_target_tree_forward(
        C.byref(cfg), C.byref(weights), b, T, _p(tok), _p(depth), _p(anc), _p(k_cache), _p(v_cache), cap,
        _p(cache_len), _p(choice), _p(tree_feat), ws.ptr, ws.nbytes, _stream()))


def target_expert_counts(cfg: ModelCfg, b, n_tree, ws: Workspace, counts):
    """counts [n_layers][n_experts] int32 <- the last mixture-of-experts tree forward's routing."""
    _dev(counts, torch.int32, "counts")
    _check("dflash_target_expert_counts", load().dflash_target_expert_counts(
        C.byref(cfg), b, n_tree, ws.ptr, ws.nbytes, _p(counts), _stream()))


def draft_block_workspace_size(cfg: ModelCfg, b, max_new):
    return load().dflash_draft_block_workspace_size(C.byref(cfg), b, max_new)


def draft_block(cfg: ModelCfg, weights: ModelWeights, new_feat, n_new, ctx_k, ctx_v, ctx_len, bonus, logprobs,
                ws: Workspace):
    b = bonus.shape[0]
    max_new = new_feat.shape[1] if new_feat is not None else 0
    cap = ctx_k.shape[3]
    _check("dflash_draft_block", load().dflash_draft_block(
        C.byref(cfg), C.byref(weights), b, _p(new_feat), max_new, _p(n_new), _p(ctx_k), _p(ctx_v), _p(ctx_len), cap,
        _p(bonus), _p(logprobs), ws.ptr, ws.nbytes, _stream()))


def linear(X, W, out, accumulate=False, ws: Workspace = None):
    """out (+)= X W^T; X [M][K] bf16, W [N][K] bf16, out [M][N] fp32."""
    _dev(X, torch.bfloat16, "X")
    _dev(W, torch.bfloat16, "W")
    _dev(out, torch.float32, "out")
    ws = ws or Workspace(load().dflash_linear_workspace_size(), X.device)
    M, K = X.shape
    N = W.shape[0]
    _check("dflash_linear", load().dflash_linear(_p(X), _p(W), M, N, K, _p(out), int(accumulate), ws.ptr,
                                                 ws.nbytes, _stream()))
    return ws


def linear_argmax(X, W, out, ws: Workspace = None):
    """out[t] = argmax_n (X W^T)[t][n] (lowest n on ties); X [M][K] bf16, W [N][K] bf16, out [M] int32."""
    _dev(X, torch.bfloat16, "X")
    _dev(W, torch.bfloat16, "W")
    _dev(out, torch.int32, "out")
    M, K = X.shape
    N = W.shape[0]
    ws = ws or Workspace(load().dflash_linear_argmax_workspace_size(M), X.device)
    _check("dflash_linear_argmax", load().dflash_linear_argmax(_p(X), _p(W), M, N, K, _p(out), ws.ptr, ws.nbytes,
                                                               _stream()))
    return ws


def linear_sample(X, W, temperature, seed, row_seq, row_pos, out, ws: Workspace = None):
    """out[t] = the temperature draw of row t from softmax((X W^T)[t] / T), keyed to
    (seed, row_seq[t], row_pos[t]); X [M][K] bf16, W [N][K] bf16, row_seq/row_pos/out [M] int32."""
    _dev(X, torch.bfloat16, "X")
    _dev(W, torch.bfloat16, "W")
    for t, name in ((row_seq, "row_seq"), (row_pos, "row_pos"), (out, "out")):
        _dev(t, torch.int32, name)
    M, K = X.shape
    N = W.shape[0]
    ws = ws or Workspace(load().dflash_linear_sample_workspace_size(M), X.device)
    _check("dflash_linear_sample", load().dflash_linear_sample(
        _p(X), _p(W), M, N, K, float(temperature), seed & 0xFFFFFFFFFFFFFFFF, _p(row_seq), _p(row_pos), _p(out),
        ws.ptr, ws.nbytes, _stream()))
    return ws


def linear_logsoftmax(X, W, out, ws: Workspace = None):
    """out[t] = log_softmax(X W^T)[t] (fp32); X [M][K] bf16, W [N][K] bf16, out [M][N] fp32."""
    _dev(X, torch.bfloat16, "X")
    _dev(W, torch.bfloat16, "W")
    _dev(out, torch.float32, "out")
    M, K = X.shape
    N = W.shape[0]
    ws = ws or Workspace(load().dflash_linear_logsoftmax_workspace_size(M, N), X.device)
    _check("dflash_linear_logsoftmax", load().dflash_linear_logsoftmax(_p(X), _p(W), M, N, K, _p(out), ws.ptr,
                                                                       ws.nbytes, _stream()))
    return ws


def plant_logprobs(logprobs, ref, pos, rate, bias, seed, miss_bias=0.0):
    """Harness: plant agreement with reference tokens (see dflash_plant_logprobs).
    ref [b][n_pos][D] int32: tokens expected at depths 1..D of a block starting at position p."""
    _dev(logprobs, torch.float32, "logprobs")
    _dev(ref, torch.int32, "ref")
    _dev(pos, torch.int32, "pos")
    b, D, V = logprobs.shape
    assert ref.shape[0] == b and ref.shape[2] == D
    _check("dflash_plant_logprobs", load().dflash_plant_logprobs(
        _p(logprobs), b, D, V, _p(ref), ref.shape[1], _p(pos), float(rate), float(bias), float(miss_bias), int(seed),
        _stream()))


def trace_enable(on=True):
    load().dflash_trace_enable(int(on))


def trace_read(max_entries=128):
    """{tag: (total ms, launches)} since the last read (synchronises).  A tag is the kernel
    class, optionally followed by a space and the launch shape."""
    names = C.create_string_buffer(64 * max_entries)
    ms = (C.c_double * max_entries)()
    cnt = (C.c_int * max_entries)()
    n = load().dflash_trace_read(max_entries, names, ms, cnt)
    if n < 0:
        raise StatusError("dflash_trace_read", n)
    raw = names.raw
    return {raw[64 * i:64 * i + 64].split(b"\0")[0].decode(): (ms[i], cnt[i]) for i in range(n)}


def exported_symbols():
    """Names declared in include/dflash.h (used by the load/export test)."""
    return list(_SIGS)
