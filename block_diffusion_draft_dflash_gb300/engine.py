"""Device-resident models and the speculative-step driver on top of the C ABI.

``DeviceModel`` holds one transformer's bf16 weights on the GPU together with the
``df_model_cfg`` / ``df_model_weights`` structs the library reads.  ``SpecDecoder`` owns
the KV caches, the drafter's context caches, the per-step buffers and one workspace per
call, and runs a step as the four library calls in order:

    dflash_draft_block -> ddtree_build -> dflash_target_tree_forward -> accept_and_compact

Everything stays on the device; the only host work is launching.  ``prefill`` runs the
prompt through the target as a causal chain and hands its feature rows to the first
drafter call.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib


_LAYER_KEYS = ("attn_norm", "w_qkv", "q_norm", "k_norm", "w_o", "mlp_norm", "w_gate_up", "w_down", "w_router",
               "w_experts_gate_up", "w_experts_down")


def _bf16(x, device):
    return torch.as_tensor(np.ascontiguousarray(x), dtype=torch.float32).to(device=device, dtype=torch.bfloat16).contiguous()


class DeviceModel:
    """One transformer on the device (target or drafter)."""

    def __init__(self, shape, layers, final_norm, embed, fc=None, fc_norm=None, n_feat=None):
        self.shape = shape
        self.layers = layers            # list of dicts of bf16 tensors
        self.final_norm = final_norm
        self.embed = embed
        self.fc = fc
        self.fc_norm = fc_norm
        cfg = _lib.ModelCfg()
        cfg.n_layers, cfg.d_model = shape.n_layers, shape.d_model
        cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
        cfg.d_ff, cfg.vocab = shape.d_ff, shape.vocab
        if fc is not None:
            cfg.n_feat_layers = n_feat
        else:
            cfg.n_feat_layers = len(shape.feat_layers)
            for i, f in enumerate(shape.feat_layers):
                cfg.feat_layers[i] = f
        cfg.block_size = shape.block_size
        cfg.mask_id = shape.mask_token
        cfg.rms_eps, cfg.rope_theta = shape.rms_eps, shape.rope_theta
        cfg.n_experts, cfg.top_k, cfg.d_expert = shape.n_experts, shape.top_k, shape.d_expert
        self.cfg = cfg
        arr = (_lib.LayerWeights * shape.n_layers)()
        for i, L in enumerate(layers):
            for k in _LAYER_KEYS:
                if L.get(k) is not None:
                    setattr(arr[i], k, L[k].data_ptr())
        self._layer_arr = arr
        w = _lib.ModelWeights()
        w.layers = C.cast(arr, C.POINTER(_lib.LayerWeights))
        w.final_norm = final_norm.data_ptr()
        w.embed = embed.data_ptr()
        w.fc = fc.data_ptr() if fc is not None else None
        w.fc_norm = fc_norm.data_ptr() if fc_norm is not None else None
        self.weights = w

    @classmethod
    def from_host(cls, mw, device="cuda", embed=None, n_feat=None):
        """From synth.ModelWeights (numpy, bf16-representable values)."""
        layers = []
        for L in mw.layers:
            layers.append({k: _bf16(getattr(L, k), device) for k in _LAYER_KEYS if getattr(L, k) is not None})
        emb = embed if embed is not None else _bf16(mw.embed, device)
        fc = _bf16(mw.fc, device) if mw.fc is not None else None
        fcn = _bf16(mw.fc_norm, device) if mw.fc_norm is not None else None
        return cls(mw.shape, layers, _bf16(mw.final_norm, device), emb, fc, fcn, n_feat)

    @classmethod
    def random(cls, shape, seed, role, device="cuda", embed=None, n_feat=None, std=0.02):
        """Full-size random init drawn on the device (seeded per tensor name)."""
        from synth import device_normal
        d, hd, F = shape.d_model, shape.head_dim, shape.d_ff
        nqkv = (shape.n_q_heads + 2 * shape.n_kv_heads) * hd
        gain = lambda name, n: device_normal((n,), 0.1, seed, name, device, mean=1.0)
        layers = []
        E, Fe = shape.n_experts, shape.d_expert
        for i in range(shape.n_layers):
            p = f"{role}.{i}"
            L = dict(
                attn_norm=gain(p + ".attn_norm", d), w_qkv=device_normal((nqkv, d), std, seed, p + ".w_qkv", device),
                q_norm=gain(p + ".q_norm", hd), k_norm=gain(p + ".k_norm", hd),
                w_o=device_normal((d, shape.q_dim), std, seed, p + ".w_o", device),
                mlp_norm=gain(p + ".mlp_norm", d))
            if E:
                L.update(w_router=device_normal((E, d), std, seed, p + ".w_router", device),
                         w_experts_gate_up=device_normal((E, 2 * Fe, d), std, seed, p + ".w_experts_gate_up", device),
                         w_experts_down=device_normal((E, d, Fe), std, seed, p + ".w_experts_down", device))
            else:
                L.update(w_gate_up=device_normal((2 * F, d), std, seed, p + ".w_gate_up", device),
                         w_down=device_normal((d, F), std, seed, p + ".w_down", device))
            layers.append(L)
        emb = embed if embed is not None else device_normal((shape.vocab, d), std, seed, "embed", device)
        fc = fcn = None
        if n_feat is not None:
            fc = device_normal((d, n_feat * d), std, seed, role + ".fc", device)
            fcn = gain(role + ".fc_norm", d)
        return cls(shape, layers, gain(role + ".final_norm", d), emb, fc, fcn, n_feat)

    def weight_bytes(self):
        n = sum(t.numel() for L in self.layers for t in L.values()) + self.final_norm.numel()
        n += self.embed.numel()
        if self.fc is not None:
            n += self.fc.numel() + self.fc_norm.numel()
        return 2 * n


class SpecDecoder:
    """State and buffers for b sequences; `step()` runs one speculative step on the GPU.

    mode "tree": DDTree, the B most probable prefixes verified as one flattened tree.
    mode "chain": vanilla DFlash, the drafter's most likely token at each of the D
    positions verified as one chain (B is then D).
    temperature 0: greedy verification; > 0: the target draws its token after every node at
    that temperature (keyed to seed, sequence and position; see dflash.h), and the walk
    follows the drawn tokens.
    """

    def __init__(self, target: DeviceModel, drafter: DeviceModel, b: int, B: int, cap: int, prompt_len: int = 0,
                 device="cuda", mode: str = "tree", temperature: float = 0.0, seed: int = 0):
        assert mode in ("tree", "chain")
        assert temperature >= 0.0
        self.temperature, self.seed = float(temperature), int(seed)
        ts, ds = target.shape, drafter.shape
        self.t, self.d = target, drafter
        self.mode = mode
        self.L = ds.block_size
        self.D = self.L - 1
        if mode == "chain":
            B = self.D
        self.b, self.B = b, B
        self.T = B + 1
        self.cap = cap
        self.device = device
        nf = target.cfg.n_feat_layers
        self.feat_dim = nf * ts.d_model
        dev = dict(device=device)
        z16 = lambda *s: torch.zeros(s, dtype=torch.bfloat16, **dev)
        zi = lambda *s: torch.zeros(s, dtype=torch.int32, **dev)
        self.k_cache = z16(ts.n_layers, b, ts.n_kv_heads, cap, 128)
        self.v_cache = z16(ts.n_layers, b, ts.n_kv_heads, 128, cap)
        self.ctx_k = z16(ds.n_layers, b, ds.n_kv_heads, cap, 128)
        self.ctx_v = z16(ds.n_layers, b, ds.n_kv_heads, 128, cap)
        self.cache_len, self.ctx_len = zi(b), zi(b)
        self.bonus = zi(b)
        self.max_new = self.D + 1
        self.new_feat = z16(b, self.max_new, self.feat_dim)
        self.n_new = zi(b)
        self.logprobs = torch.zeros(b, self.D, ds.vocab, dtype=torch.float32, **dev)
        T = self.T
        W = (T + 31) // 32
        self.tree = dict(tok=zi(b, T), parent=zi(b, T), depth=zi(b, T),
                         score=torch.zeros(b, T, dtype=torch.float32, **dev), anc=zi(b, T, W))
        self.choice = zi(b, T)
        self.tree_feat = z16(b, T, self.feat_dim)
        self.acc = dict(n_new=self.n_new, acc_tok=zi(b, self.max_new), n_acc=zi(b), new_bonus=self.bonus,
                        src_slot=zi(b, self.max_new))
        self.ws_draft = _lib.Workspace(_lib.draft_block_workspace_size(drafter.cfg, b, self.max_new), device)
        self.ws_tree = _lib.Workspace(_lib.chain_build_workspace_size(b, self.D) if mode == "chain" else
                                      _lib.ddtree_build_workspace_size(b, self.D, ds.vocab, B), device)
        self.ws_verify = _lib.Workspace(_lib.target_tree_forward_workspace_size(target.cfg, b, T), device)
        self.ws_accept = _lib.Workspace(_lib.accept_and_compact_workspace_size(b, T), device)
        self.prompt_len = prompt_len
        if prompt_len:
            self.prompt_feat = z16(b, prompt_len, self.feat_dim)
            self.ws_prefill = _lib.Workspace(_lib.target_tree_forward_workspace_size(target.cfg, b, prompt_len), device)
            self.ws_draft0 = _lib.Workspace(_lib.draft_block_workspace_size(drafter.cfg, b, prompt_len), device)
        self.first = False
        self.plant = None  # optional callable(logprobs) run between draft and tree build (harness only)

    # ------------------------------------------------------------------ phases
    def prefill(self, prompt: torch.Tensor):
        """Prompt pass through the target (chain tree at N = 0); sets the first bonus token."""
        b, P = prompt.shape
        assert P == self.prompt_len
        choice = torch.zeros(b, P, dtype=torch.int32, device=self.device)
        self.cache_len.zero_()
        self.ctx_len.zero_()
        # depth and ancestor rows omitted: the library runs the rows as a causal chain
        _lib.target_tree_forward(self.t.cfg, self.t.weights, prompt.to(torch.int32).contiguous(), None, None,
                                 self.k_cache, self.v_cache, self.cache_len, choice, self.prompt_feat, self.ws_prefill,
                                 self.temperature, self.seed)
        self.cache_len.fill_(P)
        self.bonus.copy_(choice[:, -1])
        self.n_new.fill_(P)
        self.first = True
        return choice

    def draft(self):
        if self.first:
            _lib.draft_block(self.d.cfg, self.d.weights, self.prompt_feat, self.n_new, self.ctx_k, self.ctx_v,
                             self.ctx_len, self.bonus, self.logprobs, self.ws_draft0)
            self.first = False
        else:
            _lib.draft_block(self.d.cfg, self.d.weights, self.new_feat, self.n_new, self.ctx_k, self.ctx_v,
                             self.ctx_len, self.bonus, self.logprobs, self.ws_draft)

    def build_tree(self):
        if self.mode == "chain":
            _lib.chain_build(self.logprobs, self.tree, self.ws_tree, root_tok=self.bonus)
        else:
            _lib.ddtree_build(self.logprobs, self.B, self.tree, self.ws_tree, root_tok=self.bonus)

    def verify(self):
        _lib.target_tree_forward(self.t.cfg, self.t.weights, self.tree["tok"], self.tree["depth"], self.tree["anc"],
                                 self.k_cache, self.v_cache, self.cache_len, self.choice, self.tree_feat,
                                 self.ws_verify, self.temperature, self.seed)

    def accept(self):
        _lib.accept_and_compact(self.choice, self.tree["tok"], self.tree["parent"], self.k_cache, self.v_cache,
                                self.cache_len, self.tree_feat, self.new_feat, self.acc, self.ws_accept)

    def step(self):
        self.draft()
        if self.plant is not None:
            self.plant(self)
        self.build_tree()
        self.verify()
        self.accept()

    def capture(self):
        """Capture one step (four library calls) into a CUDA graph; replay with `graph.replay()`.

        Every kernel reads its per-sequence lengths from device memory, so one captured
        step can be replayed for every later step.  Call after at least one eager step.
        """
        assert not self.first, "run the first (context-building) step eagerly"
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.step()
        torch.cuda.current_stream().wait_stream(s)
        self.graph = g
        return g

    def status(self):
        """First device-side error of any call (0 if none); synchronises the stream."""
        for ws in (self.ws_draft, self.ws_tree, self.ws_verify, self.ws_accept):
            s = ws.status()
            if s:
                return s
        return 0
