"""Device-resident draft layers built from host arrays, wired to the C ABI.

``DraftLayer`` owns the device copies of one layer's weights, its KV cache
and rotary table, and the ``mtp_layer_desc`` that points at them.
``DraftChain`` holds several layers that share the lm_head and the embedding
table (the three-layer MiMo-style chain).
"""

from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib as L
from .api import _p, affine4, attn_geom, moe_weights, workspace


def _dev(a, device):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device)


class DeviceAffine:
    def __init__(self, w, device, n=None, k=None):
        q, s, b = w
        self.q = _dev(np.asarray(q).reshape(-1, np.asarray(q).shape[-1]), device)
        self.s = _dev(np.asarray(s).reshape(-1, np.asarray(s).shape[-1]), device)
        self.b = _dev(np.asarray(b).reshape(-1, np.asarray(b).shape[-1]), device)
        self.desc = affine4(self.q, self.s, self.b, n, k)


class SharedHead:
    """lm_head and embedding table shared by the layers of a chain."""

    def __init__(self, shared: dict, device="cuda"):
        self.lm_head = DeviceAffine(shared["lm_head"], device)
        self.embed = _dev(shared["embed"], device) if "embed" in shared else None


class DraftLayer:
    def __init__(self, cfg, weights: dict, shared: SharedHead, state: dict, m_max: int | None = None,
                 device="cuda", bf16_stacks: bool = False):
        self.cfg = cfg
        self.device = device
        self.m_max = cfg.m if m_max is None else m_max
        H = cfg.hidden
        self.t = {}
        for name in ("enorm", "hnorm", "attn_norm", "post_norm", "final_norm", "q_norm", "k_norm",
                     "sinks"):
            if name in weights:
                self.t[name] = _dev(weights[name], device)
        self.aff = {}
        for name in ("eh_proj", "wq", "wk", "wv", "wo", "ffn_gate", "ffn_up", "ffn_down",
                     "sh_gate", "sh_up", "sh_down"):
            if name in weights:
                self.aff[name] = DeviceAffine(weights[name], device)
        self.shared = shared
        self.k_cache = _dev(state["k_cache"], device)
        self.v_cache = _dev(state["v_cache"], device)
        self.cache_cap = self.k_cache.shape[1]
        self.rope = torch.empty(self.cache_cap * cfg.rot_dim, dtype=torch.float32, device=device)
        from .api import mtp_rope_table
        mtp_rope_table(self.rope, self.cache_cap, cfg.rot_dim, cfg.rope_theta)
        self.moe = None
        if cfg.moe:
            E, Ie = cfg.n_experts, cfg.expert_intermediate
            for name in ("exp_gate", "exp_up", "exp_down"):
                q, s, b = weights[name]
                flat = (q.reshape(-1, q.shape[-1]), s.reshape(-1, s.shape[-1]), b.reshape(-1, b.shape[-1]))
                if bf16_stacks:
                    # the stacks as MlxAffineMoeStack holds them: float32 scales and
                    # biases cast to bfloat16 (round to nearest even) at upload
                    from .api import affine4_bf16_scales
                    d = DeviceAffine.__new__(DeviceAffine)
                    d.q = _dev(flat[0], device)
                    d.s = torch.from_numpy(np.ascontiguousarray(flat[1])).to(torch.bfloat16).to(device)
                    d.b = torch.from_numpy(np.ascontiguousarray(flat[2])).to(torch.bfloat16).to(device)
                    d.desc = affine4_bf16_scales(d.q, d.s, d.b)
                    self.aff[name] = d
                else:
                    self.aff[name] = DeviceAffine(flat, device)
            self.t["router"] = _dev(weights["router"], device)
            self.t["sh_gate_inp"] = _dev(weights["sh_gate_inp"], device)
            self.moe = moe_weights(E, cfg.top_k, Ie, cfg.shared_intermediate, self.t["router"],
                                   self.aff["exp_gate"].desc, self.aff["exp_up"].desc,
                                   self.aff["exp_down"].desc, self.aff["sh_gate"].desc,
                                   self.aff["sh_up"].desc, self.aff["sh_down"].desc,
                                   self.t["sh_gate_inp"], scales_bf16=bf16_stacks)
        g = attn_geom(cfg.n_heads, cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v, cfg.rot_dim,
                      cfg.window, cfg.gated_q, cfg.eps)
        d = L.LayerDesc()
        d.hidden, d.vocab = H, cfg.vocab
        d.intermediate = 0 if cfg.moe else cfg.intermediate
        d.eps = cfg.eps
        d.attn = g
        d.enorm, d.hnorm = _p(self.t["enorm"]), _p(self.t["hnorm"])
        d.eh_proj = self.aff["eh_proj"].desc
        d.attn_norm = _p(self.t["attn_norm"])
        d.wq, d.wk, d.wv, d.wo = (self.aff[n].desc for n in ("wq", "wk", "wv", "wo"))
        d.q_norm = _p(self.t.get("q_norm"))
        d.k_norm = _p(self.t.get("k_norm"))
        d.sinks = _p(self.t.get("sinks"))
        d.post_norm = _p(self.t["post_norm"])
        if not cfg.moe:
            d.ffn_gate, d.ffn_up, d.ffn_down = (self.aff[n].desc for n in ("ffn_gate", "ffn_up", "ffn_down"))
        d.moe = C.pointer(self.moe) if self.moe is not None else None
        d.final_norm = _p(self.t["final_norm"])
        d.lm_head = shared.lm_head.desc
        d.embed = _p(shared.embed)
        d.rope = _p(self.rope)
        d.k_cache, d.v_cache = _p(self.k_cache), _p(self.v_cache)
        d.cache_cap = self.cache_cap
        self.desc = d
        self.ws = workspace(L.load().mtp_draft_workspace_bytes(C.byref(d), self.m_max))

    def forward(self, hidden, cache_len, tokens=None, embed_rows=None, token=None, value=None,
                hidden_out=None, u2=None, logits=None, stream=None, pos_base=0):
        """Enqueues one draft step; outputs are written into the given device tensors."""
        from .api import mtp_draft_forward
        si = L.StepIn(_p(tokens), _p(embed_rows), _p(hidden), int(cache_len), int(hidden.shape[0]),
                      int(pos_base))
        so = L.StepOut(_p(token), _p(value), _p(hidden_out), _p(u2), _p(logits))
        mtp_draft_forward(self.desc, si, so, self.ws, stream)


    def catch_up(self, target, seq, cache_len, tokens=None, embed_rows=None, pending=None,
                 pos_base=0, stream=None):
        """Enqueues the K/V catch-up of a target batch of ``seq`` rows."""
        from .api import mtp_kv_catch_up
        need = L.load().mtp_kv_catch_up_workspace_bytes(C.byref(self.desc), int(seq))
        if getattr(self, "catch_ws", None) is None or self.catch_ws.numel() < need:
            self.catch_ws = workspace(need)
        mtp_kv_catch_up(self.desc, tokens, embed_rows, target, pending, seq, cache_len, pos_base,
                        self.catch_ws, stream)


class DraftChain:
    """Layers sharing lm_head and embedding, drafted by ``mtp_draft_chain``."""

    def __init__(self, layers: list[DraftLayer]):
        self.layers = layers
        self.ws = max((lyr.ws for lyr in layers), key=lambda t: t.numel())

    def forward(self, hidden, seq, cache_lens, values, hidden_out=None, stream=None, u2=None,
                logits=None):
        from .api import mtp_draft_chain
        mtp_draft_chain([lyr.desc for lyr in self.layers], hidden, seq, cache_lens,
                        int(hidden.shape[0]), values, hidden_out, self.ws, stream, u2=u2,
                        logits=logits)
