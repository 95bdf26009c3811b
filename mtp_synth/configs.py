"""Shapes of the draft-layer workloads and their seeded inputs.

Five workloads: a tiny dense layer, a Qwen-style dense layer with a
sigmoid-gated query projection, a MiMo-style three-layer chain with
sliding-window attention and per-head sinks, a sweep of bare quantised
matmuls, and a MoE layer.  ``scaled`` builds a smaller layer with the same
structure for tests that must run the oracle in seconds.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class LayerConfig:
    name: str
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    intermediate: int
    vocab: int
    cache_len: int
    m: int = 1
    rope_theta: float = 1e6
    gated_q: bool = False
    qk_norm: bool = True
    window: int = 0              # <= 0: full causal attention
    sinks: bool = False
    n_layers: int = 1            # > 1: chained draft layers sharing embedding and lm_head
    n_experts: int = 0           # > 0: MoE FFN
    top_k: int = 0
    expert_intermediate: int = 0
    shared_intermediate: int = 0
    eps: float = 1e-6
    seed: int = 1000

    @property
    def moe(self) -> bool:
        return self.n_experts > 0

    @property
    def q_rows(self) -> int:
        return self.n_heads * self.head_dim_qk * (2 if self.gated_q else 1)

    @property
    def rot_dim(self) -> int:
        return self.head_dim_qk

    @property
    def cache_cap(self) -> int:
        return self.cache_len + self.m

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class SweepConfig:
    name: str
    ms: tuple
    shapes: tuple   # (N, K)
    seed: int = 1003


CONFIGS = {
    "tiny_dense": LayerConfig(
        name="tiny_dense", hidden=256, n_heads=4, n_kv_heads=2, head_dim_qk=64, head_dim_v=64,
        intermediate=512, vocab=4096, cache_len=64, rope_theta=1e6, seed=1000),
    "qwen_dense": LayerConfig(
        name="qwen_dense", hidden=5120, n_heads=40, n_kv_heads=8, head_dim_qk=128, head_dim_v=128,
        intermediate=17408, vocab=151936, cache_len=4096, gated_q=True, rope_theta=1e6, seed=1001),
    "mimo_chain": LayerConfig(
        name="mimo_chain", hidden=4096, n_heads=32, n_kv_heads=8, head_dim_qk=192, head_dim_v=128,
        intermediate=16384, vocab=152576, cache_len=320, m=4, rope_theta=1e4, qk_norm=False,
        window=128, sinks=True, n_layers=3, seed=1002),
    "qmatmul_sweep": SweepConfig(
        name="qmatmul_sweep", ms=(1, 2, 4, 8, 16),
        shapes=((5120, 5120), (17408, 5120), (5120, 17408), (151936, 5120)), seed=1003),
    "moe": LayerConfig(
        name="moe", hidden=2048, n_heads=16, n_kv_heads=2, head_dim_qk=256, head_dim_v=256,
        intermediate=0, vocab=151936, cache_len=2048, rope_theta=1e6, n_experts=256, top_k=8,
        expert_intermediate=512, shared_intermediate=512, seed=1004),
}


def layer_config(name: str) -> LayerConfig:
    return CONFIGS[name]


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    """A smaller layer with the structure of ``cfg`` (used where the oracle must finish in seconds)."""
    return cfg.with_(**kw)


def layer_prefix(cfg: LayerConfig, layer: int) -> str:
    return f"{cfg.name}.L{layer}."


def make_layer_weights(cfg: LayerConfig, layer: int = 0) -> dict:
    """All weights of draft layer ``layer`` (lm_head and embedding are separate, shared)."""
    from . import affine4_weight, norm_weight, normal_f32

    s = cfg.seed
    p = layer_prefix(cfg, layer)
    H = cfg.hidden
    w = {
        "enorm": norm_weight(s, p + "enorm", H),
        "hnorm": norm_weight(s, p + "hnorm", H),
        "eh_proj": affine4_weight(s, p + "eh_proj", H, 2 * H),
        "attn_norm": norm_weight(s, p + "attn_norm", H),
        "wq": affine4_weight(s, p + "wq", cfg.q_rows, H),
        "wk": affine4_weight(s, p + "wk", cfg.n_kv_heads * cfg.head_dim_qk, H),
        "wv": affine4_weight(s, p + "wv", cfg.n_kv_heads * cfg.head_dim_v, H),
        "wo": affine4_weight(s, p + "wo", H, cfg.n_heads * cfg.head_dim_v),
        "post_norm": norm_weight(s, p + "post_norm", H),
        "final_norm": norm_weight(s, p + "final_norm", H),
    }
    if cfg.qk_norm:
        w["q_norm"] = norm_weight(s, p + "q_norm", cfg.head_dim_qk)
        w["k_norm"] = norm_weight(s, p + "k_norm", cfg.head_dim_qk)
    if cfg.sinks:
        w["sinks"] = normal_f32(s, p + "sinks", (cfg.n_heads,))
    if cfg.moe:
        E, Ie, Is = cfg.n_experts, cfg.expert_intermediate, cfg.shared_intermediate
        w["router"] = normal_f32(s, p + "router", (E, H), 0.0, 0.02)
        for name, (n, k) in (("exp_gate", (Ie, H)), ("exp_up", (Ie, H)), ("exp_down", (H, Ie))):
            q, sc, b = affine4_weight(s, p + name, E * n, k)
            w[name] = (q.reshape(E, n, k // 8), sc.reshape(E, n, k // 32), b.reshape(E, n, k // 32))
        w["sh_gate"] = affine4_weight(s, p + "sh_gate", Is, H)
        w["sh_up"] = affine4_weight(s, p + "sh_up", Is, H)
        w["sh_down"] = affine4_weight(s, p + "sh_down", H, Is)
        w["sh_gate_inp"] = normal_f32(s, p + "sh_gate_inp", (H,), 0.0, 0.02)
    else:
        I = cfg.intermediate
        w["ffn_gate"] = affine4_weight(s, p + "ffn_gate", I, H)
        w["ffn_up"] = affine4_weight(s, p + "ffn_up", I, H)
        w["ffn_down"] = affine4_weight(s, p + "ffn_down", H, I)
    return w


def make_shared(cfg: LayerConfig, embed_rows=None) -> dict:
    """lm_head (affine [V, H]) and the float32 embedding table (or only ``embed_rows`` of it)."""
    from . import affine4_weight, embedding_rows

    s = cfg.seed
    out = {"lm_head": affine4_weight(s, cfg.name + ".lm_head", cfg.vocab, cfg.hidden)}
    if embed_rows is None:
        out["embed"] = embedding_rows(s, cfg.name + ".embed", cfg.vocab, cfg.hidden)
    else:
        out["embed_rows"] = embedding_rows(s, cfg.name + ".embed", cfg.vocab, cfg.hidden, embed_rows)
    return out


def make_state(cfg: LayerConfig, layer: int = 0) -> dict:
    """KV cache of one layer: ``[n_kv, cap, d]`` with the first ``cache_len`` rows filled."""
    from . import normal

    s = cfg.seed
    p = layer_prefix(cfg, layer)
    L, cap = cfg.cache_len, cfg.cache_cap
    kc = np.zeros((cfg.n_kv_heads, cap, cfg.head_dim_qk), dtype=np.float32)
    vc = np.zeros((cfg.n_kv_heads, cap, cfg.head_dim_v), dtype=np.float32)
    kc[:, :L] = normal(s, p + "kcache", cfg.n_kv_heads * L * cfg.head_dim_qk).reshape(
        cfg.n_kv_heads, L, cfg.head_dim_qk)
    vc[:, :L] = normal(s, p + "vcache", cfg.n_kv_heads * L * cfg.head_dim_v).reshape(
        cfg.n_kv_heads, L, cfg.head_dim_v)
    return {"k_cache": kc, "v_cache": vc}


def make_step(cfg: LayerConfig) -> dict:
    """Step inputs: target hiddens ``[m, H]`` and the token sequence.

    For a single layer the ``m`` tokens are the rows' tokens.  For a chain of
    ``n_layers`` layers, ``tokens`` holds the ``m`` known tokens
    ``x_{t-m+2} .. x_{t+1}``; layer ``k`` row ``i`` embeds element ``i + k``
    of ``tokens`` followed by the drafts of the earlier layers.
    """
    from . import normal_f32, tokens

    s = cfg.seed
    return {
        "hidden": normal_f32(s, cfg.name + ".hidden", (cfg.m, cfg.hidden)),
        "tokens": tokens(s, cfg.name + ".tokens", cfg.m, cfg.vocab),
    }
