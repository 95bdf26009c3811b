"""Thin torch-facing wrappers with the C ABI's names (argument marshalling only)."""

from __future__ import annotations

import ctypes as C

import torch

from . import _lib as L
from ._lib import Affine4, AttnGeom, MimoLayerState, MoeWeights, SpecStats, check


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors are required")
    if not t.is_contiguous():
        raise ValueError("contiguous tensors are required")
    return t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def affine4(q: torch.Tensor, s: torch.Tensor, b: torch.Tensor, n: int | None = None,
            k: int | None = None) -> Affine4:
    """Descriptor of an affine 4-bit weight held in device tensors ``q [n, k/8]``, ``s``/``b [n, k/32]``."""
    if q.dtype not in (torch.int32, torch.uint32) or s.dtype != torch.float32 or b.dtype != torch.float32:
        raise TypeError("codes must be int32/uint32, scales and biases float32")
    n = q.shape[0] if n is None else n
    k = q.shape[-1] * 8 if k is None else k
    return Affine4(_p(q), _p(s), _p(b), int(n), int(k))


def attn_geom(n_heads, n_kv_heads, head_dim_qk, head_dim_v, rot_dim=None, window=0, gated_q=False,
              eps=1e-6, scale=0.0) -> AttnGeom:
    return AttnGeom(n_heads, n_kv_heads, head_dim_qk, head_dim_v,
                    head_dim_qk if rot_dim is None else rot_dim, window, int(bool(gated_q)),
                    eps, scale)


def moe_weights(n_experts, top_k, expert_inter, shared_inter, router, exp_gate, exp_up, exp_down,
                sh_gate, sh_up, sh_down, sh_gate_inp, scales_bf16=False) -> MoeWeights:
    return MoeWeights(n_experts, top_k, expert_inter, shared_inter, _p(router), exp_gate, exp_up,
                      exp_down, sh_gate, sh_up, sh_down, _p(sh_gate_inp), int(bool(scales_bf16)))


def affine4_bf16_scales(q: torch.Tensor, s: torch.Tensor, b: torch.Tensor) -> Affine4:
    """Descriptor of an expert stack with bfloat16 scales and biases (``s``/``b``
    bfloat16 device tensors ``[n, k/32]``); only MoE stacks take it."""
    if q.dtype not in (torch.int32, torch.uint32) or s.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("codes must be int32/uint32, scales and biases bfloat16")
    return Affine4(_p(q), _p(s), _p(b), int(q.shape[0]), int(q.shape[-1] * 8))


def workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A cleared workspace of ``nbytes`` bytes (uint8 device tensor)."""
    ws = torch.empty(max(int(nbytes), 1024), dtype=torch.uint8, device=device)
    mtp_workspace_init(ws, stream)
    return ws


def mtp_workspace_init(ws: torch.Tensor, stream=None):
    check(L.load().mtp_workspace_init(_p(ws), ws.numel(), _stream(stream)), "mtp_workspace_init")


def mtp_workspace_status(ws: torch.Tensor, stream=None) -> int:
    code = C.c_int32(0)
    check(L.load().mtp_workspace_status(_p(ws), C.byref(code), _stream(stream)),
          "mtp_workspace_status")
    return code.value


class launch_timing:
    """Context manager around mtp_timing_begin / mtp_timing_end: ``events`` are
    torch.cuda.Event(enable_timing=True) objects; after the block,
    ``durations_ms()`` gives each launch's time (events i -> i + 1)."""

    def __init__(self, events):
        self.events = events
        self._handles = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
        self.n = 0

    def __enter__(self):
        check(L.load().mtp_timing_begin(self._handles, len(self.events)), "mtp_timing_begin")
        return self

    def __exit__(self, *exc):
        n = C.c_int32(0)
        st = L.load().mtp_timing_end(C.byref(n))
        self.n = n.value
        if exc[0] is None:
            check(st, "mtp_timing_end")
        return False

    def durations_ms(self):
        self.events[self.n - 1].synchronize()
        return [self.events[i].elapsed_time(self.events[i + 1]) for i in range(self.n - 1)]


def mtp_workspace_set_wait_limit(ws: torch.Tensor, polls: int, stream=None):
    check(L.load().mtp_workspace_set_wait_limit(_p(ws), int(polls), _stream(stream)),
          "mtp_workspace_set_wait_limit")


def mtp_rope_table(table: torch.Tensor, max_pos: int, rot_dim: int, theta: float, stream=None):
    check(L.load().mtp_rope_table(_p(table), max_pos, rot_dim, float(theta), _stream(stream)),
          "mtp_rope_table")


def qmatmul_affine4(x, w: Affine4, y, m: int, ws=None, stream=None):
    lib = L.load()
    if ws is None:
        ws = workspace(lib.qmatmul_affine4_workspace_bytes(m, w.k), stream=stream)
    check(lib.qmatmul_affine4(_p(x), C.byref(w), _p(y), m, _p(ws), ws.numel(), _stream(stream)),
          "qmatmul_affine4")
    return ws


def rmsnorm_residual(a, delta, w, out_norm, out_sum, rows, dim, eps, stream=None):
    check(L.load().rmsnorm_residual(_p(a), _p(delta), _p(w), _p(out_norm), _p(out_sum), rows, dim,
                                    eps, _stream(stream)), "rmsnorm_residual")


def attn_decode_sink(g: AttnGeom, qp, kp, vp, q_norm, k_norm, rope, sinks, k_cache, v_cache,
                     cache_len, cache_cap, m, out, ws=None, stream=None):
    lib = L.load()
    if ws is None:
        ws = workspace(lib.attn_decode_sink_workspace_bytes(C.byref(g), m, cache_len), stream=stream)
    check(lib.attn_decode_sink(C.byref(g), _p(qp), _p(kp), _p(vp), _p(q_norm), _p(k_norm),
                               _p(rope), _p(sinks), _p(k_cache), _p(v_cache), cache_len, cache_cap,
                               m, _p(out), _p(ws), ws.numel(), _stream(stream)),
          "attn_decode_sink")
    return ws


def attn_decode_sink_noalloc(g: AttnGeom, qp, kp, vp, q_norm, k_norm, rope, sinks, k_cache,
                             v_cache, cache_len, cache_cap, m, out, stream=None):
    """attn_decode_sink on the library's static device scratch (no workspace argument)."""
    check(L.load().attn_decode_sink_noalloc(C.byref(g), _p(qp), _p(kp), _p(vp), _p(q_norm),
                                            _p(k_norm), _p(rope), _p(sinks), _p(k_cache),
                                            _p(v_cache), cache_len, cache_cap, m, _p(out),
                                            _stream(stream)),
          "attn_decode_sink_noalloc")


def lmhead_argmax(y, norm_w, eps, w: Affine4, token, value, logits=None, y_normed=None, ws=None,
                  stream=None):
    lib = L.load()
    if ws is None:
        ws = workspace(lib.lmhead_argmax_workspace_bytes(w.k, w.n), stream=stream)
    check(lib.lmhead_argmax(_p(y), _p(norm_w), eps, C.byref(w), _p(token), _p(value), _p(logits),
                            _p(y_normed), _p(ws), ws.numel(), _stream(stream)), "lmhead_argmax")
    return ws


def verify_head_argmax(h, rows, norm_w, eps, w: Affine4, logit_multiplier, softcap, tokens,
                       values, logits=None, ws=None, stream=None):
    lib = L.load()
    if ws is None:
        ws = workspace(lib.verify_head_workspace_bytes(rows, w.k, w.n), stream=stream)
    check(lib.verify_head_argmax(_p(h), rows, _p(norm_w), eps, C.byref(w), logit_multiplier,
                                 softcap, _p(tokens), _p(values), _p(logits), _p(ws), ws.numel(),
                                 _stream(stream)), "verify_head_argmax")
    return ws


def moe_ffn(w: MoeWeights, u1, post_norm, eps, hidden, u2, sel=None, weight=None, ws=None,
            stream=None):
    lib = L.load()
    if ws is None:
        ws = workspace(lib.moe_ffn_workspace_bytes(C.byref(w), hidden), stream=stream)
    check(lib.moe_ffn(C.byref(w), _p(u1), _p(post_norm), eps, hidden, _p(u2), _p(sel), _p(weight),
                      _p(ws), ws.numel(), _stream(stream)), "moe_ffn")
    return ws


def mtp_draft_forward(desc, step_in, step_out, ws, stream=None):
    check(L.load().mtp_draft_forward(C.byref(desc), C.byref(step_in), C.byref(step_out), _p(ws),
                                     ws.numel(), _stream(stream)), "mtp_draft_forward")


def mtp_draft_chain(descs, hidden, seq, cache_lens, m, values, hidden_out, ws, stream=None,
                    u2=None, logits=None):
    arr = (L.LayerDesc * len(descs))(*descs)
    lens = (C.c_int32 * len(descs))(*cache_lens)
    check(L.load().mtp_draft_chain(arr, len(descs), _p(hidden), _p(seq), lens, m, _p(values),
                                   _p(hidden_out), _p(u2), _p(logits), _p(ws), ws.numel(),
                                   _stream(stream)),
          "mtp_draft_chain")


def mtp_kv_catch_up(desc, tokens, embed_rows, target, pending, seq, cache_len, pos_base=0, ws=None,
                    stream=None):
    lib = L.load()
    if ws is None:
        ws = workspace(lib.mtp_kv_catch_up_workspace_bytes(C.byref(desc), seq), stream=stream)
    check(lib.mtp_kv_catch_up(C.byref(desc), _p(tokens), _p(embed_rows), _p(target), _p(pending),
                              int(seq), int(cache_len), int(pos_base), _p(ws), ws.numel(),
                              _stream(stream)), "mtp_kv_catch_up")
    return ws


def mtp_draft_steps(desc, k_steps, hidden, tokens, cache_len, values, hidden_out, ws, pos_base=0,
                    stream=None):
    check(L.load().mtp_draft_steps(C.byref(desc), int(k_steps), _p(hidden), _p(tokens),
                                   int(cache_len), int(pos_base), _p(values), _p(hidden_out),
                                   _p(ws), ws.numel(), _stream(stream)), "mtp_draft_steps")


def mtp_mimo_draft_round(descs, states, hist, hist_lo, hist_end, t, ids, ids_len, values, ws,
                         catch_ws, stream=None) -> int:
    """The device half of a MiMo round; ``states`` is a ctypes array of
    MimoLayerState updated in place; returns the number of drafts."""
    arr = (L.LayerDesc * len(descs))(*descs)
    n = C.c_int32(0)
    check(L.load().mtp_mimo_draft_round(arr, len(descs), states, _p(hist), int(hist_lo),
                                        int(hist_end), int(t), _p(ids), int(ids_len), _p(values),
                                        _p(ws), ws.numel(), _p(catch_ws),
                                        0 if catch_ws is None else catch_ws.numel(),
                                        _stream(stream), C.byref(n)), "mtp_mimo_draft_round")
    return n.value


# ------------------------------------------------------------- speculation bookkeeping (host)
def _i32_array(values):
    vals = [int(v) for v in values]
    return (C.c_int32 * max(1, len(vals)))(*vals), len(vals)


def mtp_spec_accept(drafts, verify_tokens) -> int:
    """Length of the drafts' prefix that equals the verifier's greedy tokens."""
    d, k = _i32_array(drafts)
    v, n = _i32_array(verify_tokens)
    if n < k:
        raise ValueError("one verifier token per draft is required")
    a = L.load().mtp_spec_accept(d, v, k)
    if a < 0:
        raise ValueError("mtp_spec_accept: k outside 0..16")
    return a


def mtp_spec_note_round(stats: SpecStats, k: int, a: int, draft_ns: int = 0, verify_ns: int = 0):
    check(L.load().mtp_spec_note_round(C.byref(stats), k, a, draft_ns, verify_ns),
          "mtp_spec_note_round")


def mtp_spec_tokens_per_round(stats: SpecStats) -> float:
    return L.load().mtp_spec_tokens_per_round(C.byref(stats))


def mtp_spec_rewind(cache_len, keep: int) -> list:
    """Cache lengths after cutting every one above ``keep`` back to ``keep``."""
    arr, n = _i32_array(cache_len)
    check(L.load().mtp_spec_rewind(arr, n, keep), "mtp_spec_rewind")
    return list(arr[:n])



def mtp_mimo_plan_layer(state: MimoLayerState, layer: int, t: int, hist_lo: int, hist_end: int,
                        ids_len: int):
    """(rows to run, first position) of one layer's part of a MiMo round; updates ``state``."""
    start = C.c_int32(0)
    n = L.load().mtp_mimo_plan_layer(C.byref(state), layer, t, hist_lo, hist_end, ids_len,
                                     C.byref(start))
    if n < 0:
        raise ValueError("mtp_mimo_plan_layer: bad arguments")
    return n, start.value


def mtp_mimo_commit_layer(state: MimoLayerState, layer: int, t: int, ids_len: int):
    check(L.load().mtp_mimo_commit_layer(C.byref(state), layer, t, ids_len), "mtp_mimo_commit_layer")
