"""ctypes view of ``include/mtpdraft.h`` (argument marshalling only).

Loads the in-tree ``libmtpdraft.so``; importing this module on a machine
where the library has not been built raises, so no caller can silently fall
back to anything else.
"""

from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmtpdraft.so")

MTP_OK = 0
STATUS_NAMES = {
    0: "MTP_OK", 1: "MTP_ERR_INVALID_ARG", 2: "MTP_ERR_UNSUPPORTED", 3: "MTP_ERR_CAPACITY",
    4: "MTP_ERR_WORKSPACE", 5: "MTP_ERR_CUDA", 6: "MTP_ERR_DEVICE_TIMEOUT",
}

vp = C.c_void_p
i32 = C.c_int32
f32 = C.c_float
sz = C.c_size_t


class Affine4(C.Structure):
    _fields_ = [("q", vp), ("s", vp), ("b", vp), ("n", i32), ("k", i32)]


class AttnGeom(C.Structure):
    _fields_ = [("n_heads", i32), ("n_kv_heads", i32), ("head_dim_qk", i32), ("head_dim_v", i32),
                ("rot_dim", i32), ("window", i32), ("gated_q", i32), ("eps", f32), ("scale", f32)]


class MoeWeights(C.Structure):
    _fields_ = [("n_experts", i32), ("top_k", i32), ("expert_inter", i32), ("shared_inter", i32),
                ("router", vp), ("exp_gate", Affine4), ("exp_up", Affine4), ("exp_down", Affine4),
                ("sh_gate", Affine4), ("sh_up", Affine4), ("sh_down", Affine4),
                ("sh_gate_inp", vp), ("scales_bf16", i32)]


class LayerDesc(C.Structure):
    _fields_ = [("hidden", i32), ("vocab", i32), ("intermediate", i32), ("eps", f32),
                ("attn", AttnGeom),
                ("enorm", vp), ("hnorm", vp), ("eh_proj", Affine4), ("attn_norm", vp),
                ("wq", Affine4), ("wk", Affine4), ("wv", Affine4), ("wo", Affine4),
                ("q_norm", vp), ("k_norm", vp), ("sinks", vp), ("post_norm", vp),
                ("ffn_gate", Affine4), ("ffn_up", Affine4), ("ffn_down", Affine4),
                ("moe", C.POINTER(MoeWeights)), ("final_norm", vp), ("lm_head", Affine4),
                ("embed", vp), ("rope", vp), ("k_cache", vp), ("v_cache", vp),
                ("cache_cap", i32)]


class StepIn(C.Structure):
    _fields_ = [("d_tokens", vp), ("d_embed_rows", vp), ("d_hidden", vp), ("cache_len", i32),
                ("m", i32), ("pos_base", i32)]


class MimoLayerState(C.Structure):
    _fields_ = [("committed", i32), ("base", i32), ("kv_len", i32)]


SPEC_MAX_DEPTH = 16


class SpecStats(C.Structure):
    _fields_ = [("rounds", C.c_uint64), ("drafted", C.c_uint64), ("accepted", C.c_uint64),
                ("accept_hist", C.c_uint64 * (SPEC_MAX_DEPTH + 1)),
                ("depth_drafted", C.c_uint64 * SPEC_MAX_DEPTH),
                ("depth_accepted", C.c_uint64 * SPEC_MAX_DEPTH),
                ("draft_ns", C.c_uint64), ("verify_ns", C.c_uint64)]


class StepOut(C.Structure):
    _fields_ = [("d_token", vp), ("d_value", vp), ("d_hidden_out", vp), ("d_u2", vp),
                ("d_logits", vp)]


EXPORTS = {
    # name: (restype, argtypes)
    "mtp_last_error": (C.c_char_p, []),
    "mtp_version": (C.c_int, []),
    "mtp_workspace_init": (C.c_int, [vp, sz, vp]),
    "mtp_workspace_status": (C.c_int, [vp, C.POINTER(i32), vp]),
    "mtp_workspace_set_wait_limit": (C.c_int, [vp, i32, vp]),
    "mtp_timing_begin": (C.c_int, [C.POINTER(vp), i32]),
    "mtp_timing_end": (C.c_int, [C.POINTER(i32)]),
    "qmatmul_affine4_workspace_bytes": (sz, [i32, i32]),
    "qmatmul_affine4": (C.c_int, [vp, C.POINTER(Affine4), vp, i32, vp, sz, vp]),
    "rmsnorm_residual": (C.c_int, [vp, vp, vp, vp, vp, i32, i32, f32, vp]),
    "mtp_rope_table": (C.c_int, [vp, i32, i32, C.c_double, vp]),
    "attn_decode_sink_workspace_bytes": (sz, [C.POINTER(AttnGeom), i32, i32]),
    "attn_decode_sink": (C.c_int, [C.POINTER(AttnGeom), vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                   i32, i32, vp, vp, sz, vp]),
    "attn_decode_sink_noalloc": (C.c_int, [C.POINTER(AttnGeom), vp, vp, vp, vp, vp, vp, vp, vp,
                                           vp, i32, i32, i32, vp, vp]),
    "lmhead_argmax_workspace_bytes": (sz, [i32, i32]),
    "lmhead_argmax": (C.c_int, [vp, vp, f32, C.POINTER(Affine4), vp, vp, vp, vp, vp, sz, vp]),
    "verify_head_workspace_bytes": (sz, [i32, i32, i32]),
    "mtp_spec_accept": (i32, [C.POINTER(i32), C.POINTER(i32), i32]),
    "mtp_spec_note_round": (C.c_int, [C.POINTER(SpecStats), i32, i32, C.c_uint64, C.c_uint64]),
    "mtp_spec_tokens_per_round": (C.c_double, [C.POINTER(SpecStats)]),
    "mtp_spec_rewind": (C.c_int, [C.POINTER(i32), i32, i32]),
    "verify_head_argmax": (C.c_int, [vp, i32, vp, f32, C.POINTER(Affine4), f32, f32, vp, vp, vp,
                                     vp, sz, vp]),
    "moe_ffn_workspace_bytes": (sz, [C.POINTER(MoeWeights), i32]),
    "moe_ffn": (C.c_int, [C.POINTER(MoeWeights), vp, vp, f32, i32, vp, vp, vp, vp, sz, vp]),
    "mtp_draft_workspace_bytes": (sz, [C.POINTER(LayerDesc), i32]),
    "mtp_draft_forward": (C.c_int, [C.POINTER(LayerDesc), C.POINTER(StepIn), C.POINTER(StepOut),
                                    vp, sz, vp]),
    "mtp_draft_chain": (C.c_int, [C.POINTER(LayerDesc), i32, vp, vp, C.POINTER(i32), i32, vp, vp,
                                  vp, vp, vp, sz, vp]),
    "mtp_draft_steps": (C.c_int, [C.POINTER(LayerDesc), i32, vp, vp, i32, i32, vp, vp, vp, sz, vp]),
    "mtp_mimo_plan_layer": (i32, [C.POINTER(MimoLayerState), i32, i32, i32, i32, i32, C.POINTER(i32)]),
    "mtp_mimo_commit_layer": (C.c_int, [C.POINTER(MimoLayerState), i32, i32, i32]),
    "mtp_mimo_draft_round": (C.c_int, [C.POINTER(LayerDesc), i32, C.POINTER(MimoLayerState), vp, i32,
                                       i32, i32, vp, i32, vp, vp, sz, vp, sz, vp, C.POINTER(i32)]),
    "mtp_kv_catch_up_workspace_bytes": (sz, [C.POINTER(LayerDesc), i32]),
    "mtp_kv_catch_up": (C.c_int, [C.POINTER(LayerDesc), vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]),
}


def header_symbols():
    """Function names declared in ``include/mtpdraft.h``."""
    import re
    path = os.path.join(HERE, "..", "include", "mtpdraft.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    skip = {"sizeof", "defined", "if"}
    return sorted({n for n in names if n not in skip})


_lib = None


def load():
    """Loads the library and binds every exported function (raises when it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "mtp_speculative_draft_gb300.build.build() (nvcc, sm_103a)")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MtpError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().mtp_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def check(status: int, where: str):
    if status != MTP_OK:
        raise MtpError(status, where)
