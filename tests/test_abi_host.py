"""The C-ABI library builds, loads and exports what its header declares;
host-side validation rejects bad calls before anything reaches a GPU."""

import ctypes as C
import os
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mtp_speculative_draft_gb300 import build, _lib
    build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported_and_bound(lib):
    from mtp_speculative_draft_gb300 import _lib
    declared = set(_lib.header_symbols())
    assert declared, "no declarations parsed from the header"
    assert declared == set(_lib.EXPORTS), declared ^ set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_struct_layouts_match_c(lib):
    from mtp_speculative_draft_gb300 import _lib
    src = r'''
    #include <stdio.h>
    #include <stddef.h>
    #include "mtpdraft.h"
    int main(void) {
      printf("%zu %zu %zu %zu %zu %zu\n", sizeof(mtp_affine4), sizeof(mtp_attn_geom),
             sizeof(mtp_moe_weights), sizeof(mtp_layer_desc), sizeof(mtp_step_in), sizeof(mtp_step_out));
      printf("%zu %zu %zu\n", offsetof(mtp_layer_desc, lm_head), offsetof(mtp_layer_desc, cache_cap),
             offsetof(mtp_moe_weights, sh_gate_inp));
      printf("%zu %zu %zu\n", sizeof(mtp_spec_stats), offsetof(mtp_spec_stats, depth_accepted),
             offsetof(mtp_spec_stats, verify_ns));
      return 0; }
    '''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    got = [int(v) for v in out]
    want = [C.sizeof(_lib.Affine4), C.sizeof(_lib.AttnGeom), C.sizeof(_lib.MoeWeights),
            C.sizeof(_lib.LayerDesc), C.sizeof(_lib.StepIn), C.sizeof(_lib.StepOut),
            _lib.LayerDesc.lm_head.offset, _lib.LayerDesc.cache_cap.offset,
            _lib.MoeWeights.sh_gate_inp.offset,
            C.sizeof(_lib.SpecStats), _lib.SpecStats.depth_accepted.offset,
            _lib.SpecStats.verify_ns.offset]
    assert got == want


def _fake_affine(n, k, base=0x10000):
    from mtp_speculative_draft_gb300 import _lib
    return _lib.Affine4(base, base + 0x100000, base + 0x200000, n, k)


def test_qmatmul_rejects_bad_calls(lib):
    from mtp_speculative_draft_gb300 import _lib
    w = _fake_affine(64, 256)
    x, y, ws = C.c_void_p(0x1000), C.c_void_p(0x2000), C.c_void_p(0x3000)
    assert lib.qmatmul_affine4(None, C.byref(w), y, 1, ws, 1 << 20, None) == 1
    assert lib.qmatmul_affine4(x, C.byref(w), y, 17, ws, 1 << 20, None) == 2
    assert lib.qmatmul_affine4(x, C.byref(w), y, 0, ws, 1 << 20, None) == 2
    bad_k = _fake_affine(64, 100)
    assert lib.qmatmul_affine4(x, C.byref(bad_k), y, 1, ws, 1 << 20, None) == 2
    assert b"multiple of 32" in lib.mtp_last_error()
    mis = _lib.Affine4(0x10004, 0x20000, 0x30000, 64, 256)
    assert lib.qmatmul_affine4(x, C.byref(mis), y, 1, ws, 1 << 20, None) == 1
    assert lib.qmatmul_affine4(x, C.byref(w), y, 1, ws, 16, None) == 4
    need = lib.qmatmul_affine4_workspace_bytes(4, 256)
    assert need >= 1024 + 4 * 256 * 4


def _layer(lib, **over):
    from mtp_speculative_draft_gb300 import _lib
    H, nh, nkv, d, I, V = 256, 4, 2, 64, 512, 4096
    g = _lib.AttnGeom(nh, nkv, d, d, d, 0, 0, 1e-6, 0.0)
    p = 0x100000
    D = _lib.LayerDesc()
    D.hidden, D.vocab, D.intermediate, D.eps, D.attn = H, V, I, 1e-6, g
    for name in ("enorm", "hnorm", "attn_norm", "post_norm", "final_norm", "rope", "k_cache",
                 "v_cache", "embed"):
        setattr(D, name, p)
    D.eh_proj = _fake_affine(H, 2 * H)
    D.wq, D.wk, D.wv = _fake_affine(nh * d, H), _fake_affine(nkv * d, H), _fake_affine(nkv * d, H)
    D.wo = _fake_affine(H, nh * d)
    D.ffn_gate, D.ffn_up, D.ffn_down = _fake_affine(I, H), _fake_affine(I, H), _fake_affine(H, I)
    D.lm_head = _fake_affine(V, H)
    D.cache_cap = 65
    for k, v in over.items():
        setattr(D, k, v)
    return D


def test_forward_rejects_bad_calls(lib):
    from mtp_speculative_draft_gb300 import _lib
    D = _layer(lib)
    si = _lib.StepIn(0x1000, None, 0x2000, 64, 1)
    so = _lib.StepOut(0x3000, 0x4000, None, None, None)
    ws = C.c_void_p(0x5000)
    need = lib.mtp_draft_workspace_bytes(C.byref(D), 1)
    assert need > 1024
    # cache overflow
    si2 = _lib.StepIn(0x1000, None, 0x2000, 65, 1)
    assert lib.mtp_draft_forward(C.byref(D), C.byref(si2), C.byref(so), ws, need, None) == 3
    # workspace too small
    assert lib.mtp_draft_forward(C.byref(D), C.byref(si), C.byref(so), ws, need - 256, None) == 4
    # wrong weight shape
    D2 = _layer(lib, wo=_fake_affine(256, 128))
    assert lib.mtp_draft_forward(C.byref(D2), C.byref(si), C.byref(so), ws, need, None) == 1
    assert b"wo" in lib.mtp_last_error()
    # heads that do not group
    D3 = _layer(lib, attn=_lib.AttnGeom(4, 3, 64, 64, 64, 0, 0, 1e-6, 0.0))
    assert lib.mtp_draft_forward(C.byref(D3), C.byref(si), C.byref(so), ws, need, None) == 1
    # gated q with different value head size
    D4 = _layer(lib, attn=_lib.AttnGeom(4, 2, 64, 32, 64, 0, 1, 1e-6, 0.0))
    assert lib.mtp_draft_forward(C.byref(D4), C.byref(si), C.byref(so), ws, need, None) == 2
    # missing outputs
    so2 = _lib.StepOut(None, 0x4000, None, None, None)
    assert lib.mtp_draft_forward(C.byref(D), C.byref(si), C.byref(so2), ws, need, None) == 1
    # m out of range
    si3 = _lib.StepIn(0x1000, None, 0x2000, 0, 17)
    assert lib.mtp_draft_forward(C.byref(D), C.byref(si3), C.byref(so), ws, need, None) == 2


def test_attention_and_head_reject_bad_calls(lib):
    from mtp_speculative_draft_gb300 import _lib
    g = _lib.AttnGeom(8, 2, 128, 128, 128, 0, 0, 1e-6, 0.0)
    p = C.c_void_p(0x100000)
    args = [p] * 9
    # cache overflow
    assert lib.attn_decode_sink(C.byref(g), *args, 10, 10, 1, p, p, 1 << 20, None) == 3
    # too many query rows per KV head
    assert lib.attn_decode_sink(C.byref(g), *args, 0, 100, 5, p, p, 1 << 20, None) == 2
    w = _fake_affine(1000, 96)
    assert lib.lmhead_argmax(p, None, 1e-6, C.byref(w), p, p, None, None, p, 1 << 20, None) == 2


def test_verify_head_rejects_bad_calls(lib):
    p = C.c_void_p(0x100000)
    w = _fake_affine(1000, 256)
    need = lib.verify_head_workspace_bytes(4, 256, 1000)
    assert need > 4 * 1000 * 4  # holds the logits of every row
    assert lib.verify_head_workspace_bytes(0, 256, 1000) == 0

    def call(h=p, rows=4, mult=1.0, cap=0.0, tokens=p, wt=w, ws_bytes=need):
        return lib.verify_head_argmax(h, rows, None, 1e-6, C.byref(wt), mult, cap, tokens, p, None,
                                      p, ws_bytes, None)

    assert call(h=None) == 1                       # null input
    assert call(tokens=None) == 1                  # null output
    assert call(rows=0) == 2 and call(rows=17) == 2  # rows outside 1..16
    assert call(mult=float("nan")) == 1            # multiplier must be finite
    assert call(cap=float("inf")) == 1             # softcap must be finite
    assert call(wt=_fake_affine(1000, 96)) == 2    # K % 128 != 0
    assert call(ws_bytes=need - 256) == 4          # workspace too small
    assert b"workspace" in lib.mtp_last_error()


def test_noalloc_attention_rejects_before_touching_its_scratch(lib):
    # Every argument is checked before the static scratch is looked up or
    # cleared: without a GPU an invalid call still returns its own code (a
    # CUDA call would have failed with MTP_ERR_CUDA = 5 instead).
    from mtp_speculative_draft_gb300 import _lib
    g = _lib.AttnGeom(8, 2, 128, 128, 128, 0, 0, 1e-6, 0.0)
    p = C.c_void_p(0x100000)
    full = [p] * 9
    assert lib.attn_decode_sink_noalloc(C.byref(g), None, *full[1:], 0, 10, 1, p, None) == 1
    odd = [p] * 7 + [C.c_void_p(0x100004), p]      # misaligned K cache
    assert lib.attn_decode_sink_noalloc(C.byref(g), *odd, 0, 10, 1, p, None) == 1
    assert lib.attn_decode_sink_noalloc(C.byref(g), *full, 10, 10, 1, p, None) == 3
    assert lib.attn_decode_sink_noalloc(C.byref(g), *full, 0, 10, 1, None, None) == 1
    # a geometry whose scratch exceeds the static array is refused too
    # (one KV head of 16 query heads, 256-dim heads, 4096 cached rows: about
    # 148 splits x 16 rows x 258 floats of partials)
    big = _lib.AttnGeom(16, 1, 256, 256, 256, 0, 0, 1e-6, 0.0)
    assert lib.attn_decode_sink_workspace_bytes(C.byref(big), 1, 4096) > 2 << 20
    assert lib.attn_decode_sink_noalloc(C.byref(big), *full, 4096, 4104, 1, p, None) == 4


def test_timing_session_host_rules(lib):
    # sessions need two or more events, do not nest, and count marks; with no
    # launch in between nothing is recorded (no CUDA call is made here)
    evs = (C.c_void_p * 4)(0x10, 0x20, 0x30, 0x40)
    n = C.c_int32(-1)
    assert lib.mtp_timing_begin(None, 4) == 1
    assert lib.mtp_timing_begin(evs, 1) == 1
    assert lib.mtp_timing_end(C.byref(n)) == 1            # no session open
    assert lib.mtp_timing_begin(evs, 4) == 0
    assert lib.mtp_timing_begin(evs, 4) == 1              # already open
    assert lib.mtp_timing_end(C.byref(n)) == 0 and n.value == 0
    # a rejected call launches nothing, so it makes no mark either
    assert lib.mtp_timing_begin(evs, 4) == 0
    w = _fake_affine(64, 100)
    p = C.c_void_p(0x1000)
    assert lib.qmatmul_affine4(p, C.byref(w), p, 1, p, 1 << 20, None) == 2
    assert lib.mtp_timing_end(C.byref(n)) == 0 and n.value == 0
    assert lib.mtp_workspace_set_wait_limit(None, 1, None) == 1
    assert lib.mtp_workspace_set_wait_limit(p, -1, None) == 1
