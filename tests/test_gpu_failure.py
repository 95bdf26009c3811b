"""Device-side failure paths: every one ends in an error status that the host
reads from the workspace, never in a fault or a hang.

* an out-of-range token id sets code 2 and the step uses row 0;
* with a one-poll limit (mtp_workspace_set_wait_limit) the cross-CTA waits
  that are not already satisfied give up: code 3 for the waits between the
  projections of a one-row launch, code 4 for the attention splits waiting
  for each other.  The launch then finishes part-way; mtp_workspace_init
  clears the workspace and the next step is correct again.
"""

import numpy as np
import pytest

from helpers import assert_close, assert_token
from oracle import mtp_oracle as O
from mtp_synth.configs import CONFIGS, make_layer_weights, make_shared, make_state, make_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    from mtp_speculative_draft_gb300 import build
    build.build()
    torch.cuda.init()
    return torch.device("cuda:0")


def _t(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


SMALL = CONFIGS["qwen_dense"].with_(name="qwen_small", hidden=512, n_heads=8, n_kv_heads=2,
                                    intermediate=1024 + 128, vocab=6000, cache_len=300)


def _layer(cfg, dev):
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    w, shared, st, step = make_layer_weights(cfg), make_shared(cfg), make_state(cfg), make_step(cfg)
    return DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev), (w, shared, st, step)


def _step(lyr, cfg, dev, tokens, hidden):
    import torch
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    u2 = torch.zeros((cfg.m, cfg.hidden), dtype=torch.float32, device=dev)
    logits = torch.zeros(cfg.vocab, dtype=torch.float32, device=dev)
    lyr.forward(_t(hidden, dev), cfg.cache_len, tokens=_t(tokens, dev), token=tok, value=val,
                u2=u2, logits=logits)
    torch.cuda.synchronize()
    return int(tok.item()), u2.cpu().numpy(), logits.cpu().numpy()


def test_out_of_range_token_sets_code_2(dev):
    from mtp_speculative_draft_gb300 import mtp_workspace_init, mtp_workspace_status
    cfg = SMALL
    lyr, (w, shared, st, step) = _layer(cfg, dev)
    bad = np.array([cfg.vocab + 3], dtype=np.int32)
    _, u2_bad, _ = _step(lyr, cfg, dev, bad, step["hidden"])
    assert mtp_workspace_status(lyr.ws) == 2
    # row 0 was used, and the workspace stays usable (code 2 needs no re-init)
    _, u2_zero, _ = _step(lyr, cfg, dev, np.array([0], dtype=np.int32), step["hidden"])
    assert np.array_equal(u2_bad, u2_zero)
    mtp_workspace_init(lyr.ws)
    assert mtp_workspace_status(lyr.ws) == 0


def test_phase_wait_gives_up_then_reinit(dev):
    from mtp_speculative_draft_gb300 import (mtp_workspace_init, mtp_workspace_set_wait_limit,
                                             mtp_workspace_status)
    cfg = SMALL
    lyr, (w, shared, st, step) = _layer(cfg, dev)
    mtp_workspace_set_wait_limit(lyr.ws, 1)
    _step(lyr, cfg, dev, step["tokens"], step["hidden"])
    # warps with no pre-unit poll the pre-unit count once, before it is complete
    assert mtp_workspace_status(lyr.ws) == 3
    mtp_workspace_init(lyr.ws)                     # also restores the default limit
    tok, u2, logits = _step(lyr, cfg, dev, step["tokens"], step["hidden"])
    assert mtp_workspace_status(lyr.ws) == 0
    e = shared["embed"][step["tokens"]]
    ref = O.draft_layer(cfg, w, shared["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    assert_close(u2, ref["u2"], "u2 after re-init")
    assert_close(logits, ref["logits"], "logits after re-init")
    assert_token(tok, ref["token"], ref["margin"], "token after re-init")


def test_attention_split_wait_gives_up_then_reinit(dev):
    import torch
    from mtp_speculative_draft_gb300 import (attn_decode_sink, attn_geom, mtp_rope_table,
                                             mtp_workspace_init, mtp_workspace_set_wait_limit,
                                             mtp_workspace_status)
    nh, nkv, d, L, m = 8, 2, 128, 1024, 1          # 64 tiles: many splits per KV head
    rng = np.random.default_rng(9)
    cap = L + m
    qp = rng.standard_normal((m, nh * d)).astype(np.float32)
    kp = rng.standard_normal((m, nkv * d)).astype(np.float32)
    vp = rng.standard_normal((m, nkv * d)).astype(np.float32)
    kc = np.zeros((nkv, cap, d), np.float32)
    vc = np.zeros((nkv, cap, d), np.float32)
    kc[:, :L] = rng.standard_normal((nkv, L, d))
    vc[:, :L] = rng.standard_normal((nkv, L, d))
    g = attn_geom(nh, nkv, d, d, d, 0, False, 1e-6)
    rope = torch.empty(cap * d, dtype=torch.float32, device=dev)
    mtp_rope_table(rope, cap, d, 1e6)
    kc_d, vc_d = _t(kc, dev), _t(vc, dev)
    out = torch.zeros((m, nh * d), device=dev)
    args = (g, _t(qp, dev), _t(kp, dev), _t(vp, dev), None, None, rope, None, kc_d, vc_d, L, cap, m,
            out)
    ws = attn_decode_sink(*args)
    torch.cuda.synchronize()
    mtp_workspace_set_wait_limit(ws, 1)
    attn_decode_sink(*args, ws)
    torch.cuda.synchronize()
    # every split but the last to arrive polls the arrival count once, short of it
    assert mtp_workspace_status(ws) == 4
    mtp_workspace_init(ws)
    out.zero_()
    attn_decode_sink(*args, ws)
    torch.cuda.synchronize()
    assert mtp_workspace_status(ws) == 0
    q = O.rope(qp.astype(np.float64).reshape(m, nh, d)[0], L, 1e6, d)[None]
    k = O.rope(kp.astype(np.float64).reshape(m, nkv, d)[0], L, 1e6, d)[None]
    k_all = np.concatenate([kc[:, :L], k.transpose(1, 0, 2)], axis=1)
    v_all = np.concatenate([vc[:, :L], vp.reshape(m, nkv, d).transpose(1, 0, 2)], axis=1)
    ref = O.attention(q, k_all, v_all, [L], 0, None)
    assert_close(out.cpu().numpy(), ref.reshape(m, nh * d), "attention after re-init")
