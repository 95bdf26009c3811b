"""MoE expert stacks with bfloat16 scales and biases ("hf2q 0.1.1
src/serve/forward_mlx_shared.rs", MlxAffineMoeStack) against the oracle on
the same stacks (oracle.moe_stack_bf16: the float32 values rounded to
bfloat16, ties to even), element by element, the full-size layer included."""

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


MOE_SMALL = CONFIGS["moe"].with_(name="moe_small", hidden=512, n_heads=4, n_kv_heads=2,
                                 n_experts=64, top_k=8, expert_intermediate=256,
                                 shared_intermediate=256, vocab=3000, cache_len=100)


@pytest.mark.parametrize("name", ["moe_small", "moe"])
def test_moe_layer_bf16_stacks(dev, name):
    import torch
    from mtp_speculative_draft_gb300 import mtp_workspace_status
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    cfg = MOE_SMALL if name == "moe_small" else CONFIGS["moe"]
    w, shared, st, step = make_layer_weights(cfg), make_shared(cfg), make_state(cfg), make_step(cfg)
    lyr = DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev, bf16_stacks=True)
    assert lyr.aff["exp_gate"].s.dtype == torch.bfloat16
    H = cfg.hidden
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    u2 = torch.zeros((1, H), dtype=torch.float32, device=dev)
    hid = torch.zeros(H, dtype=torch.float32, device=dev)
    logits = torch.zeros(cfg.vocab, dtype=torch.float32, device=dev)
    lyr.forward(_t(step["hidden"], dev), cfg.cache_len, tokens=_t(step["tokens"], dev), token=tok,
                value=val, hidden_out=hid, u2=u2, logits=logits)
    torch.cuda.synchronize()
    assert mtp_workspace_status(lyr.ws) == 0
    wb = dict(w)
    for nm in ("exp_gate", "exp_up", "exp_down"):
        wb[nm] = O.moe_stack_bf16(w[nm])
    e = shared["embed"][step["tokens"]]
    ref = O.draft_layer(cfg, wb, shared["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    assert_close(u2.cpu().numpy(), ref["u2"], f"{name} u2 (bf16 stacks)")
    assert_close(hid.cpu().numpy(), ref["hidden_out"], f"{name} hidden_out (bf16 stacks)")
    assert_close(logits.cpu().numpy(), ref["logits"], f"{name} logits (bf16 stacks)")
    assert_token(int(tok.item()), ref["token"], ref["margin"], f"{name} token (bf16 stacks)")
    # the rounding is visible: the float32 stacks give a different u2
    ref32 = O.draft_layer(cfg, w, shared["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e,
                          want_logits=False)
    assert np.max(np.abs(ref32["u2"] - ref["u2"])) > 1e-6


def test_moe_ffn_bf16_stacks_matches_oracle(dev):
    """The standalone moe_ffn entry point on bf16 stacks, with its routing."""
    import torch
    from mtp_speculative_draft_gb300 import moe_ffn
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    cfg = MOE_SMALL
    w, shared, st = make_layer_weights(cfg), make_shared(cfg), make_state(cfg)
    lyr = DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev, bf16_stacks=True)
    rng = np.random.default_rng(8)
    H = cfg.hidden
    u1 = rng.standard_normal((1, H)).astype(np.float32)
    u2 = torch.zeros((1, H), dtype=torch.float32, device=dev)
    sel = torch.zeros(cfg.top_k, dtype=torch.int32, device=dev)
    wt = torch.zeros(cfg.top_k + 1, dtype=torch.float32, device=dev)
    moe_ffn(lyr.moe, _t(u1, dev), lyr.t["post_norm"], cfg.eps, H, u2, sel, wt)
    torch.cuda.synchronize()
    wb = dict(w)
    for nm in ("exp_gate", "exp_up", "exp_down"):
        wb[nm] = O.moe_stack_bf16(w[nm])
    f = O.rmsnorm(u1, w["post_norm"], cfg.eps)
    ref = u1 + O.moe_ffn(f, wb, cfg)
    assert_close(u2.cpu().numpy(), ref, "moe_ffn u2 (bf16 stacks)")
    rsel, rw = O.moe_route(f[0], w["router"], cfg.top_k)
    assert sel.cpu().numpy().tolist() == rsel.tolist()
    assert_close(wt.cpu().numpy()[:cfg.top_k], rw, "routing weights")
