"""Whole draft-layer and chain parity with the CPU oracle on seeded inputs."""

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


SCALED = {
    "tiny_dense": CONFIGS["tiny_dense"],
    "qwen_small": CONFIGS["qwen_dense"].with_(name="qwen_small", hidden=512, n_heads=8, n_kv_heads=2,
                                              intermediate=1024 + 128, vocab=6000, cache_len=300),
    "qwen_small_m3": CONFIGS["qwen_dense"].with_(name="qwen_small_m3", hidden=512, n_heads=4,
                                                 n_kv_heads=2, intermediate=768, vocab=3000,
                                                 cache_len=45, m=3),
    "qwen_small_m16": CONFIGS["qwen_dense"].with_(name="qwen_small_m16", hidden=384, n_heads=2,
                                                  n_kv_heads=2, intermediate=640, vocab=2500,
                                                  cache_len=20, m=16, gated_q=False),
    "qwen_small_m9": CONFIGS["qwen_dense"].with_(name="qwen_small_m9", hidden=256, n_heads=2,
                                                 n_kv_heads=2, intermediate=384, vocab=1000,
                                                 cache_len=33, m=9),
    "moe_small": CONFIGS["moe"].with_(name="moe_small", hidden=512, n_heads=4, n_kv_heads=2,
                                      n_experts=64, top_k=8, expert_intermediate=256,
                                      shared_intermediate=256, vocab=3000, cache_len=100),
    # degenerate caches: the first draft after an empty cache (the new keys alone)
    "qwen_small_empty": CONFIGS["qwen_dense"].with_(name="qwen_small_empty", hidden=512, n_heads=8,
                                                    n_kv_heads=2, intermediate=1024 + 128,
                                                    vocab=6000, cache_len=0),
    "qwen_small_m3_empty": CONFIGS["qwen_dense"].with_(name="qwen_small_m3_empty", hidden=512,
                                                       n_heads=4, n_kv_heads=2, intermediate=768,
                                                       vocab=3000, cache_len=0, m=3),
    "moe_small_empty": CONFIGS["moe"].with_(name="moe_small_empty", hidden=512, n_heads=4,
                                            n_kv_heads=2, n_experts=64, top_k=8,
                                            expert_intermediate=256, shared_intermediate=256,
                                            vocab=3000, cache_len=0),
}


def run_layer(cfg, dev, sample_rows=None):
    """Runs one layer on the GPU and in the oracle; returns both result dicts."""
    import torch
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    w = make_layer_weights(cfg)
    step = make_step(cfg)
    shared = make_shared(cfg)
    st = make_state(cfg)
    lyr = DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev)
    H, m = cfg.hidden, cfg.m
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    hid = torch.zeros(H, dtype=torch.float32, device=dev)
    u2 = torch.zeros((m, H), dtype=torch.float32, device=dev)
    logits = torch.zeros(cfg.vocab, dtype=torch.float32, device=dev)
    lyr.forward(_t(step["hidden"], dev), cfg.cache_len, tokens=_t(step["tokens"], dev), token=tok,
                value=val, hidden_out=hid, u2=u2, logits=logits)
    torch.cuda.synchronize()
    gpu = {"token": int(tok.item()), "value": float(val.item()), "hidden_out": hid.cpu().numpy(),
           "u2": u2.cpu().numpy(), "logits": logits.cpu().numpy(),
           "k_new": lyr.k_cache[:, cfg.cache_len:cfg.cache_len + m].cpu().numpy(),
           "v_new": lyr.v_cache[:, cfg.cache_len:cfg.cache_len + m].cpu().numpy()}
    e = shared["embed"][step["tokens"]]
    ref = O.draft_layer(cfg, w, shared["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e,
                        want_logits=sample_rows is None)
    return gpu, ref, lyr, (w, shared, st, step)


def check_layer(gpu, ref, cfg, name):
    assert_close(gpu["u2"], ref["u2"], f"{name} u2")
    assert_close(gpu["hidden_out"], ref["hidden_out"], f"{name} hidden_out")
    assert_close(gpu["k_new"], ref["k_new"].transpose(1, 0, 2), f"{name} appended K")
    assert_close(gpu["v_new"], ref["v_new"].transpose(1, 0, 2), f"{name} appended V")
    if "logits" in ref:
        assert_close(gpu["logits"], ref["logits"], f"{name} logits")
        assert_token(gpu["token"], ref["token"], ref["margin"], name)


@pytest.mark.parametrize("name", list(SCALED))
def test_layer_scaled(dev, name):
    cfg = SCALED[name]
    gpu, ref, lyr, _ = run_layer(cfg, dev)
    check_layer(gpu, ref, cfg, name)
    assert gpu["token"] == int(np.argmax(gpu["logits"]))


def test_layer_repeat_is_bitwise(dev):
    import torch
    cfg = SCALED["qwen_small"]
    gpu1, _, lyr, (w, shared, st, step) = run_layer(cfg, dev)
    # same step again (the cache rows it appends are rewritten identically)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    u2 = torch.zeros((cfg.m, cfg.hidden), device=dev)
    lyr.forward(_t(step["hidden"], dev), cfg.cache_len, tokens=_t(step["tokens"], dev), token=tok,
                value=val, u2=u2)
    torch.cuda.synchronize()
    assert np.array_equal(u2.cpu().numpy(), gpu1["u2"])
    assert int(tok.item()) == gpu1["token"]


def test_layer_embedding_rows_mode(dev):
    """Caller-provided embedding rows give the same result as the table gather."""
    import torch
    cfg = SCALED["tiny_dense"]
    gpu, ref, lyr, (w, shared, st, step) = run_layer(cfg, dev)
    lyr.desc.embed = None
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    u2 = torch.zeros((cfg.m, cfg.hidden), device=dev)
    rows = _t(shared["embed"][step["tokens"]], dev)
    lyr.forward(_t(step["hidden"], dev), cfg.cache_len, embed_rows=rows, token=tok, value=val, u2=u2)
    torch.cuda.synchronize()
    assert np.array_equal(u2.cpu().numpy(), gpu["u2"])


def _chain(cfg, dev):
    import torch
    from mtp_speculative_draft_gb300.layer import DraftChain, DraftLayer, SharedHead
    shared = make_shared(cfg)
    sh = SharedHead(shared, dev)
    ws = [make_layer_weights(cfg, k) for k in range(cfg.n_layers)]
    sts = [make_state(cfg, k) for k in range(cfg.n_layers)]
    layers = [DraftLayer(cfg, ws[k], sh, sts[k], device=dev) for k in range(cfg.n_layers)]
    chain = DraftChain(layers)
    step = make_step(cfg)
    seq = torch.zeros(cfg.m + cfg.n_layers, dtype=torch.int32, device=dev)
    seq[:cfg.m] = _t(step["tokens"], dev)
    nl, m, H = cfg.n_layers, cfg.m, cfg.hidden
    values = torch.zeros(nl, dtype=torch.float32, device=dev)
    hout = torch.zeros((nl, H), dtype=torch.float32, device=dev)
    u2 = torch.zeros((nl, m, H), dtype=torch.float32, device=dev)
    logits = torch.zeros((nl, cfg.vocab), dtype=torch.float32, device=dev)
    chain.forward(_t(step["hidden"], dev), seq, [cfg.cache_len] * nl, values, hout, u2=u2,
                  logits=logits)
    torch.cuda.synchronize()
    drafts = seq.cpu().numpy()[m:].tolist()
    gpu = {"values": values.cpu().numpy(), "hidden_out": hout.cpu().numpy(), "u2": u2.cpu().numpy(),
           "logits": logits.cpu().numpy(),
           "k_new": [lyr.k_cache[:, cfg.cache_len:cfg.cache_len + m].cpu().numpy() for lyr in layers],
           "v_new": [lyr.v_cache[:, cfg.cache_len:cfg.cache_len + m].cpu().numpy() for lyr in layers]}
    return drafts, gpu, (shared, ws, sts, step)


def check_chain(cfg, drafts, gpu, ref, name):
    """Element-wise parity of every layer of a chain: u2, appended K/V rows,
    the full last-row logits, hidden_out, the draft's value and its token."""
    for k in range(cfg.n_layers):
        r = ref[k]
        assert_close(gpu["u2"][k], r["u2"], f"{name} layer {k} u2")
        assert_close(gpu["hidden_out"][k], r["hidden_out"], f"{name} layer {k} hidden_out")
        assert_close(gpu["k_new"][k], r["k_new"].transpose(1, 0, 2), f"{name} layer {k} appended K")
        assert_close(gpu["v_new"][k], r["v_new"].transpose(1, 0, 2), f"{name} layer {k} appended V")
        assert_close(gpu["logits"][k], r["logits"], f"{name} layer {k} logits")
        assert_token(drafts[k], r["token"], r["margin"], f"{name} layer {k}")
        assert drafts[k] == int(np.argmax(gpu["logits"][k]))
        rms = np.sqrt(np.mean(r["logits"] ** 2))
        assert abs(gpu["values"][k] - r["logits"][drafts[k]]) <= 1e-3 * max(abs(r["value"]), rms)


def test_chain_scaled(dev):
    cfg = CONFIGS["mimo_chain"].with_(name="mimo_small", hidden=512, n_heads=8, n_kv_heads=2,
                                      intermediate=1024, vocab=5000, cache_len=40, window=16)
    drafts, gpu, (shared, ws, sts, step) = _chain(cfg, dev)
    embed = lambda t: shared["embed"][t]  # noqa: E731
    caches = [(s["k_cache"], s["v_cache"]) for s in sts]
    # the oracle follows the GPU's drafts where a near-tie allows either token
    ref = O.draft_chain(cfg, ws, shared["lm_head"], embed, caches, step["hidden"], step["tokens"],
                        forced=drafts)
    check_chain(cfg, drafts, gpu, ref, "chain")


# ------------------------------------------------------------------ full size
@pytest.mark.parametrize("name", ["qwen_dense", "moe"])
def test_layer_full_size(dev, name):
    """Full-size layer against the oracle element by element, the full
    151 936-entry logit vector included, and its token under the margin rule."""
    cfg = CONFIGS[name]
    gpu, ref, lyr, (w, shared, st, step) = run_layer(cfg, dev)
    check_layer(gpu, ref, cfg, name)
    assert gpu["token"] == int(np.argmax(gpu["logits"]))


def test_chain_full_size(dev):
    """The three-layer chain at full size ("cortiq-engine 0.8.49 src/mimo_mtp.rs",
    "How the three layers chain", mimo_mtp_draft): every layer's u2, appended
    K/V rows, 152 576 logits, hidden_out and draft, element by element."""
    cfg = CONFIGS["mimo_chain"]
    drafts, gpu, (shared, ws, sts, step) = _chain(cfg, dev)
    embed = lambda t: shared["embed"][t]  # noqa: E731
    caches = [(s["k_cache"], s["v_cache"]) for s in sts]
    ref = O.draft_chain(cfg, ws, shared["lm_head"], embed, caches, step["hidden"], step["tokens"],
                        forced=drafts)
    check_chain(cfg, drafts, gpu, ref, "chain")
