"""Device-resident draft drivers against the oracle.

* mtp_draft_steps: k chained one-row steps of one layer, each reading the
  previous step's normed row and draft token on the device ("hf2q 0.1.13
  src/inference/models/qwen35/mtp.rs", forward_draft_with_hidden).
* mtp_mimo_draft_round in a speculative loop driven by a CPU fake verifier
  (a fixed accept pattern): per-layer committed/base state, provisional rows
  dropped each round, a history gap that restarts the caches of the layers
  whose committed rows fell out of the history, the
  accepted prefix and the generation's counters ("cortiq-engine 0.8.49
  src/mimo_mtp.rs", mimo_mtp_draft and mimo_spec_round).
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


QWEN_SMALL = CONFIGS["qwen_dense"].with_(name="qwen_small", hidden=512, n_heads=8, n_kv_heads=2,
                                         intermediate=1024 + 128, vocab=6000, cache_len=300)


@pytest.mark.parametrize("name,k", [("qwen_small", 4), ("qwen_dense", 3)])
def test_draft_steps_match_oracle_self_chain(dev, name, k):
    import torch
    from mtp_speculative_draft_gb300 import mtp_draft_steps, mtp_workspace_status
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    cfg = QWEN_SMALL if name == "qwen_small" else CONFIGS["qwen_dense"]
    w, shared = make_layer_weights(cfg), make_shared(cfg)
    st = make_state(cfg.with_(m=k))
    step = make_step(cfg)
    lyr = DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev)
    H = cfg.hidden
    tokens = torch.zeros(k + 1, dtype=torch.int32, device=dev)
    tokens[0] = int(step["tokens"][0])
    values = torch.zeros(k, dtype=torch.float32, device=dev)
    hout = torch.zeros((k, H), dtype=torch.float32, device=dev)
    mtp_draft_steps(lyr.desc, k, _t(step["hidden"][0], dev), tokens, cfg.cache_len, values, hout,
                    lyr.ws)
    torch.cuda.synchronize()
    assert mtp_workspace_status(lyr.ws) == 0
    drafts = tokens.cpu().numpy()[1:].tolist()
    embed = lambda t: shared["embed"][t]  # noqa: E731
    kc, vc = lyr.k_cache.cpu().numpy(), lyr.v_cache.cpu().numpy()
    vals, hs = values.cpu().numpy(), hout.cpu().numpy()
    # each step against the oracle on the inputs the device step had: the
    # previous step's normed row and draft, and the cache rows the earlier
    # steps appended (so rounding does not compound along the chain); a
    # wrongly wired hidden or token shows up as a mismatch of that step
    toks = [int(step["tokens"][0])] + drafts
    ref = []
    for i in range(k):
        h_in = step["hidden"][0] if i == 0 else hs[i - 1]
        ref.append(O.draft_layer(cfg, w, shared["lm_head"], kc, vc, h_in[None], embed(toks[i])[None],
                                 pos0=cfg.cache_len + i))
    # the chain wiring itself: the oracle's free-running chain drafts the same tokens
    free = O.draft_steps(cfg, w, shared["lm_head"], embed, st["k_cache"], st["v_cache"],
                         step["hidden"][0], toks[0], cfg.cache_len, k, forced=drafts)
    for i, r in enumerate(free):
        assert_token(drafts[i], r["token"], r["margin"], f"{name} free chain step {i}")
    for i, r in enumerate(ref):
        assert_token(drafts[i], r["token"], r["margin"], f"{name} step {i}")
        assert_close(hs[i], r["hidden_out"], f"{name} step {i} hidden_out")
        rms = np.sqrt(np.mean(r["logits"] ** 2))
        assert abs(vals[i] - r["logits"][drafts[i]]) <= 1e-3 * max(abs(r["value"]), rms)
        assert_close(kc[:, cfg.cache_len + i], r["k_new"][0], f"{name} step {i} K row")
        assert_close(vc[:, cfg.cache_len + i], r["v_new"][0], f"{name} step {i} V row")


MIMO_SMALL = CONFIGS["mimo_chain"].with_(name="mimo_rounds", hidden=512, n_heads=8, n_kv_heads=2,
                                         intermediate=1024, vocab=5000, cache_len=0, m=1,
                                         window=16)


def test_mimo_rounds_with_a_fake_verifier(dev):
    import torch
    import mtp_synth
    from mtp_speculative_draft_gb300 import (MimoLayerState, SpecStats, mtp_mimo_draft_round,
                                             mtp_spec_accept, mtp_spec_note_round,
                                             mtp_workspace_status, workspace)
    from mtp_speculative_draft_gb300 import _lib as L
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    import ctypes as C
    cfg, K, CAP, POS = MIMO_SMALL, 3, 96, 128
    H, V = cfg.hidden, cfg.vocab
    shared = make_shared(cfg)
    sh = SharedHead(shared, dev)
    ws_l = [make_layer_weights(cfg, k) for k in range(K)]
    layers = [DraftLayer(cfg, ws_l[k], sh, make_state(cfg.with_(m=CAP), k), device=dev)
              for k in range(K)]
    # the rotary tables cover every position of the run (caches restart part-way)
    from mtp_speculative_draft_gb300 import mtp_rope_table
    for lyr in layers:
        lyr.rope = torch.empty(POS * cfg.rot_dim, dtype=torch.float32, device=dev)
        mtp_rope_table(lyr.rope, POS, cfg.rot_dim, cfg.rope_theta)
        lyr.desc.rope = lyr.rope.data_ptr()
    hist_all = mtp_synth.normal_f32(cfg.seed, "rounds.hist", (POS, H))   # target hidden by position
    d_hist = _t(hist_all, dev)
    rng = np.random.default_rng(5)
    P = 10
    ids = rng.integers(0, V, P + 1).tolist()                              # x_0 .. x_P (x_P pending)
    d_ids = torch.zeros(POS, dtype=torch.int32, device=dev)
    d_ids[:P + 1] = _t(np.array(ids, np.int32), dev)
    values = torch.zeros(K, dtype=torch.float32, device=dev)
    ws = max((lyr.ws for lyr in layers), key=lambda x: x.numel())
    catch_ws = workspace(max(L.load().mtp_kv_catch_up_workspace_bytes(C.byref(lyr.desc), POS)
                             for lyr in layers))
    states = (MimoLayerState * K)()
    stats = SpecStats()
    # oracle side
    embed = lambda tk: shared["embed"][tk]  # noqa: E731
    caches = [[np.zeros((cfg.n_kv_heads, CAP, cfg.head_dim_qk)),
               np.zeros((cfg.n_kv_heads, CAP, cfg.head_dim_v))] for _ in range(K)]
    ostates = [O.mimo_layer_state_new() for _ in range(K)]
    ostats = O.spec_stats_new()
    accept = [0, 3, 1, 2, 3, 0, 1, 2]
    t, lo, hist_end = P - 1, 0, P
    restarted = []
    for rnd, a_want in enumerate(accept):
        if rnd == 4:
            lo = t - 2                      # a history gap: only positions t-2 .. t remain
            restarted = [l for l in range(K) if ostates[l]["committed"] < lo]
            assert restarted                # (layers whose committed rows fell out restart)
        hist_ptr = d_hist[lo:]
        n = mtp_mimo_draft_round([lyr.desc for lyr in layers], states, hist_ptr, lo, hist_end, t,
                                 d_ids, len(ids), values, ws, catch_ws)
        torch.cuda.synchronize()
        assert n == K
        drafts = d_ids[t + 2:t + 2 + n].cpu().numpy().tolist()
        ref_drafts, res = O.mimo_draft_round(cfg, ws_l, shared["lm_head"], embed, caches, ostates,
                                             lambda j: hist_all[j], lo, hist_end, t, ids, K,
                                             forced=drafts)
        vals = values.cpu().numpy()
        for l in range(K):
            r = res[l]
            assert_token(drafts[l], r["token"], r["margin"], f"round {rnd} layer {l}")
            rms = np.sqrt(np.mean(r["logits"] ** 2))
            assert abs(vals[l] - r["logits"][drafts[l]]) <= 1e-3 * max(abs(r["value"]), rms)
            assert (states[l].committed, states[l].base, states[l].kv_len) == (
                ostates[l]["committed"], ostates[l]["base"], ostates[l]["kv_len"]), f"round {rnd} layer {l}"
        if rnd == 4:
            assert all(states[l].base == lo for l in restarted)
            assert all(states[l].base == 0 for l in range(K) if l not in restarted)
        # the fake verifier agrees with the first a_want drafts, then differs
        a_want = min(a_want, n)
        bonus = (drafts[a_want] + 7919) % V if a_want < n else int(rng.integers(0, V))
        verify = drafts[:a_want] + [bonus]
        a = mtp_spec_accept(drafts, verify + [0] * (n + 1 - len(verify)))
        assert a == O.spec_accept(drafts, verify) == a_want
        mtp_spec_note_round(stats, n, a)
        O.spec_note_round(ostats, n, a)
        emitted = drafts[:a] + [bonus]
        d_ids[t + 2:t + 2 + len(emitted)] = _t(np.array(emitted, np.int32), dev)
        ids += emitted
        hist_end = t + a + 2                # the backbone's hiddens of positions t+1 .. t+a+1
        t += a + 1
    assert mtp_workspace_status(ws) == 0 and mtp_workspace_status(catch_ws) == 0
    assert stats.rounds == ostats["rounds"] and stats.accepted == ostats["accepted"]
    assert list(stats.accept_hist)[:K + 1] == ostats["accept_hist"]
    for l in range(K):
        n_rows = states[l].kv_len
        assert_close(layers[l].k_cache.cpu().numpy()[:, :n_rows], caches[l][0][:, :n_rows],
                     f"layer {l} K cache")
        assert_close(layers[l].v_cache.cpu().numpy()[:, :n_rows], caches[l][1][:, :n_rows],
                     f"layer {l} V cache")
