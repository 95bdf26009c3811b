"""KV catch-up of a target batch (tcgen05 path) against the oracle's kv_catch_up.

"hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", process_target_batch and
append_attention_kv: rows i of the batch embed their token, read the target
hidden shifted one row right (the pending hidden, or zeros for a cold prompt,
at row 0), and only their K/V rows are computed and appended.  Sizes span the
four activation tile widths (16, 32, 64, 128 rows) with ragged tails.
"""

import numpy as np
import pytest

from helpers import assert_close
from oracle import mtp_oracle as O
from mtp_synth.configs import CONFIGS, make_layer_weights, make_shared, make_state

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
MIMO_SMALL = CONFIGS["mimo_chain"].with_(name="mimo_small", hidden=512, n_heads=8, n_kv_heads=2,
                                         intermediate=1024, vocab=5000, cache_len=40, m=1,
                                         n_layers=1)


def run_catch_up(cfg, dev, seq, cache_len, pos_base, pending, table=True, seed=0):
    import torch
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    w = make_layer_weights(cfg)
    shared = make_shared(cfg)
    # a cache large enough for the batch, prior rows from the workload's state
    cap = cache_len + seq + 2
    st0 = make_state(cfg.with_(cache_len=min(cfg.cache_len, cache_len), m=cap - min(cfg.cache_len, cache_len)))
    lyr = DraftLayer(cfg, w, SharedHead(shared if table else {"lm_head": shared["lm_head"]}, dev),
                     st0, device=dev)
    assert lyr.cache_cap == cap
    rng = np.random.default_rng(seed + seq)
    H = cfg.hidden
    tokens = rng.integers(0, cfg.vocab, seq).astype(np.int32)
    target = rng.standard_normal((seq, H)).astype(np.float32)
    pend = rng.standard_normal(H).astype(np.float32) if pending else None
    # the rope table must cover pos_base + cap
    if pos_base:
        from mtp_speculative_draft_gb300 import mtp_rope_table
        lyr.rope = torch.empty((pos_base + cap) * cfg.rot_dim, dtype=torch.float32, device=dev)
        mtp_rope_table(lyr.rope, pos_base + cap, cfg.rot_dim, cfg.rope_theta)
        lyr.desc.rope = lyr.rope.data_ptr()
    k_before = lyr.k_cache.cpu().numpy().copy()
    v_before = lyr.v_cache.cpu().numpy().copy()
    e = shared["embed"][tokens]
    lyr.catch_up(_t(target, dev), seq, cache_len, tokens=_t(tokens, dev) if table else None,
                 embed_rows=None if table else _t(e, dev),
                 pending=None if pend is None else _t(pend, dev), pos_base=pos_base)
    torch.cuda.synchronize()
    from mtp_speculative_draft_gb300 import mtp_workspace_status
    assert mtp_workspace_status(lyr.catch_ws) == 0
    kc, vc = lyr.k_cache.cpu().numpy(), lyr.v_cache.cpu().numpy()
    k_ref, v_ref = O.kv_catch_up(cfg, w, e, target, pending_hidden=pend, pos0=pos_base + cache_len)
    return kc, vc, k_before, v_before, k_ref, v_ref


@pytest.mark.parametrize("seq,cache_len,pos_base,pending,table", [
    (1, 0, 0, False, True),
    (5, 300, 0, True, True),
    (29, 17, 0, True, False),
    (64, 0, 0, False, True),
    (130, 300, 9, True, True),
    (200, 3, 0, True, True),
])
def test_catch_up_qwen_small(dev, seq, cache_len, pos_base, pending, table):
    cfg = QWEN_SMALL
    kc, vc, kb, vb, k_ref, v_ref = run_catch_up(cfg, dev, seq, cache_len, pos_base, pending, table)
    rows = slice(cache_len, cache_len + seq)
    assert_close(kc[:, rows], k_ref.transpose(1, 0, 2), f"catch-up K seq={seq}")
    assert_close(vc[:, rows], v_ref.transpose(1, 0, 2), f"catch-up V seq={seq}")
    # rows outside the batch are untouched
    assert np.array_equal(kc[:, :cache_len], kb[:, :cache_len])
    assert np.array_equal(kc[:, cache_len + seq:], kb[:, cache_len + seq:])
    assert np.array_equal(vc[:, :cache_len], vb[:, :cache_len])


def test_catch_up_mimo_geometry(dev):
    """QK head 192 / V head 128, no k norm, rotary base 1e4."""
    cfg = MIMO_SMALL
    seq, cache_len = 77, 40
    kc, vc, kb, vb, k_ref, v_ref = run_catch_up(cfg, dev, seq, cache_len, 0, True)
    rows = slice(cache_len, cache_len + seq)
    assert_close(kc[:, rows], k_ref.transpose(1, 0, 2), "catch-up K (192-dim heads)")
    assert_close(vc[:, rows], v_ref.transpose(1, 0, 2), "catch-up V (128-dim heads)")


def test_catch_up_split_batch_equals_whole(dev):
    """Two batches with the right pending hidden give the rows of one batch
    (within the tolerance: the split-K plan depends on the batch size)."""
    import torch
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    cfg = QWEN_SMALL
    w, shared = make_layer_weights(cfg), make_shared(cfg)
    st = make_state(cfg.with_(cache_len=0, m=80))
    sh = SharedHead(shared, dev)
    a = DraftLayer(cfg, w, sh, st, device=dev)
    b = DraftLayer(cfg, w, sh, st, device=dev)
    rng = np.random.default_rng(3)
    tokens = _t(rng.integers(0, cfg.vocab, 70).astype(np.int32), dev)
    target = _t(rng.standard_normal((70, cfg.hidden)).astype(np.float32), dev)
    a.catch_up(target, 70, 0, tokens=tokens)
    b.catch_up(target[:30], 30, 0, tokens=tokens[:30])
    b.catch_up(target[30:], 40, 30, tokens=tokens[30:], pending=target[29])
    torch.cuda.synchronize()
    assert_close(b.k_cache[:, :70].cpu().numpy(), a.k_cache[:, :70].cpu().numpy(), "split K")
    assert_close(b.v_cache[:, :70].cpu().numpy(), a.v_cache[:, :70].cpu().numpy(), "split V")


def test_catch_up_full_size(dev):
    """The Qwen-style layer (hidden 5120, 8 KV heads of 128) at 300 rows."""
    cfg = CONFIGS["qwen_dense"]
    seq, cache_len = 300, 4000
    kc, vc, kb, vb, k_ref, v_ref = run_catch_up(cfg, dev, seq, cache_len, 0, True, table=False)
    rows = slice(cache_len, cache_len + seq)
    assert_close(kc[:, rows], k_ref.transpose(1, 0, 2), "catch-up K full size")
    assert_close(vc[:, rows], v_ref.transpose(1, 0, 2), "catch-up V full size")
