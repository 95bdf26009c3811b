"""Activations beyond the f16 range reach the tensor-core products intact.

The f16 hi/lo activation split stores each 32-value group times 2^-e when its
largest |x| is 2^15 or more (the group sum keeps the true scale and the
consumer multiplies the group's weight scale by 2^e).  The target hidden the
draft layer reads is the backbone's output before its final norm ("cortiq-
engine 0.8.49 src/mimo_mtp.rs", module doc), where single activations far
above f16's 65504 occur; with the folded RMSNorms that raw row is what gets
packed.  Checked against the oracle: the quantised matmul at one row (the
one-row kernel) and at several rows (the tensor-core kernel), and a whole
draft step whose hidden carries such outliers.
"""

import numpy as np
import pytest

from helpers import assert_close, assert_token, seeded_affine
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
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(dev)


def plant_outliers(x, rng):
    """Values around and far beyond the f16 range at scattered positions,
    including one group made entirely of large values."""
    x = x.copy()
    flat = x.reshape(-1)
    vals = np.array([1.0e5, -1.0e5, 3.3e6, -7.0e4, 65519.0, 4.0e4, -2.5e5, 1.2e9], np.float32)
    pos = rng.choice(flat.size, size=len(vals), replace=False)
    flat[pos] = vals
    flat[32:64] = rng.uniform(2.0e4, 9.0e4, 32).astype(np.float32) * rng.choice([-1, 1], 32)
    return x


@pytest.mark.parametrize("m,n,k", [(1, 300, 512), (3, 130, 640), (16, 257, 512)])
def test_qmatmul_outlier_activations(dev, m, n, k):
    import torch
    from mtp_speculative_draft_gb300 import affine4, qmatmul_affine4
    rng = np.random.default_rng(17 + m)
    w = seeded_affine(rng, n, k)
    x = plant_outliers(rng.standard_normal((m, k)).astype(np.float32), rng)
    assert np.abs(x).max() > 1e6
    q, s, b = (_t(t, dev) for t in w)
    desc = affine4(q, s, b)
    y = torch.zeros((m, n), dtype=torch.float32, device=dev)
    qmatmul_affine4(_t(x, dev), desc, y, m)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got, O.qmatmul(x, w), f"qmatmul with outliers m={m} n={n} k={k}")


def test_draft_step_hidden_outliers(dev):
    """Qwen-style layer, one row: outliers in the target hidden (up to 3e5)."""
    import torch
    from mtp_speculative_draft_gb300 import mtp_workspace_status
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    cfg = CONFIGS["qwen_dense"].with_(name="qwen_small", hidden=512, n_heads=8, n_kv_heads=2,
                                      intermediate=1024 + 128, vocab=6000, cache_len=300)
    w, shared, st, step = make_layer_weights(cfg), make_shared(cfg), make_state(cfg), make_step(cfg)
    rng = np.random.default_rng(23)
    hidden = step["hidden"].copy()
    idx = rng.choice(cfg.hidden, size=6, replace=False)
    hidden[0, idx] = np.array([3.0e5, -1.5e5, 8.0e4, 6.6e4, -2.0e5, 1.0e5], np.float32)
    lyr = DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    u2 = torch.zeros((1, cfg.hidden), dtype=torch.float32, device=dev)
    logits = torch.zeros(cfg.vocab, dtype=torch.float32, device=dev)
    lyr.forward(_t(hidden, dev), cfg.cache_len, tokens=_t(step["tokens"], dev), token=tok,
                value=val, u2=u2, logits=logits)
    torch.cuda.synchronize()
    assert mtp_workspace_status(lyr.ws) == 0
    e = shared["embed"][step["tokens"]]
    ref = O.draft_layer(cfg, w, shared["lm_head"], st["k_cache"], st["v_cache"], hidden, e)
    assert_close(u2.cpu().numpy(), ref["u2"], "u2 with hidden outliers")
    assert_close(logits.cpu().numpy(), ref["logits"], "logits with hidden outliers")
    assert_token(int(tok.item()), ref["token"], ref["margin"], "token with hidden outliers")
