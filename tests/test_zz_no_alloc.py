"""attn_decode_sink_noalloc (static device scratch) against attn_decode_sink.

Collected last on purpose: the static scratch is set up by its first call, so
this file also checks that it works after every other test has run.
"""

from __future__ import annotations

import numpy as np
import pytest

from helpers import assert_close

pytestmark = pytest.mark.gpu

# (n_heads, n_kv_heads, dqk, dv, cache_len, m, window, sinks, gated, qk_norm)
CASES = [
    (40, 8, 128, 128, 4096, 1, 0, False, True, True),    # 40/8 heads, 4096 cached rows
    (32, 8, 192, 128, 320, 4, 128, True, False, False),  # window 128 with sinks, 4 rows
    (16, 2, 256, 256, 700, 2, 0, False, False, True),    # 256-dim heads, ragged last tile
    (4, 2, 64, 64, 0, 3, 0, False, False, True),         # empty cache: new rows only
]


@pytest.fixture(scope="module")
def dev():
    import torch
    from mtp_speculative_draft_gb300 import build
    build.build()
    torch.cuda.init()
    return torch.device("cuda:0")


def _inputs(case, seed):
    nh, nkv, dqk, dv, L, m, window, use_sinks, gated, qknorm = case
    rng = np.random.default_rng(seed)
    cap = L + m + 5
    qp = rng.standard_normal((m, nh * dqk * (2 if gated else 1))).astype(np.float32)
    kp = rng.standard_normal((m, nkv * dqk)).astype(np.float32)
    vp = rng.standard_normal((m, nkv * dv)).astype(np.float32)
    kc = np.zeros((nkv, cap, dqk), np.float32)
    vc = np.zeros((nkv, cap, dv), np.float32)
    kc[:, :L] = rng.standard_normal((nkv, L, dqk))
    vc[:, :L] = rng.standard_normal((nkv, L, dv))
    qn = (1 + 0.1 * rng.standard_normal(dqk)).astype(np.float32) if qknorm else None
    kn = (1 + 0.1 * rng.standard_normal(dqk)).astype(np.float32) if qknorm else None
    sinks = rng.standard_normal(nh).astype(np.float32) if use_sinks else None
    return cap, qp, kp, vp, kc, vc, qn, kn, sinks


@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_workspace_call(dev, case):
    import torch
    from mtp_speculative_draft_gb300 import (attn_decode_sink, attn_decode_sink_noalloc, attn_geom,
                                             mtp_rope_table)
    nh, nkv, dqk, dv, L, m, window, _, gated, _ = case
    cap, qp, kp, vp, kc, vc, qn, kn, sinks = _inputs(case, 7 * L + m)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    g = attn_geom(nh, nkv, dqk, dv, dqk, window, gated, 1e-6)
    rope = torch.empty(cap * dqk, dtype=torch.float32, device=dev)
    mtp_rope_table(rope, cap, dqk, 1e4 if window else 1e6)
    args = (t(qp), t(kp), t(vp), t(qn), t(kn), rope, t(sinks))

    kc_ref, vc_ref = t(kc), t(vc)
    ref = torch.zeros((m, nh * dv), device=dev)
    attn_decode_sink(g, *args, kc_ref, vc_ref, L, cap, m, ref)
    torch.cuda.synchronize()
    ref_np = ref.cpu().numpy()

    kc_na, vc_na = t(kc), t(vc)
    for call in range(2):  # two calls in a row: the second sees the counters the first left
        out = torch.full((m, nh * dv), float("nan"), device=dev)
        attn_decode_sink_noalloc(g, *args, kc_na, vc_na, L, cap, m, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref_np, f"noalloc call {call} {case}")
    assert_close(kc_na.cpu().numpy(), kc_ref.cpu().numpy(), "appended keys")
    assert np.array_equal(vc_na.cpu().numpy(), vc_ref.cpu().numpy())


def test_noalloc_rejects_oversized_scratch(dev):
    import torch
    from mtp_speculative_draft_gb300 import attn_decode_sink_noalloc, attn_geom
    from mtp_speculative_draft_gb300._lib import MtpError
    # 64 KV heads x 2 splits x 16 query rows x 258 floats: 2.11 MB of
    # partials, above the 2 MiB scratch
    nh, nkv, d, L, m = 1024, 64, 256, 512, 1
    cap = L + m
    g = attn_geom(nh, nkv, d, d, d, 0, False, 1e-6)
    z = lambda *s: torch.zeros(s, dtype=torch.float32, device=dev)  # noqa: E731
    out = z(m, nh * d)
    with pytest.raises(MtpError) as ei:
        attn_decode_sink_noalloc(g, z(m, nh * d), z(m, nkv * d), z(m, nkv * d), None, None,
                                 z(cap * d), None, z(nkv, cap, d), z(nkv, cap, d), L, cap, m, out)
    assert ei.value.status == 4  # MTP_ERR_WORKSPACE
    assert "static scratch" in str(ei.value)
