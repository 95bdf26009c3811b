"""Parity of each C-ABI entry point with the CPU oracle, on seeded inputs.

Sizes span several tiles with ragged tails; the full-size shapes of the
quantised-matmul sweep are checked on every output row.
"""

import numpy as np
import pytest

from golden.fixtures import affine_fixture, affine_fixtures
from helpers import assert_close, assert_token, seeded_affine
from oracle import mtp_oracle as O

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


def _w(w, dev):
    from mtp_speculative_draft_gb300 import affine4
    q, s, b = (_t(x, dev) for x in w)
    return (q, s, b), affine4(q, s, b)


# ------------------------------------------------------------------ qmatmul
@pytest.mark.parametrize("m,n,k", [(1, 200, 384), (2, 96, 256), (3, 130, 640), (4, 512, 1024),
                                   (8, 64, 128), (9, 100, 384), (16, 257, 512), (1, 4096, 5120)])
def test_qmatmul_tma_path(dev, m, n, k):
    import torch
    from mtp_speculative_draft_gb300 import qmatmul_affine4
    rng = np.random.default_rng(m * 1000 + n)
    w = seeded_affine(rng, n, k)
    x = rng.standard_normal((m, k)).astype(np.float32)
    keep, desc = _w(w, dev)
    y = torch.zeros((m, n), dtype=torch.float32, device=dev)
    qmatmul_affine4(_t(x, dev), desc, y, m)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), O.qmatmul(x, w), f"qmatmul m={m} n={n} k={k}")


@pytest.mark.parametrize("fx", affine_fixtures(include_derived=True), ids=lambda f: f.name)
def test_qmatmul_page_fixtures(dev, fx):
    """The pages' three qmatmul fixtures (K 96, 64, 32: the plain path) and the
    first one's formulas at K = 256 (the tensor-map path)."""
    import torch
    import mtp_synth
    from mtp_speculative_draft_gb300 import qmatmul_affine4
    codes, s, b, x = affine_fixture(fx)
    w = (mtp_synth.pack_codes(codes), s, b)
    keep, desc = _w(w, dev)
    y = torch.zeros((fx.m, fx.n), dtype=torch.float32, device=dev)
    qmatmul_affine4(_t(x, dev), desc, y, fx.m)
    torch.cuda.synchronize()
    ref = O.qmatmul(x, w)
    got = y.cpu().numpy()
    assert np.max(np.abs(got - ref)) < fx.tol        # the page's own criterion
    assert_close(got, ref, f"fixture {fx.name}")


def test_qmatmul_repeatable_bitwise(dev):
    import torch
    from mtp_speculative_draft_gb300 import qmatmul_affine4
    rng = np.random.default_rng(5)
    w = seeded_affine(rng, 1000, 1024)
    x = _t(rng.standard_normal((4, 1024)).astype(np.float32), dev)
    keep, desc = _w(w, dev)
    y1 = torch.zeros((4, 1000), device=dev)
    y2 = torch.zeros((4, 1000), device=dev)
    qmatmul_affine4(x, desc, y1, 4)
    qmatmul_affine4(x, desc, y2, 4)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


SWEEP = [(5120, 5120), (17408, 5120), (5120, 17408), (151936, 5120)]


@pytest.mark.parametrize("shape", SWEEP)
def test_qmatmul_sweep_full_size(dev, shape):
    """Full-size sweep shapes at every m in {1, 2, 4, 8, 16}, every output row
    (one oracle product of the 16 activation rows serves every m)."""
    import torch
    import mtp_synth
    from mtp_synth.configs import CONFIGS
    from mtp_speculative_draft_gb300 import qmatmul_affine4
    n, k = shape
    seed = CONFIGS["qmatmul_sweep"].seed
    w = mtp_synth.affine4_weight(seed, f"sweep.{n}x{k}", n, k)
    keep, desc = _w(w, dev)
    xall = mtp_synth.normal_f32(seed, f"sweep.x.{k}", (16, k))
    ref_all = O.qmatmul(xall, w)
    for m in (1, 2, 4, 8, 16):
        x = xall[:m]
        y = torch.zeros((m, n), dtype=torch.float32, device=dev)
        qmatmul_affine4(_t(x, dev), desc, y, m)
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), ref_all[:m], f"sweep {n}x{k} m={m}")


# ------------------------------------------------------------------ rmsnorm
def test_rmsnorm_residual(dev):
    import torch
    from mtp_speculative_draft_gb300 import rmsnorm_residual
    rng = np.random.default_rng(7)
    rows, dim = 5, 5120
    a = rng.standard_normal((rows, dim)).astype(np.float32)
    d = rng.standard_normal((rows, dim)).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(dim)).astype(np.float32)
    on = torch.zeros((rows, dim), device=dev)
    os_ = torch.zeros((rows, dim), device=dev)
    rmsnorm_residual(_t(a, dev), _t(d, dev), _t(w, dev), on, os_, rows, dim, 1e-6)
    torch.cuda.synchronize()
    s64 = a.astype(np.float64) + d
    assert_close(os_.cpu().numpy(), s64, "sum")
    assert_close(on.cpu().numpy(), O.rmsnorm(s64, w, 1e-6), "norm")
    on2 = torch.zeros((rows, dim), device=dev)
    rmsnorm_residual(_t(a, dev), None, _t(w, dev), on2, None, rows, dim, 1e-6)
    torch.cuda.synchronize()
    assert_close(on2.cpu().numpy(), O.rmsnorm(a, w, 1e-6), "norm without residual")


# ------------------------------------------------------------------ attention
ATTN_CASES = [
    # nh, nkv, dqk, dv, L, m, window, sinks, gated, qknorm
    (4, 2, 64, 64, 64, 1, 0, False, False, True),
    (40, 8, 128, 128, 4096, 1, 0, False, True, True),
    (32, 8, 192, 128, 320, 4, 128, True, False, False),
    (16, 2, 256, 256, 2048, 1, 0, False, False, True),
    (8, 2, 128, 128, 0, 3, 0, True, True, True),
    (8, 4, 64, 64, 100, 4, 5, True, False, True),
    (6, 3, 96, 64, 77, 2, 0, False, False, False),
]


@pytest.mark.parametrize("case", ATTN_CASES)
def test_attention(dev, case):
    import torch
    from mtp_speculative_draft_gb300 import attn_decode_sink, attn_geom, mtp_rope_table
    nh, nkv, dqk, dv, L, m, window, use_sinks, gated, qknorm = case
    rng = np.random.default_rng(L + m + nh)
    cap = L + m + 3
    theta = 1e4 if window else 1e6
    qrows = nh * dqk * (2 if gated else 1)
    qp = rng.standard_normal((m, qrows)).astype(np.float32)
    kp = rng.standard_normal((m, nkv * dqk)).astype(np.float32)
    vp = rng.standard_normal((m, nkv * dv)).astype(np.float32)
    kc = np.zeros((nkv, cap, dqk), np.float32)
    vc = np.zeros((nkv, cap, dv), np.float32)
    kc[:, :L] = rng.standard_normal((nkv, L, dqk))
    vc[:, :L] = rng.standard_normal((nkv, L, dv))
    qn = (1 + 0.1 * rng.standard_normal(dqk)).astype(np.float32) if qknorm else None
    kn = (1 + 0.1 * rng.standard_normal(dqk)).astype(np.float32) if qknorm else None
    sinks = rng.standard_normal(nh).astype(np.float32) if use_sinks else None
    # oracle
    q = qp.astype(np.float64).reshape(m, nh, 2 if gated else 1, dqk)
    gate = q[:, :, 1, :] if gated else None
    q = q[:, :, 0, :]
    k = kp.astype(np.float64).reshape(m, nkv, dqk)
    if qknorm:
        q = O.rmsnorm(q, qn, 1e-6)
        k = O.rmsnorm(k, kn, 1e-6)
    q = np.stack([O.rope(q[r], L + r, theta, dqk) for r in range(m)])
    k = np.stack([O.rope(k[r], L + r, theta, dqk) for r in range(m)])
    k_all = np.concatenate([kc[:, :L], k.transpose(1, 0, 2)], axis=1)
    v_all = np.concatenate([vc[:, :L], vp.reshape(m, nkv, dv).transpose(1, 0, 2)], axis=1)
    ref = O.attention(q, k_all, v_all, [L + r for r in range(m)], window, sinks)
    if gated:
        ref = ref * O.sigmoid(gate)
    # gpu
    g = attn_geom(nh, nkv, dqk, dv, dqk, window, gated, 1e-6)
    rope = torch.empty(cap * dqk, dtype=torch.float32, device=dev)
    mtp_rope_table(rope, cap, dqk, theta)
    kc_d, vc_d = _t(kc, dev), _t(vc, dev)
    out = torch.zeros((m, nh * dv), device=dev)
    t = lambda a: None if a is None else _t(a, dev)  # noqa: E731
    for _ in range(2):  # a second call must give the same answer (counters reset)
        attn_decode_sink(g, t(qp), t(kp), t(vp), t(qn), t(kn), rope, t(sinks), kc_d, vc_d, L, cap,
                         m, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref.reshape(m, nh * dv), f"attention {case}")
    assert_close(kc_d.cpu().numpy()[:, L:L + m], k.transpose(1, 0, 2), "appended keys")
    assert np.array_equal(vc_d.cpu().numpy()[:, L:L + m], vp.reshape(m, nkv, dv).transpose(1, 0, 2))
    assert np.array_equal(kc_d.cpu().numpy()[:, :L], kc[:, :L])


def test_rope_table(dev):
    import math
    import torch
    from mtp_speculative_draft_gb300 import mtp_rope_table
    rot, P, theta = 128, 4100, 1e6
    t = torch.empty(P * rot, dtype=torch.float32, device=dev)
    mtp_rope_table(t, P, rot, theta)
    torch.cuda.synchronize()
    got = t.cpu().numpy().reshape(P, rot // 2, 2)
    for p in (0, 1, 17, 4099):
        for i in (0, 1, 31, 63):
            ang = p * theta ** (-2.0 * i / rot)
            assert abs(got[p, i, 0] - math.cos(ang)) < 2e-7
            assert abs(got[p, i, 1] - math.sin(ang)) < 2e-7


# ------------------------------------------------------------------ lm head
@pytest.mark.parametrize("H,V", [(256, 4096), (512, 6000), (5120, 151936)])
def test_lmhead_argmax(dev, H, V):
    import torch
    from mtp_speculative_draft_gb300 import lmhead_argmax
    rng = np.random.default_rng(V)
    w = seeded_affine(rng, V, H)
    y = rng.standard_normal(H).astype(np.float32)
    nw = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    keep, desc = _w(w, dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    logits = torch.zeros(V, dtype=torch.float32, device=dev)
    yn = torch.zeros(H, dtype=torch.float32, device=dev)
    yref = O.rmsnorm(y, nw, 1e-6)
    ref = O.qmatmul(yref[None], w)[0]
    rtok, rval, margin = O.argmax_lowest(ref)
    for _ in range(2):
        lmhead_argmax(_t(y, dev), _t(nw, dev), 1e-6, desc, tok, val, logits, yn)
        torch.cuda.synchronize()
        assert_close(yn.cpu().numpy(), yref, "normed y")
        lg = logits.cpu().numpy()
        assert_close(lg, ref, "logits")
        assert_token(int(tok.item()), rtok, margin, "argmax")
        assert int(tok.item()) == int(np.argmax(lg))         # agrees with its own logits
        assert float(val.item()) == float(lg[int(tok.item())])


def test_lmhead_argmax_ties_lowest_index(dev):
    """All-zero weights: every logit is 0, so the lowest index must win."""
    import torch
    from mtp_speculative_draft_gb300 import lmhead_argmax
    H, V = 256, 5000
    w = (np.zeros((V, H // 8), np.uint32), np.zeros((V, H // 32), np.float32),
         np.zeros((V, H // 32), np.float32))
    keep, desc = _w(w, dev)
    tok = torch.full((1,), -1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    y = _t(np.ones(H, np.float32), dev)
    lmhead_argmax(y, None, 1e-6, desc, tok, val)
    torch.cuda.synchronize()
    assert int(tok.item()) == 0 and float(val.item()) == 0.0
    # plant a maximum near the end
    b = np.zeros((V, H // 32), np.float32)
    b[4321, :] = 1.0
    b[4999, :] = 1.0
    keep2, desc2 = _w((w[0], w[1], b), dev)
    lmhead_argmax(y, None, 1e-6, desc2, tok, val)
    torch.cuda.synchronize()
    assert int(tok.item()) == 4321 and float(val.item()) == float(H)


# ------------------------------------------------------------------ verify head
@pytest.mark.parametrize("rows,H,V,mult,cap", [
    (2, 256, 4096, 1.0, 0.0),        # plain logits
    (3, 512, 6000, 0.5, 30.0),       # ragged vocabulary, multiplier and cap
    (4, 256, 4096, 80.0, 5.0),       # cap in saturation (near-ties)
    (1, 256, 4096, 1.0, 30.0),       # one row: the one-row kernel
    (16, 256, 1000, 1.0, 0.0),       # most rows, vocabulary not a multiple of 32
    (4, 5120, 151936, 1.0, 30.0),    # the 40/8-head layer's head, 4 rows
])
def test_verify_head_argmax(dev, rows, H, V, mult, cap):
    import torch
    from mtp_speculative_draft_gb300 import verify_head_argmax
    rng = np.random.default_rng(V + rows)
    w = seeded_affine(rng, V, H)
    h = rng.standard_normal((rows, H)).astype(np.float32)
    nw = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    keep, desc = _w(w, dev)
    ref, rtok, _, margin = O.verify_head(h, nw, 1e-6, w, mult if mult != 1.0 else None,
                                         cap if cap > 0 else None)
    tok = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    val = torch.zeros(rows, dtype=torch.float32, device=dev)
    logits = torch.zeros((rows, V), dtype=torch.float32, device=dev)
    ws = None
    for call in range(2):  # the second call reuses the workspace the first left
        ws = verify_head_argmax(_t(h, dev), rows, _t(nw, dev), 1e-6, desc, mult, cap, tok, val,
                                logits, ws=ws)
        torch.cuda.synchronize()
        lg = logits.cpu().numpy()
        assert_close(lg, ref, f"verify head logits call {call}")
        t, v = tok.cpu().numpy(), val.cpu().numpy()
        for r in range(rows):
            assert_token(int(t[r]), rtok[r], margin[r], f"row {r}")
            assert int(t[r]) == int(np.argmax(lg[r]))      # agrees with its own logits
            assert float(v[r]) == float(lg[r, int(t[r])])
    # without d_logits the logits stay in the workspace: same tokens
    tok2 = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    verify_head_argmax(_t(h, dev), rows, _t(nw, dev), 1e-6, desc, mult, cap, tok2, val, None, ws=ws)
    torch.cuda.synchronize()
    assert np.array_equal(tok2.cpu().numpy(), tok.cpu().numpy())


def test_verify_head_ties_lowest_index(dev):
    """Planted equal maxima (bias-only head): each row's lowest index wins."""
    import torch
    from mtp_speculative_draft_gb300 import verify_head_argmax
    H, V, rows = 256, 5000, 3
    b = np.zeros((V, H // 32), np.float32)
    b[[4321, 4999], :] = 1.0
    b[77, :] = 0.5
    keep, desc = _w((np.zeros((V, H // 8), np.uint32), np.zeros((V, H // 32), np.float32), b), dev)
    h = np.ones((rows, H), np.float32)
    h[2] = -1.0                                       # row 2: every planted logit negated
    tok = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    val = torch.zeros(rows, dtype=torch.float32, device=dev)
    verify_head_argmax(_t(h, dev), rows, None, 1e-6, desc, 1.0, 0.0, tok, val)
    torch.cuda.synchronize()
    assert tok.cpu().tolist() == [4321, 4321, 0] and val.cpu().tolist()[:2] == [float(H)] * 2
    # a cap that saturates all three planted logits to 1.0: the lowest index wins
    verify_head_argmax(_t(h, dev), rows, None, 1e-6, desc, 1.0, 1.0, tok, val)
    torch.cuda.synchronize()
    assert tok.cpu().tolist() == [77, 77, 0]
