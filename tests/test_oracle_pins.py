"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to what the pages or the mathematics fix:
the pages' printed fixtures checked by brute force, closed forms, invariants
and special cases.  A plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand, the wrong nibble order) fails one of
them.
"""

import math

import numpy as np
import pytest

import mtp_synth
from golden.fixtures import affine_fixture, affine_fixtures
from oracle import mtp_oracle as O
from mtp_synth.configs import CONFIGS, make_layer_weights, make_shared, make_state, make_step


# ---------------------------------------------------------------------------
# generator
# ---------------------------------------------------------------------------

def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0: the first output of Vigna's reference code.
    z = np.array([mtp_synth.GOLDEN], dtype=np.uint64)
    assert int(mtp_synth._mix(z)[0]) == 0xE220A8397B1DCDAF


def test_generator_slices_match_whole():
    whole = mtp_synth.normal(7, "t", 101)
    for start in (0, 1, 2, 33, 64):
        part = mtp_synth.normal(7, "t", 101 - start, start=start)
        assert np.array_equal(part, whole[start:])
    rows = mtp_synth.embedding_rows(7, "e", 50, 12, rows=[3, 0, 49])
    table = mtp_synth.embedding_rows(7, "e", 50, 12)
    assert np.array_equal(rows, table[[3, 0, 49]])


def test_generator_distributions():
    z = mtp_synth.normal(1, "n", 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    q, s, b = mtp_synth.affine4_weight(1, "w", 64, 256)
    codes = O.unpack_codes(q)
    assert codes.min() == 0 and codes.max() == 15
    assert abs(codes.mean() - 7.5) < 0.1
    assert np.all(s >= 0)
    assert abs(float(np.mean(b + 8 * s))) < 1e-3


# ---------------------------------------------------------------------------
# packed codes and affine matmul
# ---------------------------------------------------------------------------

def test_unpack_low_nibble_first():
    # [shared.rs] from_mlx_affine_linear: column 8*kp+j at bits 4j..4j+3.
    q = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert O.unpack_codes(q).tolist() == [list(range(16))]


def test_pack_unpack_roundtrip_page_fixture():
    for fx in affine_fixtures(include_derived=True):
        codes, _, _, _ = affine_fixture(fx)
        assert np.array_equal(O.unpack_codes(mtp_synth.pack_codes(codes)), codes)


def test_page_fixture_formulas_by_hand():
    # The reader against the formulas of each page test, element by element
    # for the first entries (hand-evaluated): "hf2q 0.1.1 ... forward_mlx_shared.rs",
    # from_mlx_affine_linear_roundtrips_through_packed_kernel,
    # dispatch_qmatmul_routes_affine_weight_to_packed_kernel,
    # dispatch_qmatmul_affine_equals_direct_kernel.
    fx = {f.name: f for f in affine_fixtures()}
    assert [(f.m, f.n, f.k) for f in fx.values()] == [(16, 64, 96), (8, 32, 64), (4, 32, 32)]
    c, s, b, x = affine_fixture(fx["roundtrips_through_packed_kernel"])
    assert c.ravel()[:4].tolist() == [5, 0, 11, 6]          # (11i + 5) % 16
    assert s.ravel()[2] == np.float32(0.05) + np.float32(2.0) * np.float32(0.0017)
    assert b.ravel()[3] == np.float32(-0.13) + np.float32(3.0) * np.float32(0.0023)
    assert abs(float(x.ravel()[0]) - 0.6 * math.sin(-0.4)) < 1e-6
    assert abs(float(x.ravel()[100]) - 0.6 * math.sin(1.3 - 0.4)) < 1e-6
    c, s, b, x = affine_fixture(fx["routes_affine_weight_to_packed"])
    assert c.ravel()[:4].tolist() == [3, 10, 1, 8]           # (7i + 3) % 16
    assert s.ravel()[1] == np.float32(0.07) + np.float32(0.0011)
    assert b.ravel()[1] == np.float32(-0.09) + np.float32(0.0027)
    assert abs(float(x.ravel()[0]) - 0.5 * math.cos(-0.3)) < 1e-6
    assert abs(float(x.ravel()[50]) - 0.5 * math.cos(0.55 - 0.3)) < 1e-6
    c, s, b, x = affine_fixture(fx["affine_equals_direct_kernel"])
    assert c.ravel()[:4].tolist() == [1, 6, 11, 0]           # (5i + 1) % 16
    assert s.ravel()[5] == np.float32(0.05) + np.float32(5.0) * np.float32(0.001)
    assert b.ravel()[5] == np.float32(-0.1) + np.float32(5.0) * np.float32(0.002)
    assert abs(float(x.ravel()[0]) - 0.4 * math.sin(0.2)) < 1e-6
    assert abs(float(x.ravel()[10]) - 0.4 * math.sin(0.17 + 0.2)) < 1e-6


def test_dequant_single_word():
    q = np.zeros((1, 4), dtype=np.uint32)
    q[0, 0] = 0xF0000000          # column 7 has code 15, all others 0
    s = np.array([[2.0]], dtype=np.float32)
    b = np.array([[1.0]], dtype=np.float32)
    w = O.dequant((q, s, b))
    expect = np.ones(32)
    expect[7] = 31.0
    assert np.array_equal(w[0], expect)


def _brute_qmatmul(codes, scales, biases, x, group=32):
    # Element-by-element loop of the page's CPU reference, from unpacked codes.
    m, k = x.shape
    n = codes.shape[0]
    y = [[0.0] * n for _ in range(m)]
    for r in range(m):
        for col in range(n):
            acc = 0.0
            for kk in range(k):
                g = kk // group
                wv = float(codes[col, kk]) * float(scales[col, g]) + float(biases[col, g])
                acc += float(x[r, kk]) * wv
            y[r][col] = acc
    return np.array(y)


@pytest.mark.parametrize("fx", affine_fixtures(include_derived=True), ids=lambda f: f.name)
def test_qmatmul_page_fixtures_brute_force(fx):
    m, n, tol = fx.m, fx.n, fx.tol
    codes, s, b, x = affine_fixture(fx)
    w = (mtp_synth.pack_codes(codes), s, b)
    got = O.qmatmul(x, w)
    ref = _brute_qmatmul(codes, s, b, x)
    assert got.shape == (m, n)
    assert np.max(np.abs(got - ref)) < 1e-9          # same math, f64 both sides
    assert np.max(np.abs(got - ref)) < tol


def test_qmatmul_special_cases():
    rng = np.random.default_rng(0)
    n, k = 5, 64
    codes = rng.integers(0, 16, size=(n, k))
    x = rng.standard_normal((3, k))
    q = mtp_synth.pack_codes(codes)
    # s = 0: y = b * sum(x) per group
    b = rng.standard_normal((n, k // 32)).astype(np.float32)
    y = O.qmatmul(x, (q, np.zeros_like(b), b))
    xs = x.reshape(3, k // 32, 32).sum(axis=2)
    assert np.allclose(y, xs @ b.astype(np.float64).T, rtol=0, atol=1e-12)
    # code 8 everywhere and b = -8 s: the weight is exactly zero
    q8 = mtp_synth.pack_codes(np.full((n, k), 8))
    s = np.abs(rng.standard_normal((n, k // 32))).astype(np.float32)
    assert np.all(O.qmatmul(x, (q8, s, (-8.0 * s).astype(np.float32))) == 0.0)
    # rows selection equals the full product's columns
    w = (q, s, b)
    assert np.allclose(O.qmatmul(x, w, rows=[4, 1]), O.qmatmul(x, w)[:, [4, 1]], rtol=1e-14, atol=0)


def test_qmatmul_orientation():
    # y = x W^T: one nonzero weight row picks out one output column.
    n, k = 3, 32
    codes = np.zeros((n, k), dtype=np.int64)
    codes[2, 5] = 1
    s = np.zeros((n, 1), np.float32)
    s[2, 0] = 1.0
    x = np.arange(k, dtype=np.float64)[None, :]
    y = O.qmatmul(x, (mtp_synth.pack_codes(codes), s, np.zeros((n, 1), np.float32)))
    assert y.tolist() == [[0.0, 0.0, 5.0]]


# ---------------------------------------------------------------------------
# RMSNorm, activations, RoPE
# ---------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    w = np.array([2.0, -1.0])
    y = O.rmsnorm(np.array([3.0, 4.0]), w, 0.0)
    assert np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5) * w, rtol=1e-15)
    c, eps = 0.3, 1e-6
    y = O.rmsnorm(np.full(8, c), np.ones(8), eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps), rtol=1e-15)
    x = np.random.default_rng(1).standard_normal(64)
    assert np.allclose(O.rmsnorm(5.0 * x, np.ones(64), 0.0), O.rmsnorm(x, np.ones(64), 0.0))
    # rows are normalised independently
    xx = np.stack([x, 3 * x + 1])
    assert np.allclose(O.rmsnorm(xx, np.ones(64), eps)[1], O.rmsnorm(3 * x + 1, np.ones(64), eps))


def test_sigmoid_silu_values():
    assert O.sigmoid(0.0) == 0.5
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(O.silu(-2.0) - (-2.0 / (1.0 + math.exp(2.0)))) < 1e-15


def test_rope_pairing_and_sign():
    p, theta = 3, 1e4
    y = O.rope(np.array([1.0, 0.0, 0.0, 0.0]), p, theta, 4)
    assert np.allclose(y, [math.cos(p), 0.0, math.sin(p), 0.0], atol=1e-15)
    t1 = theta ** -0.5
    y = O.rope(np.array([0.0, 1.0, 0.0, 0.0]), p, theta, 4)
    assert np.allclose(y, [0.0, math.cos(p * t1), 0.0, math.sin(p * t1)], atol=1e-15)
    # dimensions past rot_dim pass through
    y = O.rope(np.array([1.0, 2.0, 3.0, 4.0, 5.0, 6.0]), p, theta, 4)
    assert y[4] == 5.0 and y[5] == 6.0


def test_rope_invariants():
    rng = np.random.default_rng(2)
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    assert np.allclose(O.rope(q, 0, 1e6, 64), q, rtol=0, atol=0)
    r = O.rope(q, 17, 1e6, 64)
    assert np.allclose(r[:32] ** 2 + r[32:] ** 2, q[:32] ** 2 + q[32:] ** 2)
    d1 = O.rope(q, 40, 1e6, 64) @ O.rope(k, 33, 1e6, 64)
    d2 = O.rope(q, 1007, 1e6, 64) @ O.rope(k, 1000, 1e6, 64)
    assert abs(d1 - d2) < 1e-9


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _brute_attention(q, k_all, v_all, q_pos, window, sinks):
    m, nh, d = q.shape
    nkv, _, dv = v_all.shape
    out = np.zeros((m, nh, dv))
    for r in range(m):
        p = q_pos[r]
        for h in range(nh):
            kv = h * nkv // nh
            keys = [j for j in range(p + 1) if window <= 0 or j > p - window]
            ls = [sum(q[r, h, i] * k_all[kv, j, i] for i in range(d)) / math.sqrt(d) for j in keys]
            cands = ls + ([float(sinks[h])] if sinks is not None else [])
            mx = max(cands)
            ws = [math.exp(v - mx) for v in ls]
            den = sum(ws) + (math.exp(float(sinks[h]) - mx) if sinks is not None else 0.0)
            for c in range(dv):
                out[r, h, c] = sum(wj * v_all[kv, j, c] for wj, j in zip(ws, keys)) / den
    return out


@pytest.mark.parametrize("window,use_sinks", [(0, False), (3, True), (5, False), (2, True)])
def test_attention_brute_force(window, use_sinks):
    rng = np.random.default_rng(3)
    nh, nkv, d, dv, T, m = 4, 2, 6, 5, 9, 3
    q = rng.standard_normal((m, nh, d))
    k_all = rng.standard_normal((nkv, T, d))
    v_all = rng.standard_normal((nkv, T, dv))
    pos = [T - m + r for r in range(m)]
    sinks = rng.standard_normal(nh) if use_sinks else None
    got = O.attention(q, k_all, v_all, pos, window, sinks)
    ref = _brute_attention(q, k_all, v_all, pos, window, sinks)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_attention_invariants():
    rng = np.random.default_rng(4)
    nh, nkv, d, T, m = 4, 2, 8, 12, 2
    q = rng.standard_normal((m, nh, d))
    k_all = rng.standard_normal((nkv, T, d))
    v_all = rng.standard_normal((nkv, T, d))
    pos = [T - 2, T - 1]
    full = O.attention(q, k_all, v_all, pos, 0, None)
    assert np.allclose(O.attention(q, k_all, v_all, pos, T + 5, None), full, rtol=0, atol=1e-15)
    assert np.allclose(O.attention(q, k_all, v_all, pos, 0, np.full(nh, -1e30)), full, atol=1e-15)
    # a window of one: each row sees only its own key
    one = O.attention(q, k_all, v_all, pos, 1, None)
    for r, p in enumerate(pos):
        for h in range(nh):
            assert np.allclose(one[r, h], v_all[h // 2, p])
    # one key with a sink: o = v * sigmoid(l - sink)
    k1, v1 = k_all[:, :1], v_all[:, :1]
    sinks = rng.standard_normal(nh)
    o = O.attention(q[:1], k1, v1, [0], 0, sinks)
    for h in range(nh):
        logit = (q[0, h] @ k1[h // 2, 0]) / math.sqrt(d)
        assert np.allclose(o[0, h], v1[h // 2, 0] / (1.0 + math.exp(sinks[h] - logit)))
    # identical keys: o = mean of the visible values
    ke = np.repeat(k_all[:, :1], T, axis=1)
    o = O.attention(q, ke, v_all, pos, 0, None)
    assert np.allclose(o[1, 0], v_all[0, :T].mean(axis=0))
    # grouped KV heads: heads 0,1 read KV head 0, heads 2,3 read KV head 1
    v2 = v_all.copy()
    v2[1] += 1.0
    o2 = O.attention(q, k_all, v2, pos, 0, None)
    assert np.allclose(o2[:, :2], full[:, :2]) and np.allclose(o2[:, 2:], full[:, 2:] + 1.0)


# ---------------------------------------------------------------------------
# feed-forward and routing
# ---------------------------------------------------------------------------

def _tiny_affine(rng, n, k):
    codes = rng.integers(0, 16, size=(n, k))
    s = (np.abs(rng.standard_normal((n, k // 32))) * 0.01).astype(np.float32)
    b = (-8 * s + 1e-3 * rng.standard_normal((n, k // 32))).astype(np.float32)
    return mtp_synth.pack_codes(codes), s, b


def test_swiglu_composition():
    rng = np.random.default_rng(5)
    H, I = 64, 32
    g, u, d = _tiny_affine(rng, I, H), _tiny_affine(rng, I, H), _tiny_affine(rng, H, I)
    f = rng.standard_normal((2, H))
    G, U, D = O.dequant(g), O.dequant(u), O.dequant(d)
    a = f @ G.T
    ref = ((a / (1 + np.exp(-a))) * (f @ U.T)) @ D.T
    assert np.allclose(O.swiglu(f, g, u, d), ref, rtol=1e-12, atol=1e-14)


def _tiny_moe(rng, E=6, H=64, Ie=32, Is=32, top_k=2):
    cfg = CONFIGS["moe"].with_(hidden=H, n_experts=E, top_k=top_k, expert_intermediate=Ie,
                               shared_intermediate=Is)
    w = {"router": rng.standard_normal((E, H)) * 0.3}
    for name, (n, k) in (("exp_gate", (Ie, H)), ("exp_up", (Ie, H)), ("exp_down", (H, Ie))):
        parts = [_tiny_affine(rng, n, k) for _ in range(E)]
        w[name] = tuple(np.stack([p[i] for p in parts]) for i in range(3))
    w["sh_gate"], w["sh_up"], w["sh_down"] = (_tiny_affine(rng, Is, H), _tiny_affine(rng, Is, H),
                                              _tiny_affine(rng, H, Is))
    w["sh_gate_inp"] = rng.standard_normal(H) * 0.1
    return cfg, w


def _expert(w, e):
    return {k: (w[k][0][e], w[k][1][e], w[k][2][e]) for k in ("exp_gate", "exp_up", "exp_down")}


def test_moe_all_experts_is_dense_mixture():
    rng = np.random.default_rng(6)
    cfg, w = _tiny_moe(rng, top_k=6)
    f = rng.standard_normal(cfg.hidden)
    logits = w["router"] @ f
    p = np.exp(logits - logits.max())
    p /= p.sum()
    ref = np.zeros(cfg.hidden)
    for e in range(cfg.n_experts):
        ex = _expert(w, e)
        ref += p[e] * O.swiglu(f, ex["exp_gate"], ex["exp_up"], ex["exp_down"])[0]
    ref += O.sigmoid(w["sh_gate_inp"] @ f) * O.swiglu(f, w["sh_gate"], w["sh_up"], w["sh_down"])[0]
    assert np.allclose(O.moe_ffn(f, w, cfg)[0], ref, rtol=1e-12, atol=1e-14)


def test_moe_one_hot_router_and_shared_gate():
    rng = np.random.default_rng(7)
    cfg, w = _tiny_moe(rng, top_k=1)
    f = rng.standard_normal(cfg.hidden)
    w["router"] = np.zeros((cfg.n_experts, cfg.hidden))
    w["router"][4] = f * 50.0          # expert 4 dominates
    w["sh_gate_inp"] = np.zeros(cfg.hidden)   # shared gate = sigmoid(0) = 1/2
    ex = _expert(w, 4)
    ref = O.swiglu(f, ex["exp_gate"], ex["exp_up"], ex["exp_down"])[0] \
        + 0.5 * O.swiglu(f, w["sh_gate"], w["sh_up"], w["sh_down"])[0]
    assert np.allclose(O.moe_ffn(f, w, cfg)[0], ref, rtol=1e-12, atol=1e-14)


def test_moe_route_topk_renormalised_and_ties():
    sel = O.topk_lowest_index(np.array([0.1, 0.3, 0.3, 0.05, 0.3]), 2)
    assert sel.tolist() == [1, 2]
    router = np.eye(5)
    f = np.array([0.0, 1.0, 3.0, 2.0, 0.5])
    sel, wsel = O.moe_route(f, router, 2)
    assert sel.tolist() == [2, 3]
    assert np.allclose(wsel, [math.e / (math.e + 1), 1 / (math.e + 1)])


# ---------------------------------------------------------------------------
# argmax
# ---------------------------------------------------------------------------

def test_argmax_lowest_index():
    v = np.zeros(1000)
    v[737] = 2.0
    assert O.argmax_lowest(v)[:2] == (737, 2.0)
    v[12] = 2.0
    idx, val, margin = O.argmax_lowest(v)
    assert idx == 12 and margin == 0.0
    idx, val, margin = O.argmax_lowest(np.array([1.0, 3.0, 2.5]))
    assert (idx, val, margin) == (1, 3.0, 0.5)


# ---------------------------------------------------------------------------
# verify head (final norm, lm_head, multiplier, softcap, argmax per row)
# ---------------------------------------------------------------------------

def _bias_only_head(vals, H):
    """lm_head [V, H] with zero codes and scales and per-row bias vals[v] / H,
    so a row of ones has logit vals[v] (exact: the biases are powers-of-two
    fractions of the values used below)."""
    V = len(vals)
    b = np.repeat((np.asarray(vals, np.float64) / H)[:, None], H // 32, axis=1).astype(np.float32)
    return np.zeros((V, H // 8), np.uint32), np.zeros((V, H // 32), np.float32), b


def test_verify_head_softcap_follows_tanh_series():
    # c*tanh(l/c) = l - l^3/(3c^2) + 2l^5/(15c^4) - ... for |l| << c
    H, c = 64, 10.0
    w = _bias_only_head(np.linspace(-0.0625, 0.0625, 9), H)
    ones = np.ones((1, H))
    raw = O.qmatmul(ones, w)[0]
    lg, _, _, _ = O.verify_head(ones, None, 0.0, w, final_softcap=c)
    series = raw - raw ** 3 / (3 * c * c) + 2 * raw ** 5 / (15 * c ** 4)
    assert np.max(np.abs(lg[0] - series)) < 1e-13
    assert np.max(np.abs(raw - np.linspace(-0.0625, 0.0625, 9))) < 1e-15


def test_verify_head_multiplier_comes_before_the_cap():
    H, c = 64, 10.0
    vals = np.array([-50.0, -3.0, 0.0, 0.5, 2.0, 40.0])
    w = _bias_only_head(vals, H)
    ones = np.ones((1, H))
    lg, tok, val, _ = O.verify_head(ones, None, 0.0, w, logit_multiplier=2.0, final_softcap=c)
    # capping last keeps every logit inside (-c, c); capping first and then
    # doubling would reach 2c
    assert np.all(np.abs(lg) < c) and np.max(np.abs(lg)) > 0.99 * c
    assert tok == [5] and val[0] == lg[0, 5]             # monotone map: the largest stays largest
    lg2, tok2, _, _ = O.verify_head(ones, None, 0.0, w, logit_multiplier=-1.0)
    assert np.array_equal(lg2[0], -vals) and tok2 == [0]  # a negative multiplier reverses the order
    lg3, tok3, _, _ = O.verify_head(ones, None, 0.0, w)  # neither: plain logits
    assert np.array_equal(lg3[0], vals) and tok3 == [5]


def test_verify_head_saturated_ties_go_to_lowest_index():
    H = 64
    w = _bias_only_head(np.array([1.0, 384.0, 512.0, 3.0]), H)
    lg, tok, val, margin = O.verify_head(np.ones((1, H)), None, 0.0, w, final_softcap=1.0)
    assert lg[0, 1] == lg[0, 2] == 1.0                  # tanh(384) and tanh(512) round to 1
    # the argmax is taken on the capped logits (the raw maximum is index 2)
    assert tok == [1] and val == [1.0] and margin == [0.0]


def test_verify_head_rows_are_independent_and_normed():
    rng = np.random.default_rng(5)
    H, V = 128, 300
    w = (rng.integers(0, 2 ** 32, size=(V, H // 8), dtype=np.uint64).astype(np.uint32),
         (np.abs(0.02 * rng.standard_normal((V, H // 32))) / 8).astype(np.float32),
         (1e-3 * rng.standard_normal((V, H // 32))).astype(np.float32))
    nw = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    h = rng.standard_normal((3, H))
    lg, tok, _, _ = O.verify_head(h, nw, 0.0, w, 1.5, 30.0)
    for r in range(3):
        one, t1, _, _ = O.verify_head(h[r], nw, 0.0, w, 1.5, 30.0)
        assert np.allclose(one[0], lg[r], rtol=0, atol=1e-12) and t1[0] == tok[r]
    # the final RMSNorm makes every row scale-free (eps = 0)
    scaled, ts, _, _ = O.verify_head(h * np.array([[7.0], [0.01], [-2.0]]), nw, 0.0, w, 1.5, 30.0)
    assert np.allclose(scaled[[0, 1]], lg[[0, 1]], rtol=0, atol=1e-12) and ts[:2] == tok[:2]


# ---------------------------------------------------------------------------
# whole layer and chain
# ---------------------------------------------------------------------------

def _tiny_cfg(**kw):
    base = CONFIGS["tiny_dense"].with_(hidden=64, n_heads=4, n_kv_heads=2, head_dim_qk=32,
                                       head_dim_v=32, intermediate=64, vocab=96, cache_len=5)
    return base.with_(**kw)


def _zero(w):
    q, s, b = w
    return q, np.zeros_like(s), np.zeros_like(b)


def test_layer_reduces_to_projection_and_head():
    cfg = _tiny_cfg()
    w = make_layer_weights(cfg)
    sh = make_shared(cfg)
    st = make_state(cfg)
    step = make_step(cfg)
    w["wo"] = _zero(w["wo"])
    w["ffn_down"] = _zero(w["ffn_down"])
    e = sh["embed"][step["tokens"]]
    res = O.draft_layer(cfg, w, sh["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    cat = np.concatenate([O.rmsnorm(e, w["enorm"], 1e-6), O.rmsnorm(step["hidden"], w["hnorm"], 1e-6)], 1)
    u = cat @ O.dequant(w["eh_proj"]).T
    y = O.rmsnorm(u[-1], w["final_norm"], cfg.eps)
    logits = O.dequant(sh["lm_head"]) @ y
    assert np.allclose(res["u2"], u, rtol=1e-12, atol=1e-12)
    assert np.allclose(res["hidden_out"], y, rtol=1e-12, atol=1e-12)
    assert np.allclose(res["logits"], logits, rtol=1e-12, atol=1e-12)
    assert res["token"] == int(np.argmax(logits))


def test_layer_embedding_comes_first():
    cfg = _tiny_cfg()
    w = make_layer_weights(cfg)
    sh = make_shared(cfg)
    st = make_state(cfg)
    step = make_step(cfg)
    q, s, b = w["eh_proj"]
    s, b = s.copy(), b.copy()
    H = cfg.hidden
    s[:, H // 32:] = 0.0          # columns H..2H (the hidden half) contribute nothing
    b[:, H // 32:] = 0.0
    w["eh_proj"] = (q, s, b)
    e = sh["embed"][step["tokens"]]
    r1 = O.draft_layer(cfg, w, sh["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    r2 = O.draft_layer(cfg, w, sh["lm_head"], st["k_cache"], st["v_cache"], -3 * step["hidden"], e)
    assert np.allclose(r1["u"], r2["u"], rtol=0, atol=1e-14)
    e_n = O.rmsnorm(e, w["enorm"], 1e-6)
    assert np.allclose(r1["u"], e_n @ O.dequant((q[:, :H // 8], s[:, :H // 32], b[:, :H // 32])).T)


def test_layer_attention_single_key_and_gate():
    # Empty cache: the only key is the row itself, so o = v (then gated).
    cfg = _tiny_cfg(cache_len=0, gated_q=True)
    w = make_layer_weights(cfg)
    sh = make_shared(cfg)
    st = make_state(cfg)
    step = make_step(cfg)
    e = sh["embed"][step["tokens"]]
    res = O.draft_layer(cfg, w, sh["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    x = O.rmsnorm(res["u"], w["attn_norm"], cfg.eps)
    qf = (x @ O.dequant(w["wq"]).T).reshape(cfg.n_heads, 2, cfg.head_dim_qk)
    v = (x @ O.dequant(w["wv"]).T).reshape(cfg.n_kv_heads, cfg.head_dim_v)
    o = np.stack([v[h // 2] for h in range(cfg.n_heads)]) * O.sigmoid(qf[:, 1, :])
    u1 = res["u"] + o.reshape(1, -1) @ O.dequant(w["wo"]).T
    assert np.allclose(res["u1"], u1, rtol=1e-12, atol=1e-12)
    # the appended key is normed then rotated at position 0 (identity)
    k = (x @ O.dequant(w["wk"]).T).reshape(cfg.n_kv_heads, cfg.head_dim_qk)
    assert np.allclose(res["k_new"][0], O.rmsnorm(k, w["k_norm"], cfg.eps))


def _hand_rmsnorm(v, w, eps):
    # x / sqrt(mean(x^2) + eps) * w, element by element
    ms = sum(float(t) * float(t) for t in v) / len(v)
    return [float(t) / math.sqrt(ms + eps) * float(wi) for t, wi in zip(v, w)]


def _hand_rope(v, pos, theta, rot):
    # pairs (i, i + rot/2) rotated by pos * theta^(-2i/rot)
    out = [float(t) for t in v]
    half = rot // 2
    for i in range(half):
        ang = pos * theta ** (-2.0 * i / rot)
        a, b = float(v[i]), float(v[i + half])
        out[i] = a * math.cos(ang) - b * math.sin(ang)
        out[i + half] = a * math.sin(ang) + b * math.cos(ang)
    return out


def test_layer_head_norm_comes_before_rope():
    """"hf2q 0.1.13 ... mtp.rs" forward_full_attention: the per-head q/k
    RMSNorm runs first, RoPE on the normed vector after it.  At a position
    p > 0 with a non-uniform norm weight the two orders differ, so the
    appended key pins the order (the query enters the attention the same way)."""
    cfg = _tiny_cfg(cache_len=7)
    w = make_layer_weights(cfg)
    kn = np.asarray(w["k_norm"], np.float64)
    assert np.ptp(kn) > 0.05                      # the weight is not uniform
    sh = make_shared(cfg)
    st = make_state(cfg)
    step = make_step(cfg)
    e = sh["embed"][step["tokens"]]
    res = O.draft_layer(cfg, w, sh["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    x = O.rmsnorm(res["u"], w["attn_norm"], cfg.eps)
    k = (x @ O.dequant(w["wk"]).T).reshape(cfg.n_kv_heads, cfg.head_dim_qk)
    p = cfg.cache_len
    for h in range(cfg.n_kv_heads):
        norm_then_rope = _hand_rope(_hand_rmsnorm(k[h], kn, cfg.eps), p, cfg.rope_theta, cfg.rot_dim)
        rope_then_norm = _hand_rmsnorm(_hand_rope(k[h], p, cfg.rope_theta, cfg.rot_dim), kn, cfg.eps)
        assert np.allclose(res["k_new"][0, h], norm_then_rope, rtol=1e-12, atol=1e-12)
        assert np.max(np.abs(np.subtract(norm_then_rope, rope_then_norm))) > 1e-3


def test_draft_steps_feed_the_normed_hidden():
    """[mtp.rs] forward_draft_with_hidden: the second step reads the first
    step's row after the final norm (written out here), not its pre-norm
    output, and embeds the first step's draft."""
    cfg = _tiny_cfg(cache_len=4)
    w = make_layer_weights(cfg)
    assert np.ptp(np.asarray(w["final_norm"])) > 0.05          # a non-uniform final norm
    sh = make_shared(cfg)
    st = make_state(cfg.with_(m=3))
    step = make_step(cfg)
    embed = lambda t: sh["embed"][t]  # noqa: E731
    res = O.draft_steps(cfg, w, sh["lm_head"], embed, st["k_cache"], st["v_cache"], step["hidden"][0],
                        int(step["tokens"][0]), cfg.cache_len, 2)
    u2 = res[0]["u2"][0]
    ms = sum(float(v) * float(v) for v in u2) / len(u2)
    y1 = [float(v) / math.sqrt(ms + cfg.eps) * float(g) for v, g in zip(u2, w["final_norm"])]
    assert np.allclose(res[0]["hidden_out"], y1, rtol=1e-12, atol=1e-12)
    assert res[1]["token_in"] == res[0]["token"]
    tok1 = res[0]["token"]
    cat = np.concatenate([O.rmsnorm(embed(tok1), w["enorm"], 1e-6), O.rmsnorm(np.array(y1), w["hnorm"], 1e-6)])
    assert np.allclose(res[1]["u"][0], O.dequant(w["eh_proj"]) @ cat, rtol=1e-12, atol=1e-12)
    cat_pre = np.concatenate([O.rmsnorm(embed(tok1), w["enorm"], 1e-6), O.rmsnorm(u2, w["hnorm"], 1e-6)])
    assert np.max(np.abs(O.dequant(w["eh_proj"]) @ cat_pre - res[1]["u"][0])) > 1e-3
    # the second step attends to the first step's appended row at cache row cache_len
    k2 = O.draft_layer(cfg, w, sh["lm_head"], st["k_cache"], st["v_cache"], np.array(y1)[None],
                       embed(tok1)[None], pos0=cfg.cache_len + 1, want_logits=False)
    assert not np.allclose(k2["u1"], res[1]["u1"])             # without that row the output differs


def test_mimo_plan_by_hand():
    """[mimo_mtp.rs] mimo_mtp_draft: the rows each layer runs over two rounds,
    a history gap, a stale state and rounds with nothing to draft."""
    sts = [O.mimo_layer_state_new() for _ in range(3)]
    # first round after a 6-token prompt: t = 5, ids x_0 .. x_6 known
    for l, st in enumerate(sts):
        assert O.mimo_plan_layer(st, l, 5, 0, 6, 7) == 0            # every layer runs 0 .. 5
        O.mimo_commit_layer(st, l, 5, 7)
    assert [st["committed"] for st in sts] == [6, 5, 4] and all(st["kv_len"] == 6 for st in sts)
    # one draft accepted: t = 7, ids up to x_8
    starts = []
    for l, st in enumerate(sts):
        starts.append(O.mimo_plan_layer(st, l, 7, 0, 8, 9))
        assert st["kv_len"] == starts[-1]                            # provisional rows dropped
        O.mimo_commit_layer(st, l, 7, 9)
    assert starts == [6, 5, 4]                                        # 2, 3 and 4 rows
    assert [st["committed"] for st in sts] == [8, 7, 6] and all(st["kv_len"] == 8 for st in sts)
    # a history gap: the history restarts at 20
    st = sts[0]
    assert O.mimo_plan_layer(st, 0, 24, 20, 25, 26) == 20
    assert (st["base"], st["kv_len"], st["committed"]) == (20, 0, 20)
    O.mimo_commit_layer(st, 0, 24, 26)
    assert (st["kv_len"], st["committed"]) == (5, 25)
    # a stale state (committed past t + 1) restarts too
    st2 = {"committed": 40, "base": 20, "kv_len": 21}
    assert O.mimo_plan_layer(st2, 1, 30, 22, 31, 32) == 22 and st2 == {"committed": 22, "base": 22, "kv_len": 0}
    # nothing to draft: t outside the history, or x_{t+1} unknown
    st3 = O.mimo_layer_state_new()
    assert O.mimo_plan_layer(st3, 0, 9, 0, 9, 11) is None
    assert O.mimo_plan_layer(st3, 0, 5, 0, 9, 6) is None and st3 == O.mimo_layer_state_new()


def test_mimo_first_round_equals_the_chain():
    """The first round after a prompt runs every prompt row of every layer;
    its drafts and rows equal the three-layer chain statement ("How the three
    layers chain") with the prompt's rows as the chain's rows."""
    cfg = _tiny_cfg(m=4, n_layers=3, window=3, sinks=True, qk_norm=False, head_dim_qk=48,
                    head_dim_v=32, cache_len=0, rope_theta=1e4)
    layers = [make_layer_weights(cfg, k) for k in range(3)]
    sh = make_shared(cfg)
    embed = lambda t: sh["embed"][t]  # noqa: E731
    rng = np.random.default_rng(31)
    P = cfg.m
    ids = rng.integers(0, cfg.vocab, P + 1).tolist()               # x_0 .. x_P (x_P pending)
    hid = rng.standard_normal((P, cfg.hidden))
    ref = O.draft_chain(cfg, layers, sh["lm_head"], embed,
                        [(np.zeros((cfg.n_kv_heads, P, 48)), np.zeros((cfg.n_kv_heads, P, 32)))] * 3,
                        hid, ids[1:])
    caches = [[np.zeros((cfg.n_kv_heads, P, 48)), np.zeros((cfg.n_kv_heads, P, 32))] for _ in range(3)]
    states = [O.mimo_layer_state_new() for _ in range(3)]
    drafts, res = O.mimo_draft_round(cfg, layers, sh["lm_head"], embed, caches, states,
                                     lambda j: hid[j], 0, P, P - 1, ids, 3)
    assert drafts == [r["token"] for r in ref]
    for l in range(3):
        assert np.allclose(res[l]["u2"], ref[l]["u2"], rtol=1e-12, atol=1e-12)
        assert np.allclose(caches[l][0].transpose(1, 0, 2), ref[l]["k_new"], rtol=1e-12, atol=1e-12)


def test_chain_rows_take_earlier_drafts():
    cfg = _tiny_cfg(m=4, n_layers=3, window=3, sinks=True, qk_norm=False, head_dim_qk=48,
                    cache_len=6, name="tiny_chain")
    layers = [make_layer_weights(cfg, k) for k in range(3)]
    sh = make_shared(cfg)
    caches = [(make_state(cfg, k)["k_cache"], make_state(cfg, k)["v_cache"]) for k in range(3)]
    step = make_step(cfg)
    embed = lambda t: sh["embed"][t]  # noqa: E731
    res = O.draft_chain(cfg, layers, sh["lm_head"], embed, caches, step["hidden"], step["tokens"])
    seq = list(step["tokens"]) + [r["token"] for r in res]
    for k in range(3):
        assert res[k]["tokens_in"] == seq[k: k + 4]
        e = sh["embed"][seq[k: k + 4]]
        alone = O.draft_layer(cfg, layers[k], sh["lm_head"], *caches[k], step["hidden"], e)
        assert alone["token"] == res[k]["token"]
    forced = [5, 7, None]
    res2 = O.draft_chain(cfg, layers, sh["lm_head"], embed, caches, step["hidden"], step["tokens"],
                         forced)
    assert res2[1]["tokens_in"][-1] == 5 and res2[2]["tokens_in"][-2:] == [5, 7]


# ---------------------------------------------------------------------------
# speculation bookkeeping (hand-worked rounds)
# ---------------------------------------------------------------------------

def test_spec_accept_prefix_by_hand():
    assert O.spec_accept([5, 7, 9], [5, 7, 1, 3]) == 2   # third draft rejected
    assert O.spec_accept([5, 7, 9], [4, 7, 9, 3]) == 0   # first draft rejected: nothing later counts
    assert O.spec_accept([5, 7, 9], [5, 7, 9, 0]) == 3   # all drafts; row k is the bonus token
    assert O.spec_accept([], [11]) == 0


def test_spec_stats_by_hand():
    st = O.spec_stats_new()
    for k, a in [(3, 2), (3, 0), (3, 3)]:
        O.spec_note_round(st, k, a, draft_ns=10, verify_ns=100)
    assert (st["rounds"], st["drafted"], st["accepted"]) == (3, 9, 5)
    assert st["accept_hist"] == [1, 0, 1, 1]
    assert st["depth_drafted"] == [3, 3, 3] and st["depth_accepted"] == [2, 2, 1]
    assert (st["draft_ns"], st["verify_ns"]) == (30, 300)
    assert O.spec_tokens_per_round(st) == 8 / 3           # 5 accepted + 3 own tokens over 3 rounds
    # a deeper round grows the histogram and the depth lists
    st2 = O.spec_note_round(O.spec_note_round(O.spec_stats_new(), 1, 1), 4, 2)
    assert st2["accept_hist"] == [0, 1, 1, 0, 0]
    assert st2["depth_drafted"] == [2, 1, 1, 1] and st2["depth_accepted"] == [2, 1, 0, 0]
    assert O.spec_tokens_per_round(O.spec_stats_new()) == 0.0


def test_spec_stats_invariants():
    rng = np.random.default_rng(3)
    st = O.spec_stats_new()
    for _ in range(200):
        k = int(rng.integers(0, 6))
        O.spec_note_round(st, k, int(rng.integers(0, k + 1)))
    hist = st["accept_hist"]
    assert sum(hist) == st["rounds"]
    assert sum(a * n for a, n in enumerate(hist)) == st["accepted"]
    assert sum(st["depth_accepted"]) == st["accepted"] and sum(st["depth_drafted"]) == st["drafted"]
    assert 1.0 <= O.spec_tokens_per_round(st) <= 6.0


def test_spec_rewind_by_hand():
    assert O.spec_rewind([10, 12, 7], 9) == [9, 9, 7]
    assert O.spec_rewind([10, 12, 7], 20) == [10, 12, 7]
    assert O.spec_rewind([10, 12, 7], 0) == [0, 0, 0]


# ---------------------------------------------------------------------------
# KV catch-up of a target batch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("qk_norm", [True, False])
def test_kv_catch_up_rows_equal_draft_steps(qk_norm):
    """Row i of the catch-up is the K/V row a one-row draft step appends for
    the same embedding, the shifted target hidden and position pos0 + i
    (computed there together with attention, FFN and head)."""
    cfg = _tiny_cfg(qk_norm=qk_norm)
    w = make_layer_weights(cfg)
    rng = np.random.default_rng(21)
    seq, pos0, H = 4, 6, cfg.hidden
    e = rng.standard_normal((seq, H))
    t = rng.standard_normal((seq, H))
    pend = rng.standard_normal(H)
    k, v = O.kv_catch_up(cfg, w, e, t, pending_hidden=pend, pos0=pos0)
    lm = w["eh_proj"]  # any weight serves as a head here; only the K/V rows are compared
    shifted = [pend] + [t[i - 1] for i in range(1, seq)]
    for i in range(seq):
        kc = np.zeros((cfg.n_kv_heads, pos0 + i + 1, cfg.head_dim_qk))
        vc = np.zeros((cfg.n_kv_heads, pos0 + i + 1, cfg.head_dim_v))
        one = O.draft_layer(cfg, w, lm, kc, vc, shifted[i], e[i], pos0=pos0 + i, want_logits=False)
        assert np.allclose(k[i], one["k_new"][0], rtol=0, atol=1e-12)
        assert np.allclose(v[i], one["v_new"][0], rtol=0, atol=1e-12)


def test_kv_catch_up_shift_and_cold_prompt():
    cfg = _tiny_cfg()
    w = make_layer_weights(cfg)
    rng = np.random.default_rng(22)
    seq, H = 5, cfg.hidden
    e = rng.standard_normal((seq, H))
    t = rng.standard_normal((seq, H))
    # a cold prompt's first row reads a zero hidden
    k0, v0 = O.kv_catch_up(cfg, w, e, t)
    kz, vz = O.kv_catch_up(cfg, w, e, t, pending_hidden=np.zeros(H))
    assert np.array_equal(k0, kz) and np.array_equal(v0, vz)
    # splitting the batch: the second part's pending hidden is the last target row of the first
    k1, v1 = O.kv_catch_up(cfg, w, e[:2], t[:2], pos0=0)
    k2, v2 = O.kv_catch_up(cfg, w, e[2:], t[2:], pending_hidden=t[1], pos0=2)
    assert np.allclose(np.concatenate([k1, k2]), k0, rtol=0, atol=1e-12)
    assert np.allclose(np.concatenate([v1, v2]), v0, rtol=0, atol=1e-12)
    # the last target row is never read (it belongs to the next batch)
    t2 = t.copy()
    t2[-1] += 100.0
    k3, _ = O.kv_catch_up(cfg, w, e, t2)
    assert np.array_equal(k3, k0)


# ---------------------------------------------------------------------------
# BF16 scales and biases of the expert stacks
# ---------------------------------------------------------------------------

def test_bf16_round_halfway_cases_by_hand():
    u = 2.0 ** -7  # spacing of bfloat16 at 1.0 (7 stored mantissa bits)
    assert O.bf16_round([1.0, -3.0, 0.5, 2.0 ** -10, 0.0])[:4].tolist() == [1.0, -3.0, 0.5, 2.0 ** -10]
    assert O.bf16_round(1 + u / 2)[()] == 1.0                 # halfway, 1.0 is even: down
    assert O.bf16_round(1 + 3 * u / 2)[()] == 1 + 2 * u       # halfway, 1 + u is odd: up
    assert O.bf16_round(1 + u / 2 + 2.0 ** -20)[()] == 1 + u  # just above halfway: up
    assert O.bf16_round(-(1 + u / 2 + 2.0 ** -20))[()] == -(1 + u)


def test_bf16_round_matches_library_conversion_and_bound():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ours = O.bf16_round(x)
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, lib)
    assert np.max(np.abs(ours - x) / np.abs(x.astype(np.float64))) <= 2.0 ** -8


def test_moe_stack_bf16_keeps_codes_and_rounds_only_scales():
    rng = np.random.default_rng(32)
    q = rng.integers(0, 2 ** 32, size=(6, 8), dtype=np.uint64).astype(np.uint32)
    s = (np.abs(0.02 * rng.standard_normal((6, 2))) / 8).astype(np.float32)
    b = (-8 * s + 1e-3 * rng.standard_normal((6, 2))).astype(np.float32)
    q2, s2, b2 = O.moe_stack_bf16((q, s, b))
    assert q2 is q and np.array_equal(s2, O.bf16_round(s)) and np.array_equal(b2, O.bf16_round(b))
    # exactly representable scales and biases: the dequantised matrix is unchanged
    se, be = O.bf16_round(s).astype(np.float32), O.bf16_round(b).astype(np.float32)
    assert np.array_equal(O.dequant(O.moe_stack_bf16((q, se, be))), O.dequant((q, se, be)))
