"""CPU oracle of the MTP draft-layer forward (test infrastructure only).

Plain, slow float64 numpy restatement of what the draft layer computes.  It
exists to check the CUDA path: only the tests, the smoke check and the
benchmark's CPU-baseline leg use it, and it shares no code with the CUDA
path.  Every step follows the passage it cites; steps the pages leave open
take the reading stated in the function's docstring.

Pages cited (by title and item):
  [mtp.rs]        hf2q 0.1.13 src/inference/models/qwen35/mtp.rs
  [mimo_mtp.rs]   cortiq-engine 0.8.49 src/mimo_mtp.rs
  [shared.rs]     hf2q 0.1.1 src/serve/forward_mlx_shared.rs

Weights are mlx-affine 4-bit, group 32: ``q`` uint32 ``[N, K/8]``, ``s`` and
``b`` float32 ``[N, K/32]``, element ``w[n, k] = s[n, k//32] * code + b[n,
k//32]`` with the code of column ``k`` in bits ``4*(k%8) .. 4*(k%8)+3`` of
word ``k//8``.
"""

from __future__ import annotations

import numpy as np

GROUP = 32
PACK = 8
_ROW_CHUNK = 8192


# ---------------------------------------------------------------------------
# Quantised weights
# ---------------------------------------------------------------------------

def unpack_codes(q: np.ndarray) -> np.ndarray:
    """Integer codes ``[N, K]`` of a packed weight.

    [shared.rs] ``MlxQWeight::from_mlx_affine_linear``: the code for column
    ``8*kp + j`` sits at bits ``4*j .. 4*j+3`` of word ``kp`` (low nibble at
    slot 0).
    """
    q = np.asarray(q, dtype=np.uint32)
    n, kw = q.shape
    shifts = (4 * np.arange(PACK, dtype=np.uint32))[None, None, :]
    codes = (q[:, :, None] >> shifts) & np.uint32(0xF)
    return codes.reshape(n, kw * PACK).astype(np.int64)


def dequant(w) -> np.ndarray:
    """Dense float64 ``[N, K]`` matrix ``s * code + b`` of an affine weight ``(q, s, b)``.

    [shared.rs] ``MlxAffineExtra`` (per-group scales and biases ``[N,
    K/group_size]``, bits 4, group 32) and the CPU reference in test
    ``from_mlx_affine_linear_roundtrips_through_packed_kernel``
    (``q * s + b`` per element).
    """
    q, s, b = w
    codes = unpack_codes(q).astype(np.float64)
    n, k = codes.shape
    if k % GROUP:
        raise ValueError("K must be a multiple of the group size 32")
    s64 = np.repeat(np.asarray(s, dtype=np.float64), GROUP, axis=1)
    b64 = np.repeat(np.asarray(b, dtype=np.float64), GROUP, axis=1)
    if s64.shape != (n, k) or b64.shape != (n, k):
        raise ValueError("scale/bias shape does not match [N, K/32]")
    return codes * s64 + b64


def bf16_round(x) -> np.ndarray:
    """float32 values rounded to bfloat16 (kept as float64).

    [shared.rs] ``MlxAffineMoeStack``: the expert stacks hold their scales
    and biases as BF16, cast from the float32 per-expert values at upload.
    Reading (the cast itself is not on the pages): round to nearest, ties
    to even, on the top 16 bits of the float32 pattern.
    """
    bits = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = bits >> np.uint64(16)
    rest = bits & np.uint64(0xFFFF)
    up = (rest > np.uint64(0x8000)) | ((rest == np.uint64(0x8000)) & ((keep & np.uint64(1)) == np.uint64(1)))
    keep = keep + up.astype(np.uint64)
    return (keep << np.uint64(16)).astype(np.uint32).view(np.float32).astype(np.float64)


def moe_stack_bf16(w):
    """An expert stack ``(q, s, b)`` as [shared.rs] ``MlxAffineMoeStack``
    stores it: the same codes, scales and biases rounded to BF16."""
    q, s, b = w
    return q, bf16_round(s), bf16_round(b)


def weight_shape(w):
    q, _, _ = w
    return q.shape[0], q.shape[1] * PACK


def qmatmul(x: np.ndarray, w, rows=None) -> np.ndarray:
    """``y[r, n] = sum_k x[r, k] * w[n, k]`` for an affine weight, in float64.

    [shared.rs] ``dispatch_qmatmul`` affine branch: ``y[m, N] = x[m, K] *
    W^T`` with ``W`` dequantised per element.  Output rows are independent
    dot products, so the matrix is dequantised a slab of rows at a time (or
    only ``rows``) to bound memory; no sum is split or reordered.
    """
    q, s, b = w
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    n, k = weight_shape(w)
    if x.shape[1] != k:
        raise ValueError(f"x has {x.shape[1]} columns, weight has K={k}")
    sel = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((x.shape[0], len(sel)), dtype=np.float64)
    for lo in range(0, len(sel), _ROW_CHUNK):
        r = sel[lo: lo + _ROW_CHUNK]
        wd = dequant((q[r], s[r], b[r]))
        out[:, lo: lo + len(r)] = x @ wd.T
    return out


# ---------------------------------------------------------------------------
# Normalisation, activations, rotary embedding
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """``x / sqrt(mean(x^2) + eps) * w`` over the last axis.

    [mtp.rs] ``rms_norm_with_weight`` / ``dispatch_rms_norm`` (params
    ``[eps, dim]``); [mimo_mtp.rs] ``inference::rms_norm_into``.  Reading:
    the weight multiplies directly (no ``1 + w``).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    """``z * sigmoid(z)`` ([mimo_mtp.rs] ``Act::Silu`` of the dense MLP)."""
    return np.asarray(z, dtype=np.float64) * sigmoid(z)


def rope(x: np.ndarray, pos: int, theta: float, rot_dim: int) -> np.ndarray:
    """Rotary embedding of one position over the last axis (half-split pairs).

    [mtp.rs] ``apply_imrope`` with four equal text position ids; reading:
    for text tokens this is 1-D RoPE at position ``pos``, rotating the pair
    ``(x[i], x[i + R/2])`` by ``pos * theta^(-2i/R)`` for ``i < R/2`` with
    ``R = rot_dim``; dimensions past ``R`` pass through.
    """
    x = np.asarray(x, dtype=np.float64)
    half = rot_dim // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / rot_dim)
    c, s = np.cos(ang), np.sin(ang)
    out = x.copy()
    a = x[..., :half]
    bb = x[..., half:rot_dim]
    out[..., :half] = a * c - bb * s
    out[..., half:rot_dim] = a * s + bb * c
    return out


# ---------------------------------------------------------------------------
# Attention over the layer's own cache
# ---------------------------------------------------------------------------

def attention(q, k_all, v_all, q_pos, window=0, sinks=None, scale=None):
    """Causal decode attention with an optional sliding window and sink logits.

    ``q``: ``[m, nh, dqk]`` (already normed and rotated); ``k_all``/``v_all``:
    ``[nkv, T, d]`` key/value rows at positions ``0 .. T-1``; ``q_pos[r]``
    is the position of query row ``r``.

    [mtp.rs] ``apply_sdpa_with_kv_cache`` (append then causal SDPA, grouped
    KV heads) and [mimo_mtp.rs] module doc / ``qwen_attention_batch`` (window
    128, per-head sinks).  Readings: query head ``h`` uses KV head
    ``h // (nh/nkv)``; ``scale = 1/sqrt(dqk)``; the row at position ``p``
    sees keys ``j`` with ``p - W < j <= p`` (all ``j <= p`` when ``W <=
    0``); a sink is one extra logit per head, not scaled, that enters the
    softmax denominator only.
    """
    q = np.asarray(q, dtype=np.float64)
    k_all = np.asarray(k_all, dtype=np.float64)
    v_all = np.asarray(v_all, dtype=np.float64)
    m, nh, dqk = q.shape
    nkv = k_all.shape[0]
    group = nh // nkv
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    out = np.zeros((m, nh, v_all.shape[2]), dtype=np.float64)
    for r in range(m):
        p = int(q_pos[r])
        lo = 0 if window <= 0 else max(0, p - window + 1)
        for h in range(nh):
            kv = h // group
            keys = k_all[kv, lo: p + 1]
            vals = v_all[kv, lo: p + 1]
            logits = scale * (keys @ q[r, h])
            big = logits.max()
            if sinks is not None:
                big = max(big, float(sinks[h]))
            e = np.exp(logits - big)
            denom = e.sum()
            if sinks is not None:
                denom += np.exp(float(sinks[h]) - big)
            out[r, h] = (e @ vals) / denom
    return out


# ---------------------------------------------------------------------------
# Feed-forward blocks
# ---------------------------------------------------------------------------

def swiglu(f, gate_w, up_w, down_w):
    """``W_down (silu(W_gate f) * (W_up f))`` ([mtp.rs] ``build_dense_ffn_layer_gpu_q``)."""
    g = qmatmul(f, gate_w)
    u = qmatmul(f, up_w)
    return qmatmul(silu(g) * u, down_w)


def topk_lowest_index(p: np.ndarray, k: int) -> np.ndarray:
    """Indices of the ``k`` largest entries; ties go to the lower index."""
    order = sorted(range(len(p)), key=lambda i: (-p[i], i))
    return np.array(order[:k], dtype=np.int64)


def moe_route(f_row, router, top_k):
    """Router of the MoE FFN for one row: ``(experts, weights)``.

    [mtp.rs] ``MtpFfnWeightsGpu::Moe`` (router ``ffn_gate_inp``).  Reading:
    softmax over all experts' logits ``router @ f``, keep the ``top_k``
    largest (ties to the lower index), renormalise the kept weights to sum 1.
    """
    logits = np.asarray(router, dtype=np.float64) @ np.asarray(f_row, dtype=np.float64)
    p = np.exp(logits - logits.max())
    p /= p.sum()
    sel = topk_lowest_index(p, top_k)
    wsel = p[sel] / p[sel].sum()
    return sel, wsel


def moe_ffn(f, w, cfg):
    """Routed experts plus a gated shared expert, per row ``f[r]``.

    [mtp.rs] ``MtpFfnWeightsGpu::Moe`` (8 tensors: router, stacked expert
    gate/up/down, and four shared-expert tensors) and
    ``build_moe_ffn_layer_gpu_q_into``; [shared.rs] ``MlxAffineMoeStack``
    (expert ``e`` of a stack is slab ``[e]`` of ``[E, N, K/8]``).  Reading:
    ``sum_e p_e * SwiGLU_e(f) + sigmoid(w_sg . f) * SwiGLU_shared(f)``.
    """
    f = np.atleast_2d(np.asarray(f, dtype=np.float64))
    out = np.zeros((f.shape[0], cfg.hidden), dtype=np.float64)
    eg, eu, ed = w["exp_gate"], w["exp_up"], w["exp_down"]
    for r in range(f.shape[0]):
        sel, wsel = moe_route(f[r], w["router"], cfg.top_k)
        acc = np.zeros(cfg.hidden, dtype=np.float64)
        for e, pe in zip(sel, wsel):
            ex = lambda t: (t[0][e], t[1][e], t[2][e])  # noqa: E731
            acc += pe * swiglu(f[r], ex(eg), ex(eu), ex(ed))[0]
        gate = sigmoid(np.asarray(w["sh_gate_inp"], dtype=np.float64) @ f[r])
        acc += gate * swiglu(f[r], w["sh_gate"], w["sh_up"], w["sh_down"])[0]
        out[r] = acc
    return out


# ---------------------------------------------------------------------------
# Greedy head
# ---------------------------------------------------------------------------

def argmax_lowest(v: np.ndarray):
    """``(index, value, top-2 margin)``; ties go to the lowest index.

    [mtp.rs] ``forward_shared_head_greedy`` (argmax over the vocabulary
    logits, returning index and value).
    """
    v = np.asarray(v, dtype=np.float64)
    idx = int(np.argmax(v))  # numpy returns the first maximal index
    val = float(v[idx])
    rest = np.delete(v, idx)
    margin = float(val - rest.max()) if rest.size else float("inf")
    return idx, val, margin


def verify_head(hidden_rows, norm_w, eps, lm_head, logit_multiplier=None, final_softcap=None):
    """Batched verify head: ``(logits [b, V], tokens, values, margins)``.

    [mimo_mtp.rs] ``mimo_verify_head_rows``: every row of ``hidden_rows``
    (the pending token's and the drafts' hidden rows) goes through the final
    RMSNorm (skipped when ``norm_w`` is None), the lm_head projection, then
    the optional logit multiplier (``l * m``) and after it the optional final
    softcap (``c * tanh(l / c)``).  ``mimo_spec_round`` then samples each
    row; greedy sampling is the argmax with ties to the lowest index
    (``argmax_lowest``).
    """
    h = np.atleast_2d(np.asarray(hidden_rows, dtype=np.float64))
    x = h if norm_w is None else np.stack([rmsnorm(row, norm_w, eps) for row in h])
    logits = qmatmul(x, lm_head)
    if logit_multiplier is not None:
        logits = logits * float(logit_multiplier)
    if final_softcap is not None:
        c = float(final_softcap)
        logits = c * np.tanh(logits / c)
    picks = [argmax_lowest(row) for row in logits]
    return (logits, [t for t, _, _ in picks], [v for _, v, _ in picks],
            [mg for _, _, mg in picks])


# ---------------------------------------------------------------------------
# One draft layer
# ---------------------------------------------------------------------------

def draft_layer(cfg, w, lm_head, k_cache, v_cache, hidden, embed_rows, pos0=None,
                want_logits=True, pos_base=0):
    """One MTP draft-layer step over ``m`` rows.

    Follows [mimo_mtp.rs] module doc (the four-line layer statement) with
    the step order of [mtp.rs] ``forward_draft_body``:

    1. ``project_embedding_and_hidden``: ``e_n = RMSNorm(e) * enorm``,
       ``h_n = RMSNorm(h) * hnorm`` (eps 1e-6), ``u = eh_proj [e_n ; h_n]``
       (embedding first).
    2. ``forward_full_attention``: ``x = RMSNorm(u) * attn_norm``; ``q``
       (and, when gated, ``gate``), ``k``, ``v`` projections; per-head q/k
       RMSNorm with a ``[dqk]`` weight when present; RoPE at position
       ``pos0 + r``; append ``k``, ``v`` to the cache; attention; ``o *=
       sigmoid(gate)`` when gated; ``u1 = u + W_o o``.  Reading for the gated
       projection: ``W_q`` has ``2*nh*dqk`` rows, head ``h`` owning rows
       ``[2*h*dqk, 2*h*dqk + dqk)`` for the query and the next ``dqk`` rows
       for its gate.
    3. ``forward_ffn_residual``: ``f = RMSNorm(u1) * post_norm``; ``u2 = u1
       + FFN(f)``.
    4. ``forward_shared_head_greedy`` on the last row ([mimo_mtp.rs]
       ``mimo_mtp_draft``: only row ``n-1`` reaches the head): ``y =
       RMSNorm(u2[-1]) * final_norm``, logits ``= lm_head y``, token =
       argmax.  ``y`` is also the hidden a chained step consumes ([mtp.rs]
       ``forward_draft_with_hidden``).

    ``k_cache``/``v_cache`` are ``[nkv, cap, d]`` with rows ``< pos0``
    filled; they are not modified (the appended rows are returned).  Cache
    row ``i`` holds position ``pos_base + i`` (a cache restarted part-way,
    [mimo_mtp.rs] ``base``): new row ``r`` rotates at ``pos_base + pos0 +
    r``; the causal mask and the window compare row indices, which differ
    from positions by the same ``pos_base``.
    """
    eps = cfg.eps
    H, nh, nkv, dqk, dv = cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v
    hidden = np.atleast_2d(np.asarray(hidden, dtype=np.float64))
    embed_rows = np.atleast_2d(np.asarray(embed_rows, dtype=np.float64))
    m = hidden.shape[0]
    L = cfg.cache_len if pos0 is None else pos0

    # 1. embedding / hidden projection
    e_n = rmsnorm(embed_rows, w["enorm"], 1e-6)
    h_n = rmsnorm(hidden, w["hnorm"], 1e-6)
    u = qmatmul(np.concatenate([e_n, h_n], axis=1), w["eh_proj"])

    # 2. attention
    x = rmsnorm(u, w["attn_norm"], eps)
    qf = qmatmul(x, w["wq"])
    if cfg.gated_q:
        qg = qf.reshape(m, nh, 2, dqk)
        q, gate = qg[:, :, 0, :], qg[:, :, 1, :]
    else:
        q, gate = qf.reshape(m, nh, dqk), None
    k = qmatmul(x, w["wk"]).reshape(m, nkv, dqk)
    v = qmatmul(x, w["wv"]).reshape(m, nkv, dv)
    if cfg.qk_norm:
        q = rmsnorm(q, w["q_norm"], eps)
        k = rmsnorm(k, w["k_norm"], eps)
    q = np.stack([rope(q[r], pos_base + L + r, cfg.rope_theta, cfg.rot_dim) for r in range(m)])
    k = np.stack([rope(k[r], pos_base + L + r, cfg.rope_theta, cfg.rot_dim) for r in range(m)])
    k_all = np.concatenate([np.asarray(k_cache, np.float64)[:, :L], k.transpose(1, 0, 2)], axis=1)
    v_all = np.concatenate([np.asarray(v_cache, np.float64)[:, :L], v.transpose(1, 0, 2)], axis=1)
    o = attention(q, k_all, v_all, [L + r for r in range(m)], cfg.window,
                  w.get("sinks") if cfg.sinks else None)
    if gate is not None:
        o = o * sigmoid(gate)
    u1 = u + qmatmul(o.reshape(m, nh * dv), w["wo"])

    # 3. FFN
    f = rmsnorm(u1, w["post_norm"], eps)
    if cfg.moe:
        u2 = u1 + moe_ffn(f, w, cfg)
    else:
        u2 = u1 + swiglu(f, w["ffn_gate"], w["ffn_up"], w["ffn_down"])

    # 4. greedy shared head on the last row
    y = rmsnorm(u2[-1], w["final_norm"], eps)
    out = {"u": u, "u1": u1, "u2": u2, "hidden_out": y, "k_new": k, "v_new": v,
           "q_roped": q, "attn": o}
    if want_logits:
        logits = qmatmul(y[None, :], lm_head)[0]
        tok, val, margin = argmax_lowest(logits)
        out.update(logits=logits, token=tok, value=val, margin=margin)
    return out


def kv_catch_up(cfg, w, embed_rows, target_hidden, pending_hidden=None, pos0=0):
    """KV catch-up of a target batch: ``(k_new [seq, nkv, dqk], v_new [seq, nkv, dv])``.

    [mtp.rs] ``process_target_batch``: the target's hidden rows are used
    shifted one row right (row 0 is the pending hidden, or zeros for a cold
    prompt; row ``i > 0`` is target row ``i - 1``), projected with the
    embedding rows by ``project_embedding_and_hidden``, then
    ``append_attention_kv``: attention RMSNorm, the ``W_k`` and ``W_v``
    projections, per-head k RMSNorm (when the layer has it), RoPE at each
    row's position, and the rows go to the cache at ``pos0 + i``.  Nothing
    else runs (no attention, FFN or logits).  Reading: the text rows' four
    rotary position ids are equal, so the rotation is the 1-D RoPE at
    ``pos0 + i``, as in the draft step.
    """
    eps = cfg.eps
    nkv, dqk, dv = cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v
    e = np.atleast_2d(np.asarray(embed_rows, dtype=np.float64))
    t = np.atleast_2d(np.asarray(target_hidden, dtype=np.float64))
    seq = e.shape[0]
    assert t.shape == e.shape and seq > 0
    shifted = np.zeros_like(t)
    if pending_hidden is not None:
        shifted[0] = np.asarray(pending_hidden, dtype=np.float64)
    shifted[1:] = t[:-1]
    e_n = rmsnorm(e, w["enorm"], 1e-6)
    h_n = rmsnorm(shifted, w["hnorm"], 1e-6)
    u = qmatmul(np.concatenate([e_n, h_n], axis=1), w["eh_proj"])
    x = rmsnorm(u, w["attn_norm"], eps)
    k = qmatmul(x, w["wk"]).reshape(seq, nkv, dqk)
    v = qmatmul(x, w["wv"]).reshape(seq, nkv, dv)
    if cfg.qk_norm:
        k = rmsnorm(k, w["k_norm"], eps)
    k = np.stack([rope(k[i], pos0 + i, cfg.rope_theta, cfg.rot_dim) for i in range(seq)])
    return k, v


def draft_steps(cfg, w, lm_head, embed, k_cache, v_cache, hidden, token, cache_len, k_steps,
                pos_base=0, forced=None):
    """``k_steps`` chained one-row draft steps of one layer.

    [mtp.rs] ``forward_draft_with_hidden``: a chained step reads the normed
    row the shared head returns (after ``shared_head_norm``), "the only valid
    input for a chained second MTP step", and the draft token of the step
    before.  Step ``i`` appends its K/V row at cache row ``cache_len + i``
    (position ``pos_base + cache_len + i``).  ``forced[i]``, when given,
    replaces draft ``i`` as the next step's token (near-ties).  Returns the
    steps' results; the caches are not modified.
    """
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    h = np.asarray(hidden, dtype=np.float64).reshape(1, -1)
    tok = int(token)
    out = []
    for i in range(k_steps):
        L = cache_len + i
        res = draft_layer(cfg, w, lm_head, kc, vc, h, embed(tok)[None], pos0=L, pos_base=pos_base)
        kc[:, L] = res["k_new"][0]
        vc[:, L] = res["v_new"][0]
        res["token_in"] = tok
        out.append(res)
        tok = res["token"] if forced is None or forced[i] is None else int(forced[i])
        h = res["hidden_out"][None]
    return out


def draft_chain(cfg, layers, lm_head, embed, caches, hidden, tokens, forced=None):
    """The three-layer chained draft of one speculative round.

    [mimo_mtp.rs] module doc ("How the three layers chain") and
    ``mimo_mtp_draft``: layer ``k`` takes the same target hiddens ``h_j``
    for every layer; its row ``i`` embeds token ``seq[i + k]`` where ``seq``
    is the known tokens followed by this round's drafts; the draft of layer
    ``k`` is the argmax of its last row.  ``embed(tok)`` returns one
    embedding row.  ``forced[k]``, when given, replaces draft ``k`` for the
    later layers (used when a near-tie allows either token).
    """
    m = cfg.m
    seq = [int(t) for t in tokens]
    results = []
    for k, (w, (kc, vc)) in enumerate(zip(layers, caches)):
        toks = seq[k: k + m]
        e = np.stack([embed(t) for t in toks])
        res = draft_layer(cfg, w, lm_head, kc, vc, hidden, e)
        res["tokens_in"] = toks
        results.append(res)
        nxt = res["token"] if forced is None or forced[k] is None else int(forced[k])
        seq.append(nxt)
    return results


# ---------------------------------------------------------------------------
# Speculation bookkeeping (host)
# ---------------------------------------------------------------------------

def mimo_layer_state_new():
    """One draft layer's round state of [mimo_mtp.rs] ``MimoMtp``: rows at
    positions below ``committed`` are final, ``base`` is the position of the
    cache's first row, ``kv_len`` the rows the cache holds."""
    return {"committed": 0, "base": 0, "kv_len": 0}


def mimo_plan_layer(st, layer, t, hist_lo, hist_end, ids_len):
    """First position the layer runs this round (rows ``start .. t``), or None.

    [mimo_mtp.rs] ``mimo_mtp_draft`` for a round that starts after the
    backbone processed position ``t``: nothing is drafted when the hidden
    history ``[hist_lo, hist_end)`` lacks ``t`` or fewer than ``t + 2`` ids
    are known.  A layer whose committed position lies below the history
    (a gap) or beyond ``t + 1`` (stale) restarts its cache at ``hist_lo``;
    then the rows of the previous round that were provisional (past
    ``committed``) are dropped, and the layer runs positions
    ``committed .. t``.
    """
    if hist_end <= hist_lo or t < hist_lo or t >= hist_end or ids_len < t + 2:
        return None
    if st["committed"] < hist_lo or st["committed"] > t + 1:
        st["kv_len"] = 0
        st["base"] = hist_lo
        st["committed"] = hist_lo
    keep = st["committed"] - st["base"]
    if st["kv_len"] > keep:
        st["kv_len"] = keep
    return st["committed"]


def mimo_commit_layer(st, layer, t, ids_len):
    """After the layer ran positions ``start .. t`` ([mimo_mtp.rs]
    ``mimo_mtp_draft``): the cache holds rows up to ``t``, and rows whose
    token is known (row ``j`` embeds ``ids[j + layer + 1]``) are final."""
    st["kv_len"] = t + 1 - st["base"]
    real_end = min(t + 1, max(0, ids_len - (layer + 1)))
    st["committed"] = max(st["committed"], real_end)
    return st


def mimo_draft_round(cfg, layers, lm_head, embed, caches, states, hist, hist_lo, hist_end, t, ids,
                     k, forced=None):
    """The draft half of one MiMo round ([mimo_mtp.rs] ``mimo_mtp_draft``).

    Layer ``l`` runs positions ``start .. t`` (``mimo_plan_layer``): row ``j``
    embeds ``ids[j + l + 1]`` (this round's earlier drafts past the known
    ids) and reads the target hidden ``hist(j)``; only the last row reaches
    the head and its argmax is draft ``l``.  ``caches[l]`` is ``[kc, vc]``
    (arrays ``[nkv, cap, d]``, updated in place).  ``forced[l]`` replaces
    draft ``l`` for the later layers (near-ties).  Returns the drafts and the
    layers' results.
    """
    drafts, results = [], []
    for layer in range(min(k, len(layers))):
        st = states[layer]
        start = mimo_plan_layer(st, layer, t, hist_lo, hist_end, len(ids))
        if start is None:
            return [], []
        rows = list(range(start, t + 1))
        toks = [ids[j + layer + 1] if j + layer + 1 < len(ids) else drafts[j + layer + 1 - len(ids)]
                for j in rows]
        e = np.stack([embed(tk) for tk in toks])
        h = np.stack([hist(j) for j in rows])
        kc, vc = caches[layer]
        L = st["kv_len"]
        res = draft_layer(cfg, layers[layer], lm_head, kc, vc, h, e, pos0=L, pos_base=st["base"])
        kc[:, L:L + len(rows)] = res["k_new"].transpose(1, 0, 2)
        vc[:, L:L + len(rows)] = res["v_new"].transpose(1, 0, 2)
        mimo_commit_layer(st, layer, t, len(ids))
        res["start"] = start
        results.append(res)
        drafts.append(res["token"] if forced is None or forced[layer] is None else int(forced[layer]))
    return drafts, results

def spec_accept(drafts, verify_tokens):
    """Accepted drafts of one round.

    [mimo_mtp.rs] ``mimo_spec_round``: walking the rows ``i = 0..=k`` of the
    batched verify, the verifier's token at row ``i`` is compared with draft
    ``i``; an equal token accepts the draft and the walk goes on, the first
    unequal one (or row ``k``, which has no draft) ends it.
    """
    a = 0
    for i in range(len(drafts) + 1):
        if i < len(drafts) and int(verify_tokens[i]) == int(drafts[i]):
            a += 1
        else:
            break
    return a


def spec_stats_new():
    """[mimo_mtp.rs] ``MtpStats`` with every counter at zero."""
    return {"rounds": 0, "drafted": 0, "accepted": 0, "accept_hist": [], "depth_drafted": [],
            "depth_accepted": [], "draft_ns": 0, "verify_ns": 0}


def spec_note_round(st, k, a, draft_ns=0, verify_ns=0):
    """Counter updates at the end of [mimo_mtp.rs] ``mimo_spec_round``.

    One more round, ``k`` more drafts, ``a`` more accepted; the histogram
    grows to ``k + 1`` bins and counts ``a``; the per-depth lists grow to
    ``k`` entries, every depth below ``k`` was drafted and every depth below
    ``a`` was accepted.
    """
    st["draft_ns"] += draft_ns
    st["verify_ns"] += verify_ns
    st["rounds"] += 1
    st["drafted"] += k
    st["accepted"] += a
    if len(st["accept_hist"]) <= k:
        st["accept_hist"] += [0] * (k + 1 - len(st["accept_hist"]))
    st["accept_hist"][a] += 1
    if len(st["depth_drafted"]) < k:
        st["depth_drafted"] += [0] * (k - len(st["depth_drafted"]))
        st["depth_accepted"] += [0] * (k - len(st["depth_accepted"]))
    for d in range(k):
        st["depth_drafted"][d] += 1
        if d < a:
            st["depth_accepted"][d] += 1
    return st


def spec_tokens_per_round(st):
    """[mimo_mtp.rs] ``MtpStats::tokens_per_round``: accepted drafts plus the
    verifier's own token, per round (0 before any round)."""
    if st["rounds"] == 0:
        return 0.0
    return (st["accepted"] + st["rounds"]) / st["rounds"]


def spec_rewind(cache_len, keep):
    """[mimo_mtp.rs] ``mimo_verify_rewind``: a layer holding more than ``keep``
    rows drops the rows past ``keep`` (an absolute position); shorter layers
    are left as they are."""
    return [keep if n > keep else n for n in cache_len]

