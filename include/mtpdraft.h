/*
 * mtpdraft.h -- C ABI of the MTP draft-layer forward on one sm_103a GPU.
 *
 * The draft layer (multi-token-prediction "NextN" block) drafts the next
 * token for speculative greedy decoding:
 *
 *   u   = eh_proj . [RMSNorm(embed(tok)) * enorm ; RMSNorm(hid) * hnorm]
 *   u1  = u  + o_proj(attn(RMSNorm(u) * attn_norm))     (own KV cache)
 *   u2  = u1 + FFN(RMSNorm(u1) * post_norm)            (SwiGLU or MoE)
 *   tok = argmax(lm_head(RMSNorm(u2) * final_norm))
 *
 * as stated in the module documentation of "cortiq-engine 0.8.49
 * src/mimo_mtp.rs" and implemented step by step in "hf2q 0.1.13
 * src/inference/models/qwen35/mtp.rs" (forward_draft_body,
 * project_embedding_and_hidden, forward_full_attention,
 * forward_ffn_residual, forward_shared_head_greedy).
 *
 * Every projection uses mlx-affine 4-bit group-32 weights ("hf2q 0.1.1
 * src/serve/forward_mlx_shared.rs", MlxAffineExtra / MlxQWeight): codes
 * uint32 [N][K/8] with the code of column 8*j+i in bits 4i..4i+3 of word j,
 * float32 scales and biases [N][K/32], w[n][k] = s*code + b.
 *
 * Conventions for every entry point:
 *  - Pointers named d_* or documented as device are device pointers owned by
 *    the caller; host pointers are named h_* or are descriptor structs.  The
 *    library never allocates device memory and keeps no state between calls
 *    (attn_decode_sink_noalloc alone keeps a static device scratch).
 *  - All work is enqueued on `stream` (a cudaStream_t, NULL = legacy
 *    default stream); no call synchronises the device, so calls can be
 *    captured into a CUDA graph (tensor maps are encoded on the host at
 *    enqueue time and baked into the launch).
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns a non-zero mtp_status and launches nothing.
 *    mtp_last_error() then returns a thread-local message.
 *  - Device activations are float32, row-major.
 *  - Device pointers must be 16-byte aligned.  Reduction lengths K must be
 *    multiples of 32; entry points that take a workspace state their extra
 *    shape rules.
 *  - Workspaces are caller-owned device buffers of at least the size the
 *    matching *_workspace_bytes() function returns.  Before its first use a
 *    workspace must be cleared once with mtp_workspace_init(); kernels leave
 *    it in that state again when they finish.  Calls that share a workspace
 *    must not overlap on the GPU.
 */
#ifndef MTPDRAFT_H
#define MTPDRAFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MTPDRAFT_VERSION 2

typedef enum {
    MTP_OK = 0,
    MTP_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, misaligned pointer */
    MTP_ERR_UNSUPPORTED = 2,   /* a shape the kernels do not implement */
    MTP_ERR_CAPACITY = 3,      /* cache_len + m exceeds the cache capacity */
    MTP_ERR_WORKSPACE = 4,     /* workspace missing or too small */
    MTP_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    MTP_ERR_DEVICE_TIMEOUT = 6 /* a bounded device-side wait gave up (see mtp_workspace_status) */
} mtp_status;

/* One affine 4-bit group-32 weight [n][k] (device pointers). */
typedef struct {
    const uint32_t *q;   /* [n][k/8] packed codes, low nibble first */
    const float *s;      /* [n][k/32] scales */
    const float *b;      /* [n][k/32] biases */
    int32_t n;
    int32_t k;
} mtp_affine4;

/* Thread-local description of the last failure on this thread ("" if none). */
const char *mtp_last_error(void);
int mtp_version(void);

/* Clears a workspace (device memset of `bytes`, enqueued on `stream`). */
mtp_status mtp_workspace_init(void *d_ws, size_t bytes, void *stream);

/* Reads the device error word of a workspace (synchronous device-to-host
 * copy); the first error since mtp_workspace_init is kept:
 *   0 none; 1 a wait for a TMA copy gave up; 2 a token id outside
 *   [0, vocab) (row 0 was used); 3 a wait inside a multi-projection launch
 *   for the previous projection's output gave up; 4 a wait of the attention
 *   splits of a KV head for each other's partials gave up.
 * After code 1, 3 or 4 a launch stopped part-way (its outputs are not
 * valid) and may have left completion counters set: clear the workspace
 * with mtp_workspace_init() before its next use.  Code 2 leaves the
 * workspace usable.  The waits behind codes 3 and 4 need every CTA of the
 * launch resident at once (the launches size their grids for that); a
 * device shared with other work at the same time can make them give up, so
 * check the status after steps whose results matter. */
mtp_status mtp_workspace_status(const void *d_ws, int32_t *h_code, void *stream);

/* Diagnostic hook: the cross-CTA waits of later launches on this workspace
 * (codes 3 and 4 above) give up after `polls` polls (0 restores the compiled
 * limit of about two seconds).  With a limit of one poll, waits that are not
 * already satisfied give up at once, which exercises the error path on a
 * healthy device.  Enqueued on `stream`; mtp_workspace_init() also resets
 * it to 0. */
mtp_status mtp_workspace_set_wait_limit(void *d_ws, int32_t polls, void *stream);

/* Diagnostics (per calling thread): between mtp_timing_begin and
 * mtp_timing_end every kernel launch the library enqueues from this thread
 * is preceded by a record of the next of `events` (cudaEvent_t handles the
 * caller created) on the launch's stream; mtp_timing_end records one more
 * event after the last launch and stores how many marks were made (launches
 * + 1).  The interval between events i and i + 1 is launch i alone: a record
 * between two launches removes their programmatic overlap.  Sessions do not
 * nest; more launches than events are counted but not recorded
 * (mtp_timing_end then returns MTP_ERR_INVALID_ARG).  Not for use inside
 * stream capture. */
mtp_status mtp_timing_begin(void *const *events, int32_t n_events);
mtp_status mtp_timing_end(int32_t *n_recorded);

/* ------------------------------------------------------------------------
 * qmatmul_affine4: y[r][n] = sum_k x[r][k] * (s[n][k/32]*code[n][k] + b[n][k/32])
 *
 * "hf2q 0.1.1 src/serve/forward_mlx_shared.rs", dispatch_qmatmul (affine
 * branch) and the CPU reference of its unit tests.
 *   d_x  [m][K] float32; d_y [m][N] float32 (overwritten); 1 <= m <= 16.
 *   W->k must equal K and be a multiple of 32.
 *   d_ws: workspace of qmatmul_affine4_workspace_bytes(m, K) bytes; it holds
 *         the activations in the tensor-core operand layout.
 * Activation range (this call and every projection of the draft step): the
 * tensor-core path splits each activation into f16 high and low parts.  A
 * 32-value group whose largest |x| reaches 2^15 is stored times a power of
 * two 2^-e (its largest value then lies in [2^14, 2^15)) and its weight
 * scales are multiplied back by 2^e, so every finite activation is accepted;
 * within such a group, values more than about 2^-100 times its largest may
 * flush to zero.  Inf and NaN propagate to the outputs.
 * ------------------------------------------------------------------------ */
size_t qmatmul_affine4_workspace_bytes(int32_t m, int32_t k);
mtp_status qmatmul_affine4(const float *d_x, const mtp_affine4 *W, float *d_y, int32_t m,
                           void *d_ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * rmsnorm_residual: sum = a + delta (or a when delta is NULL);
 *   out_norm = sum / sqrt(mean(sum^2) + eps) * w ; out_sum = sum (if not NULL)
 *
 * "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", forward_ffn_residual
 * (dispatch_fused_residual_norm_f32: the residual sum and its RMSNorm, both
 * written) and rms_norm_with_weight.
 *   d_a, d_delta, d_out_norm, d_out_sum: [rows][dim] float32; d_w: [dim].
 *   out_norm may alias neither input; out_sum may alias d_a.
 * ------------------------------------------------------------------------ */
mtp_status rmsnorm_residual(const float *d_a, const float *d_delta, const float *d_w,
                            float *d_out_norm, float *d_out_sum, int32_t rows, int32_t dim,
                            float eps, void *stream);

/* ------------------------------------------------------------------------
 * Attention geometry of a draft layer.
 *   q_rows = n_heads*head_dim_qk, or 2*n_heads*head_dim_qk when gated_q: head h
 *   then owns projection rows [2h*dqk, 2h*dqk+dqk) for its query and the next
 *   dqk rows for its sigmoid gate (requires head_dim_v == head_dim_qk).
 * ------------------------------------------------------------------------ */
typedef struct {
    int32_t n_heads;
    int32_t n_kv_heads;    /* divides n_heads; query head h reads KV head h / (n_heads/n_kv_heads) */
    int32_t head_dim_qk;   /* multiple of 32, <= 256 */
    int32_t head_dim_v;    /* multiple of 32, <= 256 */
    int32_t rot_dim;       /* rotated dims (even, <= head_dim_qk); pairs (i, i + rot_dim/2) */
    int32_t window;        /* > 0: row at position p sees keys p-window < j <= p; <= 0: full causal */
    int32_t gated_q;       /* 0/1 */
    float eps;             /* epsilon of the per-head q/k RMSNorm */
    float scale;           /* logit scale; 0 selects 1/sqrt(head_dim_qk) */
} mtp_attn_geom;

/* Fills d_rope[p][i] = (cos(p*theta^(-2i/rot_dim)), sin(...)) for 0 <= p < max_pos,
 * 0 <= i < rot_dim/2, angles evaluated in double precision.  d_rope holds
 * max_pos*rot_dim floats.  "hf2q 0.1.13 ... mtp.rs", apply_imrope with four
 * equal text position ids (1-D rotary embedding at the token position). */
mtp_status mtp_rope_table(float *d_rope, int32_t max_pos, int32_t rot_dim, double theta,
                          void *stream);

/* ------------------------------------------------------------------------
 * attn_decode_sink: per-head q/k RMSNorm (when q_norm/k_norm are given),
 * rotary embedding at positions cache_len + r, append of the m new K/V rows
 * to the cache, causal (optionally windowed) attention with an optional sink
 * logit per head, optional sigmoid output gate.
 *
 * "hf2q 0.1.13 ... mtp.rs" forward_full_attention (per-head norm, IMROPE,
 * apply_sdpa_with_kv_cache, apply_sigmoid_gate_multiply) and
 * "cortiq-engine 0.8.49 src/mimo_mtp.rs" module doc (window 128, sinks).
 * The sink is one extra logit per head, not scaled, entering the softmax
 * denominator only.
 *   d_qp [m][q_rows], d_kp [m][n_kv*dqk], d_vp [m][n_kv*dv]: raw projections.
 *   d_q_norm, d_k_norm: [dqk] or NULL.  d_sinks: [n_heads] or NULL.
 *   d_rope: table of mtp_rope_table with max_pos >= cache_len + m.
 *   d_k_cache [n_kv][cache_cap][dqk], d_v_cache [n_kv][cache_cap][dv]:
 *     rows < cache_len are read; rows cache_len .. cache_len+m-1 are written.
 *   d_out [m][n_heads*dv] float32.
 *   1 <= m <= 16; (n_heads/n_kv_heads)*m <= 16.
 *   Returns MTP_ERR_CAPACITY if cache_len + m > cache_cap.
 * ------------------------------------------------------------------------ */
size_t attn_decode_sink_workspace_bytes(const mtp_attn_geom *g, int32_t m, int32_t cache_len);
mtp_status attn_decode_sink(const mtp_attn_geom *g, const float *d_qp, const float *d_kp,
                            const float *d_vp, const float *d_q_norm, const float *d_k_norm,
                            const float *d_rope, const float *d_sinks, float *d_k_cache,
                            float *d_v_cache, int32_t cache_len, int32_t cache_cap, int32_t m,
                            float *d_out, void *d_ws, size_t ws_bytes, void *stream);

/* attn_decode_sink_noalloc: attn_decode_sink with the library's own static
 * device scratch (2 MiB, a file-scope __device__ array) in place of d_ws.
 * The draft-layer method has no counterpart of this call: it exists for
 * callers that hold no device memory to lend, such as a host runtime whose
 * device memory all sits in its own pools, or a plugin interface whose
 * signature carries no workspace.  It allocates no device memory.
 *  - The first call on a device looks up the scratch address and clears its
 *    header with a synchronous cudaMemset; make that first call before any
 *    stream capture.  Later calls enqueue a clear of the completion counters
 *    on `stream`, then the same launch as attn_decode_sink.
 *  - Geometries whose scratch (attn_decode_sink_workspace_bytes) exceeds
 *    2 MiB return MTP_ERR_WORKSPACE without launching anything.
 *  - Calls that overlap on one device share the scratch and race: order
 *    them (one stream, or events).
 *  - A device-side wait that gives up records its code in the scratch
 *    header, which this call does not expose; use attn_decode_sink with a
 *    workspace where that status is needed.
 * Arguments, layouts and other errors as attn_decode_sink. */
mtp_status attn_decode_sink_noalloc(const mtp_attn_geom *g, const float *d_qp,
                                    const float *d_kp, const float *d_vp,
                                    const float *d_q_norm, const float *d_k_norm,
                                    const float *d_rope, const float *d_sinks, float *d_k_cache,
                                    float *d_v_cache, int32_t cache_len, int32_t cache_cap,
                                    int32_t m, float *d_out, void *stream);

/* ------------------------------------------------------------------------
 * lmhead_argmax: y_n = RMSNorm(y)*norm_w (or y when norm_w is NULL);
 *   logits = W . y_n; token = argmax (lowest index among equal maxima).
 *
 * "hf2q 0.1.13 ... mtp.rs" forward_shared_head_greedy (norm, vocabulary
 * projection and argmax in one submission); logits stay on chip unless
 * d_logits is given.
 *   d_y [H]; W [V][H]; d_token (int32) and d_value (float) receive the result;
 *   d_logits [V] or NULL; d_y_normed [H] or NULL.  H % 128 == 0.
 * ------------------------------------------------------------------------ */
size_t lmhead_argmax_workspace_bytes(int32_t hidden, int32_t vocab);
mtp_status lmhead_argmax(const float *d_y, const float *d_norm_w, float eps,
                         const mtp_affine4 *W, int32_t *d_token, float *d_value, float *d_logits,
                         float *d_y_normed, void *d_ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * verify_head_argmax: for each of `rows` hidden rows h_r,
 *   y_r = RMSNorm(h_r)*norm_w (or h_r when norm_w is NULL);
 *   l_r = W . y_r;  l_r *= logit_multiplier;
 *   l_r = softcap * tanh(l_r / softcap)   (only when softcap > 0);
 *   token_r = argmax l_r (lowest index among equal maxima), value_r = l_r[token_r].
 *
 * "cortiq-engine 0.8.49 src/mimo_mtp.rs" mimo_verify_head_rows (the final
 * norm and the lm_head over the pending token and the k drafts in one head
 * pass, then the optional logit multiplier and final softcap, in that order)
 * as used by mimo_spec_round, whose greedy verification takes each row's
 * argmax.  The vocabulary matrix is streamed once for all rows.
 *   d_h [rows][H] row-major; rows in 1..16 (the pages use 2..4); W [V][H];
 *   logit_multiplier: 1 for none (any finite value); softcap <= 0 for none;
 *   d_tokens [rows] (int32) and d_values [rows] receive the result;
 *   d_logits [rows][V] receives the final logits, or NULL (kept in d_ws).
 *   H % 128 == 0; pointers 16-byte aligned.  Arithmetic after the projection
 *   is float32, so ties are decided on the float32 values.
 * ------------------------------------------------------------------------ */
size_t verify_head_workspace_bytes(int32_t rows, int32_t hidden, int32_t vocab);
mtp_status verify_head_argmax(const float *d_h, int32_t rows, const float *d_norm_w, float eps,
                              const mtp_affine4 *W, float logit_multiplier, float softcap,
                              int32_t *d_tokens, float *d_values, float *d_logits, void *d_ws,
                              size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * MoE feed-forward (router softmax, top-k, renormalised expert SwiGLUs plus a
 * sigmoid-gated shared expert).  "hf2q 0.1.13 ... mtp.rs" MtpFfnWeightsGpu::Moe
 * (router, stacked expert gate/up/down, four shared-expert tensors) and
 * "hf2q 0.1.1 ... forward_mlx_shared.rs" MlxAffineMoeStack (expert e of a
 * stack is slab e of [E][N][K/8]; scales and biases float32, or bfloat16 as
 * the page's stacks store them).
 * ------------------------------------------------------------------------ */
typedef struct {
    int32_t n_experts;        /* <= 1024 */
    int32_t top_k;            /* 1..16 */
    int32_t expert_inter;     /* multiple of 128 */
    int32_t shared_inter;     /* multiple of 128, 0 = no shared expert */
    const float *router;      /* [n_experts][hidden] float32 */
    mtp_affine4 exp_gate;     /* stacked: n = n_experts*expert_inter, k = hidden */
    mtp_affine4 exp_up;       /* stacked: n = n_experts*expert_inter, k = hidden */
    mtp_affine4 exp_down;     /* stacked: n = n_experts*hidden, k = expert_inter */
    mtp_affine4 sh_gate, sh_up, sh_down;
    const float *sh_gate_inp; /* [hidden]: shared expert gate = sigmoid(sh_gate_inp . f) */
    int32_t scales_bf16;      /* 1: the stacks exp_gate/exp_up/exp_down hold their scales and
                                 biases as bfloat16 [n][k/32] ("hf2q 0.1.1 ...
                                 forward_mlx_shared.rs", MlxAffineMoeStack; their s and b
                                 pointers then point at bfloat16 data); needs hidden and
                                 expert_inter multiples of 256.  0: float32.  The shared
                                 expert's are float32 either way. */
} mtp_moe_weights;

/* u2 = u1 + MoE(RMSNorm(u1)*post_norm) for one row (m = 1).
 * d_sel (int32 [top_k]) and d_weight (float [top_k+1]) receive the routing
 * decision (chosen experts and their renormalised weights, then the shared
 * gate) when not NULL. */
size_t moe_ffn_workspace_bytes(const mtp_moe_weights *w, int32_t hidden);
mtp_status moe_ffn(const mtp_moe_weights *w, const float *d_u1, const float *d_post_norm,
                   float eps, int32_t hidden, float *d_u2, int32_t *d_sel, float *d_weight,
                   void *d_ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Whole draft layer.
 * ------------------------------------------------------------------------ */
typedef struct {
    int32_t hidden;           /* multiple of 128 */
    int32_t vocab;
    int32_t intermediate;     /* dense SwiGLU width (multiple of 128); ignored when moe != NULL */
    float eps;                /* RMSNorm eps of attn/post/final norms (enorm/hnorm use 1e-6) */
    mtp_attn_geom attn;
    const float *enorm, *hnorm;      /* [hidden] */
    mtp_affine4 eh_proj;             /* [hidden][2*hidden], embedding half first */
    const float *attn_norm;          /* [hidden] */
    mtp_affine4 wq, wk, wv, wo;
    const float *q_norm, *k_norm;    /* [head_dim_qk] or NULL */
    const float *sinks;              /* [n_heads] or NULL */
    const float *post_norm;          /* [hidden] */
    mtp_affine4 ffn_gate, ffn_up, ffn_down;
    const mtp_moe_weights *moe;      /* host struct, or NULL for the dense FFN */
    const float *final_norm;         /* [hidden] */
    mtp_affine4 lm_head;             /* [vocab][hidden] */
    const float *embed;              /* [vocab][hidden] float32, or NULL (caller passes rows) */
    const float *rope;               /* mtp_rope_table with max_pos >= pos_base + cache_cap */
    float *k_cache, *v_cache;        /* [n_kv][cache_cap][d] */
    int32_t cache_cap;
} mtp_layer_desc;

typedef struct {
    const int32_t *d_tokens;         /* [m] token ids (used when embed != NULL) */
    const float *d_embed_rows;       /* [m][hidden] embedding rows (used when embed == NULL) */
    const float *d_hidden;           /* [m][hidden] target hidden states */
    int32_t cache_len;               /* rows already in the layer's cache */
    int32_t m;                       /* new rows, 1..16 */
    int32_t pos_base;                /* rotary position of cache row 0 (0 unless the cache
                                        was restarted part-way); row r rotates at
                                        pos_base + cache_len + r */
} mtp_step_in;

typedef struct {
    int32_t *d_token;                /* argmax of the last row's logits */
    float *d_value;                  /* its logit */
    float *d_hidden_out;             /* [hidden] RMSNorm(u2[m-1])*final_norm, or NULL */
    float *d_u2;                     /* [m][hidden] layer output before the final norm, or NULL */
    float *d_logits;                 /* [vocab] or NULL */
} mtp_step_out;

/* One draft-layer step over m rows at positions cache_len .. cache_len+m-1.
 * The m new K/V rows are written into the cache; the caller advances its
 * cache length by m when the call returns MTP_OK. */
size_t mtp_draft_workspace_bytes(const mtp_layer_desc *L, int32_t m);
mtp_status mtp_draft_forward(const mtp_layer_desc *L, const mtp_step_in *in,
                             const mtp_step_out *out, void *d_ws, size_t ws_bytes, void *stream);

/* Chained draft of n_layers layers ("cortiq-engine 0.8.49 src/mimo_mtp.rs",
 * "How the three layers chain" and mimo_mtp_draft): every layer reads the
 * same target hiddens d_hidden [m][hidden]; layer k row i embeds
 * d_seq[i + k], and layer k writes its draft to d_seq[m + k], so d_seq holds
 * m + n_layers int32 (the first m given).  The draft of one layer feeds the
 * next layer's embedding gather on the device, with no host round trip.
 * All layers need an embedding table.  d_values [n_layers] receives the
 * drafts' logits; d_hidden_out [n_layers][hidden] (or NULL) each layer's
 * normed last row; d_u2 [n_layers][m][hidden] (or NULL) each layer's output
 * rows before the final norm; d_logits [n_layers][vocab] (or NULL) each
 * layer's last-row logits (layers must then share the vocabulary size).
 * cache_lens[k] is layer k's cache length (host array). */
mtp_status mtp_draft_chain(const mtp_layer_desc *layers, int32_t n_layers,
                           const float *d_hidden, int32_t *d_seq, const int32_t *cache_lens,
                           int32_t m, float *d_values, float *d_hidden_out, float *d_u2,
                           float *d_logits, void *d_ws, size_t ws_bytes, void *stream);

/* k_steps chained one-row draft steps of one layer ("hf2q 0.1.13 ... mtp.rs",
 * forward_draft_with_hidden: a chained step reads the normed row the shared
 * head returns, the only valid hidden for a second MTP step).  Step i
 * embeds d_tokens[i], reads hidden h_i (h_0 = d_hidden [hidden], h_{i+1} =
 * d_hidden_out[i]), appends its K/V row at cache row cache_len + i (rotary
 * position pos_base + cache_len + i), and writes its draft to
 * d_tokens[i + 1], its logit to d_values[i] and its normed row to
 * d_hidden_out[i] ([k_steps][hidden]).  d_tokens holds k_steps + 1 int32,
 * the first given.  The layer needs an embedding table; the steps follow
 * each other on the device with no host synchronisation.  d_ws: at least
 * mtp_draft_workspace_bytes(L, 1). */
mtp_status mtp_draft_steps(const mtp_layer_desc *L, int32_t k_steps, const float *d_hidden,
                           int32_t *d_tokens, int32_t cache_len, int32_t pos_base,
                           float *d_values, float *d_hidden_out, void *d_ws, size_t ws_bytes,
                           void *stream);

/* ------------------------------------------------------------------------
 * mtp_kv_catch_up: the K/V rows of a target batch of seq tokens, written to
 * the layer's cache ("hf2q 0.1.13 ... mtp.rs", process_target_batch and
 * append_attention_kv).  Row i embeds d_tokens[i] (or d_embed_rows[i]) and
 * reads the target hidden shifted one row right: row 0 reads d_pending (the
 * target hidden of the token before the batch; NULL for a cold prompt reads
 * zeros), row i > 0 reads d_target[i - 1] (the last target row is not read).
 *   u = eh_proj [RMSNorm(e)*enorm ; RMSNorm(h)*hnorm]  (eps 1e-6)
 *   x = RMSNorm(u)*attn_norm;  k = W_k x, per-head RMSNorm by k_norm (if
 *   given), rotated at pos_base + cache_len + i;  v = W_v x.
 * Rows go to cache rows cache_len .. cache_len + seq - 1.  No attention, FFN
 * or head runs.  The projections run on the tensor cores (tcgen05) with bf16
 * hi + lo parts of the dequantised weights and of the activations.
 *   d_target [seq][hidden] (may be NULL when seq == 1); d_pending [hidden].
 *   1 <= seq <= 65535; 1..32 KV heads; the layer's q/o/FFN/head weights are
 *   not read.  Token ids outside [0, vocab) set device error code 2 (row 0
 *   is used).  The workspace (mtp_kv_catch_up_workspace_bytes) is about
 *   12 * seq * hidden bytes plus split-K partials.
 * ------------------------------------------------------------------------ */
size_t mtp_kv_catch_up_workspace_bytes(const mtp_layer_desc *L, int32_t seq);
mtp_status mtp_kv_catch_up(const mtp_layer_desc *L, const int32_t *d_tokens,
                           const float *d_embed_rows, const float *d_target,
                           const float *d_pending, int32_t seq, int32_t cache_len,
                           int32_t pos_base, void *d_ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Speculation bookkeeping of one sequence (host only: no device work, no
 * stream).  "cortiq-engine 0.8.49 src/mimo_mtp.rs": MtpStats (its counters
 * and tokens_per_round), the accepted prefix of mimo_spec_round and
 * mimo_verify_rewind.  A round drafts k tokens, the verifier scores the
 * pending token and the k drafts in one batch (verify_head_argmax gives its
 * greedy token per row), the drafts are kept while they equal the
 * verifier's token at the same depth, and every cache is cut back to the
 * kept positions.
 * ------------------------------------------------------------------------ */
#define MTP_SPEC_MAX_DEPTH 16

/* Counters of one generation; zero-initialise before the first round. */
typedef struct {
    uint64_t rounds;                                 /* verify batches */
    uint64_t drafted;                                /* drafts proposed */
    uint64_t accepted;                               /* drafts accepted */
    uint64_t accept_hist[MTP_SPEC_MAX_DEPTH + 1];    /* rounds that accepted exactly a drafts */
    uint64_t depth_drafted[MTP_SPEC_MAX_DEPTH];      /* rounds that drafted depth d (0-based) */
    uint64_t depth_accepted[MTP_SPEC_MAX_DEPTH];     /* rounds whose accepted prefix reached depth d */
    uint64_t draft_ns;                               /* time in the drafts */
    uint64_t verify_ns;                              /* time in the verify */
} mtp_spec_stats;

/* The accepted prefix: the largest a <= k with drafts[i] == verify_tokens[i]
 * for every i < a, where verify_tokens[i] is the verifier's greedy token on
 * the row after the pending token and drafts[0..i-1] (host arrays; entry k,
 * the round's own next token, is not read).  Returns -1 when a pointer is
 * NULL with k > 0 or k is outside 0..MTP_SPEC_MAX_DEPTH. */
int32_t mtp_spec_accept(const int32_t *drafts, const int32_t *verify_tokens, int32_t k);

/* Adds one round of k drafts with a accepted (0 <= a <= k <= MTP_SPEC_MAX_DEPTH)
 * and its draft and verify times; MTP_ERR_INVALID_ARG otherwise (s unchanged). */
mtp_status mtp_spec_note_round(mtp_spec_stats *s, int32_t k, int32_t a, uint64_t draft_ns,
                               uint64_t verify_ns);

/* Tokens a round emits on average: (accepted + rounds) / rounds (the
 * accepted drafts plus the verifier's own token); 0 before the first round. */
double mtp_spec_tokens_per_round(const mtp_spec_stats *s);

/* After a rejected suffix: every cache_len[l] above `keep` becomes `keep`
 * (an absolute row count, not a step back from a possibly stale cursor);
 * lengths at or below it are unchanged.  MTP_ERR_INVALID_ARG on a NULL
 * array with n_layers > 0, n_layers < 0 or keep < 0. */
mtp_status mtp_spec_rewind(int32_t *cache_len, int32_t n_layers, int32_t keep);

/* One draft layer's round state ("cortiq-engine 0.8.49 src/mimo_mtp.rs",
 * MimoMtp): cache rows at positions below `committed` are final, `base` is
 * the position of the cache's first row, `kv_len` the rows the cache holds.
 * Zero-initialise before the first round. */
typedef struct {
    int32_t committed;
    int32_t base;
    int32_t kv_len;
} mtp_mimo_layer_state;

/* Plans layer `layer`'s part of a round that starts after the backbone
 * processed position t (mimo_mtp_draft): the target-hidden history holds
 * positions [hist_lo, hist_end) and ids_len token ids are known (x_{t+1}
 * among them).  Returns the number of rows to run, n = t + 1 - *start (rows
 * at positions *start .. t; row j embeds token j + layer + 1, a round's
 * earlier draft past the known ids), 0 when nothing is drafted this round
 * (the history lacks t, or ids_len < t + 2), -1 on a NULL pointer.  Updates
 * *st: a committed position below the history (a gap) or beyond t + 1 (a
 * stale state) restarts the cache at hist_lo (kv_len = 0, base = committed
 * = hist_lo); the previous round's provisional rows are dropped (kv_len =
 * committed - base).  The rows go to cache rows *start - base onwards, at
 * rotary positions *start onwards (pos_base = base). */
int32_t mtp_mimo_plan_layer(mtp_mimo_layer_state *st, int32_t layer, int32_t t, int32_t hist_lo,
                            int32_t hist_end, int32_t ids_len, int32_t *start);

/* After the layer ran its rows: kv_len = t + 1 - base, and committed rises to
 * min(t + 1, ids_len - layer - 1) (the rows whose token is known). */
mtp_status mtp_mimo_commit_layer(mtp_mimo_layer_state *st, int32_t layer, int32_t t,
                                 int32_t ids_len);

/* The draft half of one MiMo round on the device (mimo_mtp_draft): for each
 * layer l < n_layers in order, mtp_mimo_plan_layer, then its rows: positions
 * start .. t - 1 only add K/V rows (mtp_kv_catch_up: row j embeds
 * d_ids[j + l + 1] and reads target hidden row j), and position t runs a
 * one-row draft step whose argmax goes to d_ids[t + l + 2] and its logit to
 * d_values[l]; then mtp_mimo_commit_layer.  Only the last row of a layer
 * reaches the head and its output depends on the earlier rows only through
 * their K/V rows, so this equals running all n rows through the layer.
 *   d_hist: target hidden rows [hist_end - hist_lo][hidden] for positions
 *     hist_lo .. hist_end - 1;  d_ids: token ids by position, at least
 *     t + n_layers + 2 entries (the first ids_len known);
 *   states[n_layers] are updated on the host as the launches are enqueued;
 *   d_ws: mtp_draft_workspace_bytes(layer, 1) for every layer;
 *   d_catch_ws: mtp_kv_catch_up_workspace_bytes(layer, rows) for the most
 *     rows a layer catches up (t - hist_lo after a restart).
 * *n_drafts receives the number of layers run (0: no draft this round).
 * The layers need an embedding table.  No host synchronisation. */
mtp_status mtp_mimo_draft_round(const mtp_layer_desc *layers, int32_t n_layers,
                                mtp_mimo_layer_state *states, const float *d_hist,
                                int32_t hist_lo, int32_t hist_end, int32_t t, int32_t *d_ids,
                                int32_t ids_len, float *d_values, void *d_ws, size_t ws_bytes,
                                void *d_catch_ws, size_t catch_ws_bytes, void *stream,
                                int32_t *n_drafts);

#ifdef __cplusplus
}
#endif

#endif /* MTPDRAFT_H */
