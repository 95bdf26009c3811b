// Speculation bookkeeping of one sequence: host code only.
//
// "cortiq-engine 0.8.49 src/mimo_mtp.rs": the counters of MtpStats and its
// tokens_per_round, the accepted prefix and the counter updates at the end
// of mimo_spec_round, the absolute rewind of mimo_verify_rewind, and the
// per-layer committed/base state of mimo_mtp_draft.
#include "host.h"

extern "C" {

int32_t mtp_spec_accept(const int32_t* drafts, const int32_t* verify_tokens, int32_t k) {
  if (k < 0 || k > MTP_SPEC_MAX_DEPTH) return -1;
  if (k > 0 && (!drafts || !verify_tokens)) return -1;
  int32_t a = 0;
  while (a < k && drafts[a] == verify_tokens[a]) ++a;  // the first mismatch ends the prefix
  return a;
}

mtp_status mtp_spec_note_round(mtp_spec_stats* s, int32_t k, int32_t a, uint64_t draft_ns,
                               uint64_t verify_ns) {
  if (!s) return mtp::fail(MTP_ERR_INVALID_ARG, "mtp_spec_note_round: null stats");
  if (k < 0 || k > MTP_SPEC_MAX_DEPTH || a < 0 || a > k)
    return mtp::fail(MTP_ERR_INVALID_ARG, "mtp_spec_note_round: need 0 <= a <= k <= 16");
  s->rounds += 1;
  s->drafted += (uint64_t)k;
  s->accepted += (uint64_t)a;
  s->accept_hist[a] += 1;
  for (int32_t d = 0; d < k; ++d) {
    s->depth_drafted[d] += 1;
    if (d < a) s->depth_accepted[d] += 1;
  }
  s->draft_ns += draft_ns;
  s->verify_ns += verify_ns;
  return MTP_OK;
}

double mtp_spec_tokens_per_round(const mtp_spec_stats* s) {
  if (!s || s->rounds == 0) return 0.0;
  return (double)(s->accepted + s->rounds) / (double)s->rounds;
}

mtp_status mtp_spec_rewind(int32_t* cache_len, int32_t n_layers, int32_t keep) {
  if (n_layers < 0 || keep < 0 || (n_layers > 0 && !cache_len))
    return mtp::fail(MTP_ERR_INVALID_ARG, "mtp_spec_rewind: bad arguments");
  for (int32_t l = 0; l < n_layers; ++l)
    if (cache_len[l] > keep) cache_len[l] = keep;
  return MTP_OK;
}

int32_t mtp_mimo_plan_layer(mtp_mimo_layer_state* st, int32_t layer, int32_t t, int32_t hist_lo,
                            int32_t hist_end, int32_t ids_len, int32_t* start) {
  if (!st || !start || layer < 0) return -1;
  // no draft this round: the history lacks position t, or x_{t+1} is unknown
  if (hist_end <= hist_lo || t < hist_lo || t >= hist_end || ids_len < t + 2) return 0;
  if (st->committed < hist_lo || st->committed > t + 1) {
    // a history gap (first round after a long prompt) or a stale state
    st->kv_len = 0;
    st->base = hist_lo;
    st->committed = hist_lo;
  }
  const int32_t keep = st->committed - st->base;  // drop last round's provisional rows
  if (st->kv_len > keep) st->kv_len = keep;
  *start = st->committed;
  return t + 1 - st->committed;
}

mtp_status mtp_mimo_commit_layer(mtp_mimo_layer_state* st, int32_t layer, int32_t t,
                                 int32_t ids_len) {
  if (!st || layer < 0 || t + 1 < st->base)
    return mtp::fail(MTP_ERR_INVALID_ARG, "mtp_mimo_commit_layer: bad arguments");
  st->kv_len = t + 1 - st->base;
  int32_t real_end = ids_len - (layer + 1);  // row j embeds token j + layer + 1
  if (real_end < 0) real_end = 0;
  if (real_end > t + 1) real_end = t + 1;
  if (real_end > st->committed) st->committed = real_end;
  return MTP_OK;
}

}  // extern "C"
