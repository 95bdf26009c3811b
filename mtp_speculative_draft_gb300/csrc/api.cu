// C ABI of the draft-layer library: host-side validation, workspace layout and
// the launch sequence of each entry point.  Every step of the path runs in
// this library's kernels; the host only checks arguments, encodes tensor maps
// and enqueues launches.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "host.h"

namespace mtp {

static thread_local std::string g_last_error;

mtp_status fail(mtp_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}
mtp_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MTP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  cache[dev] = n;
  return n;
}

mtp_status check_affine(const mtp_affine4* w, int n, int k, const char* name, bool need_tma) {
  if (!w) return fail(MTP_ERR_INVALID_ARG, std::string(name) + ": null weight descriptor");
  if (!w->q || !w->s || !w->b)
    return fail(MTP_ERR_INVALID_ARG, std::string(name) + ": null weight pointer");
  if (w->n <= 0 || w->k <= 0)
    return fail(MTP_ERR_INVALID_ARG, std::string(name) + ": non-positive shape");
  if ((n >= 0 && w->n != n) || (k >= 0 && w->k != k))
    return fail(MTP_ERR_INVALID_ARG, std::string(name) + ": shape [" + std::to_string(w->n) +
                                         ", " + std::to_string(w->k) + "], expected [" +
                                         std::to_string(n) + ", " + std::to_string(k) + "]");
  if (w->k % kGroup)
    return fail(MTP_ERR_UNSUPPORTED, std::string(name) + ": K must be a multiple of 32");
  if (!aligned16(w->q) || !aligned16(w->s) || !aligned16(w->b))
    return fail(MTP_ERR_INVALID_ARG, std::string(name) + ": pointers must be 16-byte aligned");
  if (need_tma && w->k % 128)
    return fail(MTP_ERR_UNSUPPORTED,
                std::string(name) + ": K must be a multiple of 128 on this path");
  return MTP_OK;
}

// Tensor maps are pure functions of (pointer, shape); cache them so a warm
// call encodes nothing.
static mtp_status qmat_cached(QMat* out, const mtp_affine4& w, const char* name,
                              bool sb_bf16 = false) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, const void*, const void*, int, int, int, bool>, QMat> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  auto key = std::make_tuple((const void*)w.q, (const void*)w.s, (const void*)w.b, w.n, w.k, dev,
                             sb_bf16);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return MTP_OK;
    }
  }
  mtp_status st = encode_qmat(out, w, name, sb_bf16);
  if (st != MTP_OK) return st;
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = *out;
  return MTP_OK;
}

// Launch-timing session of this thread (mtp_timing_begin / mtp_timing_end).
struct TimingSession {
  void* const* events = nullptr;
  int n_events = 0;
  int recorded = 0;
  cudaStream_t last = nullptr;
  cudaError_t err = cudaSuccess;
};
static thread_local TimingSession g_timing;

void launch_mark(cudaStream_t st) {
  TimingSession& t = g_timing;
  if (!t.events) return;
  if (t.recorded < t.n_events) {
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(t.events[t.recorded]), st);
    if (e != cudaSuccess && t.err == cudaSuccess) t.err = e;
  }
  ++t.recorded;
  t.last = st;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Bump allocator over a caller workspace.
struct Carve {
  uint8_t* base;
  size_t off = sizeof(WsHeader);
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t bytes) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align256(off + bytes);
    return p;
  }
};

static WsHeader* header(void* ws) { return static_cast<WsHeader*>(ws); }

// Split-K partials and per-tile counters used by the GEMV launches of a call.
static GemvScratch carve_scratch(Carve& cv) {
  GemvScratch sc;
  sc.part_bytes = gemv_scratch_part_bytes();
  sc.part = cv.take<float>(sc.part_bytes);
  sc.cnt = cv.take<unsigned>(sizeof(unsigned) * kGemvCounters);
  sc.cnt_len = kGemvCounters - 8;  // the last 8: phase and pre-unit counters
  sc.phase_done = sc.cnt ? sc.cnt + sc.cnt_len : nullptr;
  return sc;
}

// Counter slots inside WsHeader::counters.
constexpr int kCntAttn = 0;      // [2 * n_kv] arrivals and departures (n_kv <= 64)
constexpr int kCntArgmax = 128;
constexpr int kCntRouter = 129;

static GemvSeg plain_seg(int tiles_end, int n, int mat, float* out, int ld, const float* res) {
  GemvSeg s = {};
  s.tile_end = tiles_end;
  s.n = n;
  s.mat = mat;
  s.sel_idx = -1;
  s.row_mult = 0;
  s.w_idx = -1;
  s.out_col0 = 0;
  s.ld = ld;
  s.out = out;
  s.res = res;
  return s;
}

static int tiles_of(int n) { return (n + 31) / 32; }

}  // namespace mtp

using namespace mtp;

extern "C" {

const char* mtp_last_error(void) { return g_last_error.c_str(); }
int mtp_version(void) { return MTPDRAFT_VERSION; }

mtp_status mtp_workspace_init(void* d_ws, size_t bytes, void* stream) {
  if (!d_ws || bytes < sizeof(WsHeader))
    return fail(MTP_ERR_WORKSPACE, "workspace smaller than its 1 KB header");
  cudaError_t e = cudaMemsetAsync(d_ws, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace init");
  return MTP_OK;
}

mtp_status mtp_workspace_status(const void* d_ws, int32_t* h_code, void* stream) {
  if (!d_ws || !h_code) return fail(MTP_ERR_INVALID_ARG, "null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h_code, d_ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace status");
  return MTP_OK;
}

mtp_status mtp_timing_begin(void* const* events, int32_t n_events) {
  if (!events || n_events < 2) return fail(MTP_ERR_INVALID_ARG, "timing: need at least two events");
  if (g_timing.events) return fail(MTP_ERR_INVALID_ARG, "timing: a session is already open on this thread");
  g_timing = TimingSession{};
  g_timing.events = events;
  g_timing.n_events = n_events;
  return MTP_OK;
}

mtp_status mtp_timing_end(int32_t* n_recorded) {
  TimingSession t = g_timing;
  g_timing = TimingSession{};
  if (!t.events) return fail(MTP_ERR_INVALID_ARG, "timing: no session is open on this thread");
  if (t.recorded > 0) {  // the closing event, after the last launch
    if (t.recorded < t.n_events) {
      cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(t.events[t.recorded]), t.last);
      if (e != cudaSuccess && t.err == cudaSuccess) t.err = e;
    }
    ++t.recorded;
  }
  if (n_recorded) *n_recorded = t.recorded;
  if (t.err != cudaSuccess) return cuda_fail(t.err, "timing: event record");
  if (t.recorded > t.n_events)
    return fail(MTP_ERR_INVALID_ARG, "timing: more launches than events (" +
                                         std::to_string(t.recorded) + " marks)");
  return MTP_OK;
}

mtp_status mtp_workspace_set_wait_limit(void* d_ws, int32_t polls, void* stream) {
  if (!d_ws) return fail(MTP_ERR_INVALID_ARG, "null workspace");
  if (polls < 0) return fail(MTP_ERR_INVALID_ARG, "polls must be >= 0");
  // pageable source: the copy has read `polls` when the call returns
  const int32_t v = polls;
  cudaError_t e = cudaMemcpyAsync(&header(d_ws)->wait_limit, &v, sizeof(v), cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace wait limit");
  return MTP_OK;
}

mtp_status mtp_rope_table(float* d_rope, int32_t max_pos, int32_t rot_dim, double theta,
                          void* stream) {
  if (!d_rope) return fail(MTP_ERR_INVALID_ARG, "rope table: null pointer");
  if (max_pos <= 0 || rot_dim <= 0 || rot_dim % 2 || !(theta > 0.0))
    return fail(MTP_ERR_INVALID_ARG, "rope table: bad max_pos/rot_dim/theta");
  cudaError_t e = launch_rope_table(d_rope, max_pos, rot_dim, theta,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
  return MTP_OK;
}

// ------------------------------------------------------------------ qmatmul
size_t qmatmul_affine4_workspace_bytes(int32_t m, int32_t k) {
  if (m <= 0 || k <= 0) return 0;
  Carve cv(nullptr);
  cv.take<uint8_t>(xpack_bytes(m, k));
  carve_scratch(cv);
  return cv.off + 256;
}

mtp_status qmatmul_affine4(const float* d_x, const mtp_affine4* W, float* d_y, int32_t m,
                           void* d_ws, size_t ws_bytes, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!d_x || !d_y) return fail(MTP_ERR_INVALID_ARG, "qmatmul_affine4: null x or y");
  if (m < 1 || m > 16) return fail(MTP_ERR_UNSUPPORTED, "qmatmul_affine4: m must be in 1..16");
  mtp_status s = check_affine(W, -1, -1, "qmatmul_affine4 weight", false);
  if (s != MTP_OK) return s;
  if (!aligned16(d_x) || !aligned16(d_y))
    return fail(MTP_ERR_INVALID_ARG, "qmatmul_affine4: x and y must be 16-byte aligned");
  const int K = W->k, N = W->n;
  if (K % 128 != 0) {
    // Scale rows are not 16-byte aligned: plain CUDA-core path.
    cudaError_t e = launch_gemv_simple(d_x, m, K, *W, d_y, st);
    if (e != cudaSuccess) return cuda_fail(e, "qmatmul_affine4 launch");
    return MTP_OK;
  }
  if (!d_ws || ws_bytes < qmatmul_affine4_workspace_bytes(m, K))
    return fail(MTP_ERR_WORKSPACE, "qmatmul_affine4: workspace too small");
  Carve cv(d_ws);
  const size_t G = K / kGroup;
  uint4* xp = cv.take<uint4>(xpack_bytes(m, K));
  float2* xs = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(xp) + xpack_xs_offset(m, K));
  const GemvScratch sc = carve_scratch(cv);
  GemvParams p = {};
  s = qmat_cached(&p.mat[0], *W, "qmatmul_affine4 weight");
  if (s != MTP_OK) return s;
  p.xp = xp;
  p.xs = xs;
  p.m = m;
  p.K = K;
  p.nseg = 1;
  p.seg[0] = plain_seg(tiles_of(N), N, 0, d_y, N, nullptr);
  p.err = &header(d_ws)->err;
  cudaError_t e = launch_pack(d_x, m, K, xp, xs, st);
  if (e == cudaSuccess) e = launch_gemv(1, m > 8 ? 2 : 1, kEpiStore, p, tiles_of(N), sc, st);
  if (e != cudaSuccess) return cuda_fail(e, "qmatmul_affine4 launch");
  return MTP_OK;
}

// ------------------------------------------------------------------ rmsnorm
mtp_status rmsnorm_residual(const float* d_a, const float* d_delta, const float* d_w,
                            float* d_out_norm, float* d_out_sum, int32_t rows, int32_t dim,
                            float eps, void* stream) {
  if (!d_a || !d_w || !d_out_norm) return fail(MTP_ERR_INVALID_ARG, "rmsnorm_residual: null pointer");
  if (rows <= 0 || rows > 65535 || dim <= 0 || dim % 32)
    return fail(MTP_ERR_UNSUPPORTED, "rmsnorm_residual: rows in 1..65535, dim a multiple of 32");
  if (!(eps >= 0.f)) return fail(MTP_ERR_INVALID_ARG, "rmsnorm_residual: eps must be >= 0");
  if (!aligned16(d_a) || !aligned16(d_w) || (d_delta && !aligned16(d_delta)) || !aligned16(d_out_norm) ||
      (d_out_sum && !aligned16(d_out_sum)))
    return fail(MTP_ERR_INVALID_ARG, "rmsnorm_residual: pointers must be 16-byte aligned");
  if (d_out_norm == d_a || d_out_norm == d_delta)
    return fail(MTP_ERR_INVALID_ARG, "rmsnorm_residual: out_norm may not alias an input");
  NormSeg sg = {};
  sg.src = d_a;
  sg.delta = d_delta;
  sg.w = d_w;
  sg.eps = eps;
  sg.dim = dim;
  sg.src_ld = dim;
  sg.out_sum = d_out_sum;
  sg.out_norm = d_out_norm;
  cudaError_t e = launch_norm_pack(&sg, 1, rows, nullptr, nullptr, nullptr,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm_residual launch");
  return MTP_OK;
}

// ------------------------------------------------------------------ attention
static mtp_status check_geom(const mtp_attn_geom* g, int m) {
  if (!g) return fail(MTP_ERR_INVALID_ARG, "attention geometry: null");
  if (g->n_heads <= 0 || g->n_kv_heads <= 0 || g->n_heads % g->n_kv_heads)
    return fail(MTP_ERR_INVALID_ARG, "attention: n_kv_heads must divide n_heads");
  if (g->n_kv_heads > 64) return fail(MTP_ERR_UNSUPPORTED, "attention: at most 64 KV heads");
  if (g->head_dim_qk <= 0 || g->head_dim_qk % 32 || g->head_dim_qk > 256 ||
      g->head_dim_v <= 0 || g->head_dim_v % 32 || g->head_dim_v > 256)
    return fail(MTP_ERR_UNSUPPORTED, "attention: head dims must be multiples of 32, <= 256");
  if (g->rot_dim < 0 || g->rot_dim % 2 || g->rot_dim > g->head_dim_qk)
    return fail(MTP_ERR_INVALID_ARG, "attention: rot_dim must be even and <= head_dim_qk");
  if (g->gated_q && g->head_dim_v != g->head_dim_qk)
    return fail(MTP_ERR_UNSUPPORTED, "attention: gated q needs head_dim_v == head_dim_qk");
  if (m < 1 || m > 16) return fail(MTP_ERR_UNSUPPORTED, "attention: m must be in 1..16");
  if ((g->n_heads / g->n_kv_heads) * m > 16)
    return fail(MTP_ERR_UNSUPPORTED, "attention: (n_heads/n_kv_heads)*m must be <= 16");
  if (!attn_supported((g->n_heads / g->n_kv_heads) * m, g->head_dim_qk, g->head_dim_v, m))
    return fail(MTP_ERR_UNSUPPORTED, "attention: query rows and head dims exceed one CTA");
  if (!(g->eps >= 0.f) || !(g->scale >= 0.f))
    return fail(MTP_ERR_INVALID_ARG, "attention: eps and scale must be >= 0");
  return MTP_OK;
}

size_t attn_decode_sink_workspace_bytes(const mtp_attn_geom* g, int32_t m, int32_t cache_len) {
  if (!g || g->n_kv_heads <= 0 || m <= 0 || cache_len < 0) return 0;
  const int cached = g->window > 0 ? std::min(cache_len, g->window - 1) : cache_len;
  const int ns = attn_splits_bound(g->n_kv_heads, cached);
  const int qg = (g->n_heads / g->n_kv_heads) * m;
  return sizeof(WsHeader) + align256(attn_part_bytes(g->n_kv_heads, ns, qg, g->head_dim_v)) + 256;
}

static AttnParams make_attn(const mtp_attn_geom* g, const float* qp, const float* kp,
                            const float* vp, const float* qn, const float* kn, const float* rope,
                            const float* sinks, float* kc, float* vc, int L, int cap, int m) {
  AttnParams a = {};
  a.nh = g->n_heads;
  a.nkv = g->n_kv_heads;
  a.dqk = g->head_dim_qk;
  a.dv = g->head_dim_v;
  a.rot = g->rot_dim;
  a.window = g->window;
  a.gated = g->gated_q ? 1 : 0;
  a.eps = g->eps;
  a.scale = g->scale > 0.f ? g->scale : 1.f / std::sqrt((float)g->head_dim_qk);
  a.qp = qp;
  a.kp = kp;
  a.vp = vp;
  a.qn = qn;
  a.kn = kn;
  a.rope = rope;
  a.sinks = sinks;
  a.kc = kc;
  a.vc = vc;
  a.L = L;
  a.cap = cap;
  a.m = m;
  a.nsplit = attn_splits(a.nkv, g->window > 0 ? std::min(L, g->window - 1) : L,
                         (a.nh / a.nkv) * m, a.dqk, a.dv, m);
  a.merge_in_kernel = 1;
  return a;
}

// Every check of attn_decode_sink's arguments except the workspace (shared
// with attn_decode_sink_noalloc, which runs it before touching its scratch).
static mtp_status check_attn_args(const mtp_attn_geom* g, const float* d_qp, const float* d_kp,
                                  const float* d_vp, const float* d_rope, const float* d_k_cache,
                                  const float* d_v_cache, int32_t cache_len, int32_t cache_cap,
                                  int32_t m, const float* d_out, const char* who) {
  mtp_status s = check_geom(g, m);
  if (s != MTP_OK) return s;
  const std::string w(who);
  if (!d_qp || !d_kp || !d_vp || !d_rope || !d_k_cache || !d_v_cache || !d_out)
    return fail(MTP_ERR_INVALID_ARG, w + ": null pointer");
  if (!aligned16(d_qp) || !aligned16(d_kp) || !aligned16(d_vp) || !aligned16(d_k_cache) ||
      !aligned16(d_v_cache) || !aligned16(d_out))
    return fail(MTP_ERR_INVALID_ARG, w + ": pointers must be 16-byte aligned");
  if (cache_len < 0 || cache_cap <= 0) return fail(MTP_ERR_INVALID_ARG, w + ": bad cache length");
  if (cache_len + m > cache_cap)
    return fail(MTP_ERR_CAPACITY, w + ": cache_len + m exceeds the cache capacity");
  return MTP_OK;
}

mtp_status attn_decode_sink(const mtp_attn_geom* g, const float* d_qp, const float* d_kp,
                            const float* d_vp, const float* d_q_norm, const float* d_k_norm,
                            const float* d_rope, const float* d_sinks, float* d_k_cache,
                            float* d_v_cache, int32_t cache_len, int32_t cache_cap, int32_t m,
                            float* d_out, void* d_ws, size_t ws_bytes, void* stream) {
  mtp_status s = check_attn_args(g, d_qp, d_kp, d_vp, d_rope, d_k_cache, d_v_cache, cache_len,
                                 cache_cap, m, d_out, "attn_decode_sink");
  if (s != MTP_OK) return s;
  if (!d_ws || ws_bytes < attn_decode_sink_workspace_bytes(g, m, cache_len))
    return fail(MTP_ERR_WORKSPACE, "attn_decode_sink: workspace too small");
  AttnParams a = make_attn(g, d_qp, d_kp, d_vp, d_q_norm, d_k_norm, d_rope, d_sinks, d_k_cache,
                           d_v_cache, cache_len, cache_cap, m);
  Carve cv(d_ws);
  a.part = cv.take<float>(attn_part_bytes(a.nkv, a.nsplit, (a.nh / a.nkv) * m, a.dv));
  a.counters = header(d_ws)->counters + kCntAttn;
  a.err = &header(d_ws)->err;
  a.out = d_out;
  cudaError_t e = launch_attn(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_sink launch");
  return MTP_OK;
}

// ------------------------------------------------------------------ lm head
size_t lmhead_argmax_workspace_bytes(int32_t hidden, int32_t vocab) {
  if (hidden <= 0 || vocab <= 0) return 0;
  Carve cv(nullptr);
  cv.take<uint8_t>(xpack_bytes(1, hidden));
  cv.take<uint8_t>(8 * 4096);
  carve_scratch(cv);
  return cv.off + 256;
}

static mtp_status enqueue_head(const float* y_src, const float* norm_w, float eps, int H,
                               const mtp_affine4& W, int32_t* tok, float* val, float* logits,
                               float* y_normed, uint4* xp, float2* xs, unsigned long long* partial,
                               const GemvScratch& sc, void* ws, cudaStream_t st) {
  NormSeg sg = {};
  sg.src = y_src;
  sg.w = norm_w;
  sg.eps = eps;
  sg.dim = H;
  sg.src_ld = H;
  sg.out_norm = y_normed;
  cudaError_t e = launch_norm_pack(&sg, 1, 1, xp, xs, &header(ws)->err, st);
  if (e != cudaSuccess) return cuda_fail(e, "lm head norm launch");
  GemvParams p = {};
  mtp_status s = qmat_cached(&p.mat[0], W, "lm_head");
  if (s != MTP_OK) return s;
  p.xp = xp;
  p.xs = xs;
  p.m = 1;
  p.K = H;
  p.nseg = 1;
  p.seg[0] = plain_seg(tiles_of(W.n), W.n, 0, nullptr, W.n, nullptr);
  p.am_partial = partial;
  p.am_counter = header(ws)->counters + kCntArgmax;
  p.am_token = tok;
  p.am_value = val;
  p.logits = logits;
  p.err = &header(ws)->err;
  e = launch_gemv(1, 1, kEpiArgmax, p, tiles_of(W.n), sc, st);
  if (e != cudaSuccess) return cuda_fail(e, "lm head launch");
  return MTP_OK;
}

mtp_status lmhead_argmax(const float* d_y, const float* d_norm_w, float eps,
                         const mtp_affine4* W, int32_t* d_token, float* d_value, float* d_logits,
                         float* d_y_normed, void* d_ws, size_t ws_bytes, void* stream) {
  if (!d_y || !d_token || !d_value) return fail(MTP_ERR_INVALID_ARG, "lmhead_argmax: null pointer");
  mtp_status s = check_affine(W, -1, -1, "lm_head", true);
  if (s != MTP_OK) return s;
  if (!aligned16(d_y) || (d_norm_w && !aligned16(d_norm_w)) || (d_logits && !aligned16(d_logits)) ||
      (d_y_normed && !aligned16(d_y_normed)))
    return fail(MTP_ERR_INVALID_ARG, "lmhead_argmax: pointers must be 16-byte aligned");
  if (!(eps >= 0.f)) return fail(MTP_ERR_INVALID_ARG, "lmhead_argmax: eps must be >= 0");
  if (!d_ws || ws_bytes < lmhead_argmax_workspace_bytes(W->k, W->n))
    return fail(MTP_ERR_WORKSPACE, "lmhead_argmax: workspace too small");
  Carve cv(d_ws);
  const int H = W->k;
  uint4* xp = cv.take<uint4>(xpack_bytes(1, H));
  float2* xs = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(xp) + xpack_xs_offset(1, H));
  auto* partial = cv.take<unsigned long long>(8 * 4096);
  const GemvScratch sc = carve_scratch(cv);
  return enqueue_head(d_y, d_norm_w, eps, H, *W, d_token, d_value, d_logits, d_y_normed, xp, xs,
                      partial, sc, d_ws, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ verify head
size_t verify_head_workspace_bytes(int32_t rows, int32_t hidden, int32_t vocab) {
  if (rows <= 0 || hidden <= 0 || vocab <= 0) return 0;
  Carve cv(nullptr);
  cv.take<uint8_t>(xpack_bytes(rows, hidden));
  cv.take<float>((size_t)rows * vocab * sizeof(float));
  cv.take<unsigned long long>(16 * sizeof(unsigned long long));
  cv.take<unsigned>(16 * sizeof(unsigned));
  carve_scratch(cv);
  return cv.off + 256;
}

mtp_status verify_head_argmax(const float* d_h, int32_t rows, const float* d_norm_w, float eps,
                              const mtp_affine4* W, float logit_multiplier, float softcap,
                              int32_t* d_tokens, float* d_values, float* d_logits, void* d_ws,
                              size_t ws_bytes, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!d_h || !d_tokens || !d_values)
    return fail(MTP_ERR_INVALID_ARG, "verify_head_argmax: null pointer");
  if (rows < 1 || rows > 16) return fail(MTP_ERR_UNSUPPORTED, "verify_head_argmax: rows must be in 1..16");
  mtp_status s = check_affine(W, -1, -1, "lm_head", true);
  if (s != MTP_OK) return s;
  if (!aligned16(d_h) || (d_norm_w && !aligned16(d_norm_w)) || (d_logits && !aligned16(d_logits)))
    return fail(MTP_ERR_INVALID_ARG, "verify_head_argmax: pointers must be 16-byte aligned");
  if (!(eps >= 0.f)) return fail(MTP_ERR_INVALID_ARG, "verify_head_argmax: eps must be >= 0");
  if (!std::isfinite(logit_multiplier) || std::isnan(softcap) || std::isinf(softcap))
    return fail(MTP_ERR_INVALID_ARG, "verify_head_argmax: multiplier and softcap must be finite");
  const int H = W->k, V = W->n;
  if (!d_ws || ws_bytes < verify_head_workspace_bytes(rows, H, V))
    return fail(MTP_ERR_WORKSPACE, "verify_head_argmax: workspace too small");
  Carve cv(d_ws);
  uint4* xp = cv.take<uint4>(xpack_bytes(rows, H));
  float2* xs = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(xp) + xpack_xs_offset(rows, H));
  float* own_logits = cv.take<float>((size_t)rows * V * sizeof(float));
  auto* keys = cv.take<unsigned long long>(16 * sizeof(unsigned long long));
  auto* cnt = cv.take<unsigned>(16 * sizeof(unsigned));
  const GemvScratch sc = carve_scratch(cv);
  float* logits = d_logits ? d_logits : own_logits;
  // 1. final norm of every row, packed for the projection
  NormSeg sg = {};
  sg.src = d_h;
  sg.w = d_norm_w;
  sg.eps = eps;
  sg.dim = H;
  sg.src_ld = H;
  cudaError_t e = launch_norm_pack(&sg, 1, rows, xp, xs, &header(d_ws)->err, st);
  if (e != cudaSuccess) return cuda_fail(e, "verify head norm launch");
  // 2. logits of all rows in one pass over the vocabulary matrix
  GemvParams p = {};
  s = qmat_cached(&p.mat[0], *W, "lm_head");
  if (s != MTP_OK) return s;
  p.xp = xp;
  p.xs = xs;
  p.m = rows;
  p.K = H;
  p.nseg = 1;
  p.seg[0] = plain_seg(tiles_of(V), V, 0, logits, V, nullptr);
  p.err = &header(d_ws)->err;
  e = launch_gemv(1, rows > 8 ? 2 : 1, kEpiStore, p, tiles_of(V), sc, st);
  if (e != cudaSuccess) return cuda_fail(e, "verify head projection launch");
  // 3. multiplier, softcap and argmax per row
  e = launch_rows_argmax(logits, rows, V, logit_multiplier, softcap, d_tokens, d_values, keys, cnt,
                         st);
  if (e != cudaSuccess) return cuda_fail(e, "verify head argmax launch");
  return MTP_OK;
}

// ------------------------------------------------------------------ MoE
static mtp_status check_moe(const mtp_moe_weights* w, int H) {
  if (!w || !w->router) return fail(MTP_ERR_INVALID_ARG, "moe: null weights");
  if (w->n_experts <= 0 || w->n_experts > 1024)
    return fail(MTP_ERR_UNSUPPORTED, "moe: n_experts must be in 1..1024");
  if (w->top_k < 1 || w->top_k > 16 || w->top_k > w->n_experts)
    return fail(MTP_ERR_UNSUPPORTED, "moe: top_k must be in 1..min(16, n_experts)");
  if (w->expert_inter <= 0 || w->expert_inter % 256)
    return fail(MTP_ERR_UNSUPPORTED, "moe: expert_inter must be a multiple of 256");
  if (w->shared_inter != w->expert_inter)
    return fail(MTP_ERR_UNSUPPORTED, "moe: shared_inter must equal expert_inter");
  if (H > 16384) return fail(MTP_ERR_UNSUPPORTED, "moe: hidden must be <= 16384");
  const int E = w->n_experts, I = w->expert_inter;
  mtp_status s;
  if ((s = check_affine(&w->exp_gate, E * I, H, "exp_gate", true)) != MTP_OK) return s;
  if ((s = check_affine(&w->exp_up, E * I, H, "exp_up", true)) != MTP_OK) return s;
  if ((s = check_affine(&w->exp_down, E * H, I, "exp_down", true)) != MTP_OK) return s;
  if ((s = check_affine(&w->sh_gate, I, H, "sh_gate", true)) != MTP_OK) return s;
  if ((s = check_affine(&w->sh_up, I, H, "sh_up", true)) != MTP_OK) return s;
  if ((s = check_affine(&w->sh_down, H, I, "sh_down", true)) != MTP_OK) return s;
  if (!w->sh_gate_inp) return fail(MTP_ERR_INVALID_ARG, "moe: null sh_gate_inp");
  if (w->scales_bf16 != 0 && w->scales_bf16 != 1)
    return fail(MTP_ERR_INVALID_ARG, "moe: scales_bf16 must be 0 or 1");
  if (w->scales_bf16 && (H % 256 || I % 256))
    return fail(MTP_ERR_UNSUPPORTED, "moe: bfloat16 stacks need hidden and expert_inter multiples of 256");
  if (!aligned16(w->router)) return fail(MTP_ERR_INVALID_ARG, "moe: router must be 16-byte aligned");
  return MTP_OK;
}

struct MoeScratch {
  GemvScratch gemv;
  float* logits;
  int* sel;
  float* weight;
  uint4* xp_f;
  float2* xs_f;
  uint4* xp_h;
  float2* xs_h;
};

static void carve_moe(Carve& cv, const mtp_moe_weights* w, int H, MoeScratch* m) {
  m->logits = cv.take<float>(sizeof(float) * w->n_experts);
  m->sel = cv.take<int>(sizeof(int) * 16);
  m->weight = cv.take<float>(sizeof(float) * 17);
  m->xp_f = cv.take<uint4>(xpack_bytes(1, H));
  m->xs_f = nullptr;
  m->xs_h = nullptr;
  const int Kh = (w->top_k + 1) * w->expert_inter;
  m->xp_h = cv.take<uint4>(xpack_bytes(1, Kh));
  if (m->xp_f) m->xs_f = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(m->xp_f) + xpack_xs_offset(1, H));
  if (m->xp_h) m->xs_h = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(m->xp_h) + xpack_xs_offset(1, Kh));
  m->gemv = carve_scratch(cv);
}

// Launches the router and fills the one-row phases of the experts: gate/up
// with SwiGLU over the routed and shared experts (rows chosen by the router),
// then down + residual into u2.
static mtp_status moe_router_and_phases(const mtp_moe_weights* w, const float* u1,
                                        const float* post_norm, float eps, int H, float* u2,
                                        const MoeScratch& sc, void* ws, cudaStream_t st,
                                        GemvParams* gu_out, GemvParams* dn_out, int* gu_tiles,
                                        int* dn_tiles) {
  const int E = w->n_experts, I = w->expert_inter, K = w->top_k;
  RouterParams r = {};
  r.u1 = u1;
  r.post_norm = post_norm;
  r.eps = eps;
  r.H = H;
  r.router = w->router;
  r.E = E;
  r.top_k = K;
  r.sh_gate_inp = w->sh_gate_inp;
  r.logits = sc.logits;
  r.counter = header(ws)->counters + kCntRouter;
  r.sel = sc.sel;
  r.weight = sc.weight;
  r.xp = sc.xp_f;
  r.xs = sc.xs_f;
  r.err = &header(ws)->err;
  cudaError_t e = launch_router(r, st);
  if (e != cudaSuccess) return cuda_fail(e, "moe router launch");

  // routed + shared expert gate/up with SwiGLU, scaled by the routing weights
  GemvParams p = {};
  mtp_status s;
  const bool bf = w->scales_bf16 != 0;
  if ((s = qmat_cached(&p.mat[0], w->exp_gate, "exp_gate", bf)) != MTP_OK) return s;
  if ((s = qmat_cached(&p.mat[1], w->exp_up, "exp_up", bf)) != MTP_OK) return s;
  p.sbf_mask = bf ? 0x3 : 0;  // routed stacks in slots 0 and 1, the shared expert f32
  if ((s = qmat_cached(&p.mat[2], w->sh_gate, "sh_gate")) != MTP_OK) return s;
  if ((s = qmat_cached(&p.mat[3], w->sh_up, "sh_up")) != MTP_OK) return s;
  p.xp = sc.xp_f;
  p.xs = sc.xs_f;
  p.m = 1;
  p.K = H;
  const int tpe = tiles_of(I);
  p.nseg = K + 1;
  for (int i = 0; i <= K; ++i) {
    GemvSeg g = plain_seg((i + 1) * tpe, I, i < K ? 0 : 2, nullptr, 0, nullptr);
    g.sel_idx = i < K ? i : -1;
    g.row_mult = I;
    g.w_idx = i;
    g.out_col0 = i * I;
    p.seg[i] = g;
  }
  p.rowsel = sc.sel;
  p.segw = sc.weight;
  p.rowsel_after_wait = 1;
  p.out_xp = sc.xp_h;
  p.out_xs = sc.xs_h;
  p.out_m = 1;
  p.err = &header(ws)->err;
  p.epi = kEpiSwiglu;

  // down projections over the concatenated expert activations, + residual
  GemvParams d = {};
  if ((s = qmat_cached(&d.mat[0], w->exp_down, "exp_down", bf)) != MTP_OK) return s;
  d.sbf_mask = bf ? 0x1 : 0;
  if ((s = qmat_cached(&d.mat[1], w->sh_down, "sh_down")) != MTP_OK) return s;
  d.xp = sc.xp_h;
  d.xs = sc.xs_h;
  d.m = 1;
  d.K = (K + 1) * I;
  d.nseg = 1;
  d.seg[0] = plain_seg(tiles_of(H), H, 0, u2, H, u1);
  d.rowsel = sc.sel;
  d.rowsel_after_wait = 1;
  d.kseg_len = I;
  d.nkseg = K + 1;
  d.kseg_row_mult = H;
  d.kseg_last_mat = 1;
  d.err = &header(ws)->err;
  d.epi = kEpiStore;
  *gu_out = p;
  *dn_out = d;
  *gu_tiles = (K + 1) * tpe;
  *dn_tiles = tiles_of(H);
  return MTP_OK;
}

// The MoE FFN alone: router, gate/up launch, down launch.
static mtp_status enqueue_moe(const mtp_moe_weights* w, const float* u1, const float* post_norm,
                              float eps, int H, float* u2, const MoeScratch& sc, void* ws,
                              cudaStream_t st) {
  GemvParams gu = {}, dn = {};
  int tg = 0, td = 0;
  mtp_status s = moe_router_and_phases(w, u1, post_norm, eps, H, u2, sc, ws, st, &gu, &dn, &tg, &td);
  if (s != MTP_OK) return s;
  cudaError_t e = launch_gemv(2, 1, kEpiSwiglu, gu, tg, sc.gemv, st);
  if (e != cudaSuccess) return cuda_fail(e, "moe expert gate/up launch");
  e = launch_gemv(1, 1, kEpiStore, dn, td, sc.gemv, st);
  if (e != cudaSuccess) return cuda_fail(e, "moe expert down launch");
  return MTP_OK;
}

size_t moe_ffn_workspace_bytes(const mtp_moe_weights* w, int32_t hidden) {
  if (!w || hidden <= 0 || w->n_experts <= 0 || w->top_k <= 0) return 0;
  Carve cv(nullptr);
  MoeScratch sc;
  carve_moe(cv, w, hidden, &sc);
  return cv.off + 256;
}

mtp_status moe_ffn(const mtp_moe_weights* w, const float* d_u1, const float* d_post_norm,
                   float eps, int32_t hidden, float* d_u2, int32_t* d_sel, float* d_weight,
                   void* d_ws, size_t ws_bytes, void* stream) {
  if (!d_u1 || !d_post_norm || !d_u2) return fail(MTP_ERR_INVALID_ARG, "moe_ffn: null pointer");
  if (hidden <= 0 || hidden % 128) return fail(MTP_ERR_UNSUPPORTED, "moe_ffn: hidden % 128 != 0");
  mtp_status s = check_moe(w, hidden);
  if (s != MTP_OK) return s;
  if (!aligned16(d_u1) || !aligned16(d_u2))
    return fail(MTP_ERR_INVALID_ARG, "moe_ffn: pointers must be 16-byte aligned");
  if (d_u2 == d_u1) return fail(MTP_ERR_INVALID_ARG, "moe_ffn: u2 may not alias u1");
  if (!d_ws || ws_bytes < moe_ffn_workspace_bytes(w, hidden))
    return fail(MTP_ERR_WORKSPACE, "moe_ffn: workspace too small");
  Carve cv(d_ws);
  MoeScratch sc;
  carve_moe(cv, w, hidden, &sc);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = enqueue_moe(w, d_u1, d_post_norm, eps, hidden, d_u2, sc, d_ws, st);
  if (s != MTP_OK) return s;
  cudaError_t e = cudaSuccess;
  if (d_sel) e = cudaMemcpyAsync(d_sel, sc.sel, sizeof(int) * w->top_k, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && d_weight)
    e = cudaMemcpyAsync(d_weight, sc.weight, sizeof(float) * (w->top_k + 1),
                        cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "moe_ffn routing copy");
  return MTP_OK;
}

// ------------------------------------------------------------------ layer
struct LayerWs {
  uint4* xa;
  float2* xsa;
  uint4* xb;
  float2* xsb;
  float *u, *u1, *u2, *qp, *kp, *vp;
  float* part;
  unsigned long long* am_partial;
  float *ss0, *ss1, *ss2;  // per-tile sums of squares of u, u1, u2 (folded RMSNorms)
  float* ss_pre;           // per-group raw sums of squares of the embedding and hidden rows
  GemvScratch gemv;
  MoeScratch moe;
};

static int layer_kmax(const mtp_layer_desc* L) {
  const int H = L->hidden;
  int k = 2 * H;
  k = std::max(k, L->attn.n_heads * L->attn.head_dim_v);
  if (L->moe) k = std::max(k, (L->moe->top_k + 1) * L->moe->expert_inter);
  else k = std::max(k, L->intermediate);
  return k;
}

static void carve_layer(Carve& cv, const mtp_layer_desc* L, int m, LayerWs* w) {
  const int H = L->hidden;
  const int Kmax = layer_kmax(L);
  const mtp_attn_geom& g = L->attn;
  const int qrows = g.n_heads * g.head_dim_qk * (g.gated_q ? 2 : 1);
  auto xp_pair = [&](uint4** xp, float2** xs) {
    *xp = cv.take<uint4>(xpack_bytes(m, Kmax));
    *xs = *xp ? reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(*xp) + xpack_xs_offset(m, Kmax))
              : nullptr;
  };
  xp_pair(&w->xa, &w->xsa);
  xp_pair(&w->xb, &w->xsb);
  w->u = cv.take<float>(sizeof(float) * m * H);
  w->u1 = cv.take<float>(sizeof(float) * m * H);
  w->u2 = cv.take<float>(sizeof(float) * m * H);
  w->qp = cv.take<float>(sizeof(float) * m * qrows);
  w->kp = cv.take<float>(sizeof(float) * m * g.n_kv_heads * g.head_dim_qk);
  w->vp = cv.take<float>(sizeof(float) * m * g.n_kv_heads * g.head_dim_v);
  const int cached = g.window > 0 ? std::min(L->cache_cap, g.window - 1) : L->cache_cap;
  const int ns = attn_splits_bound(g.n_kv_heads, cached);
  w->part = cv.take<float>(attn_part_bytes(g.n_kv_heads, ns, (g.n_heads / g.n_kv_heads) * m,
                                           g.head_dim_v));
  w->am_partial = cv.take<unsigned long long>(8 * 4096);
  w->ss0 = cv.take<float>(sizeof(float) * m * (H / kGroup));
  w->ss1 = cv.take<float>(sizeof(float) * m * (H / kGroup));
  w->ss2 = cv.take<float>(sizeof(float) * m * (H / kGroup));
  w->ss_pre = cv.take<float>(sizeof(float) * 2 * (H / kGroup));
  w->gemv = carve_scratch(cv);
  if (L->moe) carve_moe(cv, L->moe, H, &w->moe);
}

static mtp_status check_layer(const mtp_layer_desc* L, int m) {
  if (!L) return fail(MTP_ERR_INVALID_ARG, "layer descriptor is null");
  const int H = L->hidden;
  if (H <= 0 || H % 128) return fail(MTP_ERR_UNSUPPORTED, "layer: hidden must be a multiple of 128");
  if (L->vocab <= 0) return fail(MTP_ERR_INVALID_ARG, "layer: vocab must be positive");
  mtp_status s = check_geom(&L->attn, m);
  if (s != MTP_OK) return s;
  const mtp_attn_geom& g = L->attn;
  if ((g.n_heads * g.head_dim_v) % 128)
    return fail(MTP_ERR_UNSUPPORTED, "layer: n_heads*head_dim_v must be a multiple of 128");
  if (!(L->eps >= 0.f)) return fail(MTP_ERR_INVALID_ARG, "layer: eps must be >= 0");
  const float* norms[] = {L->enorm, L->hnorm, L->attn_norm, L->post_norm, L->final_norm};
  for (const float* p : norms)
    if (!p || !aligned16(p))
      return fail(MTP_ERR_INVALID_ARG, "layer: norm weights must be non-null and 16-byte aligned");
  const int qrows = g.n_heads * g.head_dim_qk * (g.gated_q ? 2 : 1);
  if ((s = check_affine(&L->eh_proj, H, 2 * H, "eh_proj", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->wq, qrows, H, "wq", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->wk, g.n_kv_heads * g.head_dim_qk, H, "wk", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->wv, g.n_kv_heads * g.head_dim_v, H, "wv", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->wo, H, g.n_heads * g.head_dim_v, "wo", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->lm_head, L->vocab, H, "lm_head", true)) != MTP_OK) return s;
  if (L->moe) {
    if (m != 1) return fail(MTP_ERR_UNSUPPORTED, "layer: the MoE FFN supports m = 1");
    if ((s = check_moe(L->moe, H)) != MTP_OK) return s;
  } else {
    const int I = L->intermediate;
    if (I <= 0 || I % 128)
      return fail(MTP_ERR_UNSUPPORTED, "layer: intermediate must be a multiple of 128");
    if ((s = check_affine(&L->ffn_gate, I, H, "ffn_gate", true)) != MTP_OK) return s;
    if ((s = check_affine(&L->ffn_up, I, H, "ffn_up", true)) != MTP_OK) return s;
    if ((s = check_affine(&L->ffn_down, H, I, "ffn_down", true)) != MTP_OK) return s;
  }
  if (!L->rope || !L->k_cache || !L->v_cache || L->cache_cap <= 0)
    return fail(MTP_ERR_INVALID_ARG, "layer: rope table and KV cache are required");
  if (!aligned16(L->k_cache) || !aligned16(L->v_cache) || (L->embed && !aligned16(L->embed)))
    return fail(MTP_ERR_INVALID_ARG, "layer: cache and embedding must be 16-byte aligned");
  return MTP_OK;
}

size_t mtp_draft_workspace_bytes(const mtp_layer_desc* L, int32_t m) {
  if (!L || m <= 0 || L->hidden <= 0 || L->attn.n_kv_heads <= 0 || L->attn.n_heads <= 0) return 0;
  Carve cv(nullptr);
  LayerWs w;
  carve_layer(cv, L, m, &w);
  return cv.off + 256;
}

static mtp_status enqueue_layer(const mtp_layer_desc* L, const mtp_step_in* in,
                                const mtp_step_out* out, void* ws, cudaStream_t st) {
  const int H = L->hidden, m = in->m;
  const mtp_attn_geom& g = L->attn;
  Carve cv(ws);
  LayerWs w;
  carve_layer(cv, L, m, &w);
  int* err = &header(ws)->err;
  cudaError_t e;
  mtp_status s;

  // 1. embedding gather + enorm/hnorm, packed [e_n ; h_n]
  NormSeg segs[2] = {};
  if (L->embed) {
    segs[0].table = L->embed;
    segs[0].tokens = in->d_tokens;
    segs[0].vocab = L->vocab;
  } else {
    segs[0].src = in->d_embed_rows;
  }
  segs[0].w = L->enorm;
  segs[0].eps = 1e-6f;
  segs[0].dim = H;
  segs[0].src_ld = H;
  segs[1].src = in->d_hidden;
  segs[1].w = L->hnorm;
  segs[1].eps = 1e-6f;
  segs[1].dim = H;
  segs[1].src_ld = H;
  // one activation row: consecutive projections share one launch (phases), and
  // the embedding/hidden pack runs inside it (its RMSNorms fold into eh_proj)
  const bool rows = (m == 1);
  const bool pre_pack = rows && H % 256 == 0;
  PreParams pre_a = {};
  if (pre_pack) {
    pre_a.kind = kPreEmbedPack;
    pre_a.units = 2 * H / kGroup;
    pre_a.xp = w.xa;
    pre_a.xs = w.xsa;
    pre_a.table = L->embed;
    pre_a.tokens = in->d_tokens;
    pre_a.vocab = L->vocab;
    pre_a.rows = in->d_embed_rows;
    pre_a.hidden = in->d_hidden;
    pre_a.w0 = L->enorm;
    pre_a.w1 = L->hnorm;
    pre_a.dim = H;
    pre_a.eps = 1e-6f;
    pre_a.ss = w.ss_pre;
  } else if ((e = launch_norm_pack(segs, 2, m, w.xa, w.xsa, err, st)) != cudaSuccess) {
    return cuda_fail(e, "eh norm launch");
  }

  // 2. u = eh_proj [e_n ; h_n]
  GemvParams p = {};
  if ((s = qmat_cached(&p.mat[0], L->eh_proj, "eh_proj")) != MTP_OK) return s;
  p.xp = w.xa;
  p.xs = w.xsa;
  p.m = m;
  p.K = 2 * H;
  p.nseg = 1;
  p.seg[0] = plain_seg(tiles_of(H), H, 0, w.u, H, nullptr);
  p.err = err;
  // the attention RMSNorm is folded into the q/k/v projection: pack u * attn_norm
  // and the per-tile sums of u^2 here, scale the projections' rows there
  const int ht = H / kGroup;
  p.pack_w = L->attn_norm;
  p.pack_c0 = 0;
  p.out_xp = w.xb;
  p.out_xs = w.xsb;
  p.out_m = m;
  p.ss_out = w.ss0;
  p.epi = kEpiStore;
  const int nt = m > 8 ? 2 : 1;
  if (!rows && (e = launch_gemv(1, nt, kEpiStore, p, tiles_of(H), w.gemv, st)) != cudaSuccess)
    return cuda_fail(e, "eh_proj launch");

  // 3. x = RMSNorm(u) * attn_norm: folded (rows of step 4 scaled by rsqrt(mean u^2 + eps))

  // 4. q (+gate), k, v projections in one launch
  const int qrows = g.n_heads * g.head_dim_qk * (g.gated_q ? 2 : 1);
  const int krows = g.n_kv_heads * g.head_dim_qk, vrows = g.n_kv_heads * g.head_dim_v;
  GemvParams q = {};
  if ((s = qmat_cached(&q.mat[0], L->wq, "wq")) != MTP_OK) return s;
  if ((s = qmat_cached(&q.mat[1], L->wk, "wk")) != MTP_OK) return s;
  if ((s = qmat_cached(&q.mat[2], L->wv, "wv")) != MTP_OK) return s;
  q.xp = w.xb;
  q.xs = w.xsb;
  q.m = m;
  q.K = H;
  q.nseg = 3;
  q.in_ss = w.ss0;
  q.in_ss_n = ht;
  q.in_ss_dim = H;
  q.in_ss_eps = L->eps;
  const int tq = tiles_of(qrows), tk = tiles_of(krows), tv = tiles_of(vrows);
  q.seg[0] = plain_seg(tq, qrows, 0, w.qp, qrows, nullptr);
  q.seg[1] = plain_seg(tq + tk, krows, 1, w.kp, krows, nullptr);
  q.seg[2] = plain_seg(tq + tk + tv, vrows, 2, w.vp, vrows, nullptr);
  q.err = err;
  q.epi = kEpiStore;
  if (rows) {
    GemvParams ph[2] = {p, q};
    const int tl[2] = {tiles_of(H), tq + tk + tv};
    if ((e = launch_gemv_rows(ph, tl, 2, w.gemv, err, st, pre_pack ? &pre_a : nullptr)) !=
        cudaSuccess)
      return cuda_fail(e, "eh_proj + qkv launch");
  } else if ((e = launch_gemv(1, nt, kEpiStore, q, tq + tk + tv, w.gemv, st)) != cudaSuccess) {
    return cuda_fail(e, "qkv launch");
  }

  // 5. attention (norm + rope + append + split-K + sink + gate), packed output
  AttnParams a = make_attn(&g, w.qp, w.kp, w.vp, L->q_norm, L->k_norm, L->rope, L->sinks,
                           L->k_cache, L->v_cache, in->cache_len, L->cache_cap, m);
  a.pos_base = in->pos_base;
  a.part = w.part;
  a.counters = header(ws)->counters + kCntAttn;
  a.err = err;
  a.prefetch_before_wait = 1;  // the q/k/v projection signals only after its own wait
  // one row, dense FFN: the next launch merges the splits before o_proj
  const bool fused_tail = rows && !L->moe;  // o, gate/up, down and lm_head in one launch
  a.merge_in_kernel = rows ? 0 : 1;  // one row: the o_proj launch merges the splits
  a.out = nullptr;
  a.out_xp = w.xa;
  a.out_xs = w.xsa;
  if ((e = launch_attn(a, st)) != cudaSuccess) return cuda_fail(e, "attention launch");
  PreParams pre_b = {};  // the split merge, as pre-units of the o_proj launch (m = 1)
  pre_b.kind = kPreAttnMerge;
  pre_b.units = g.n_heads * g.head_dim_v / kGroup;
  pre_b.xp = w.xa;
  pre_b.xs = w.xsa;
  pre_b.part = w.part;
  pre_b.part_o = attn_part_outputs(w.part, g.n_kv_heads, a.nsplit, g.n_heads / g.n_kv_heads);
  pre_b.nkv = g.n_kv_heads;
  pre_b.ns = a.nsplit;
  pre_b.G = g.n_heads / g.n_kv_heads;
  pre_b.dv = g.head_dim_v;
  pre_b.dqk = g.head_dim_qk;
  pre_b.gated = g.gated_q ? 1 : 0;
  pre_b.sinks = L->sinks;
  pre_b.qp = w.qp;

  // 6. u1 = u + W_o o
  const int ko = g.n_heads * g.head_dim_v;
  GemvParams o = {};
  if ((s = qmat_cached(&o.mat[0], L->wo, "wo")) != MTP_OK) return s;
  o.xp = w.xa;
  o.xs = w.xsa;
  o.m = m;
  o.K = ko;
  o.nseg = 1;
  o.seg[0] = plain_seg(tiles_of(H), H, 0, w.u1, H, w.u);
  o.err = err;
  if (!L->moe) {  // post-attention RMSNorm folded into the gate/up projection
    o.pack_w = L->post_norm;
    o.pack_c0 = 0;
    o.out_xp = w.xb;
    o.out_xs = w.xsb;
    o.out_m = m;
    o.ss_out = w.ss1;
  }
  o.epi = kEpiStore;
  if (rows && !fused_tail) {
    const int to = tiles_of(H);
    if ((e = launch_gemv_rows(&o, &to, 1, w.gemv, err, st, &pre_b)) != cudaSuccess)
      return cuda_fail(e, "split merge + o_proj launch");
  } else if (!fused_tail &&
             (e = launch_gemv(1, nt, kEpiStore, o, tiles_of(H), w.gemv, st)) != cudaSuccess) {
    return cuda_fail(e, "o_proj launch");
  }

  float* u2 = out->d_u2 ? out->d_u2 : w.u2;
  if (L->moe && rows) {
    // one row: the experts' gate/up, down (+ residual, final norm folded)
    // and lm_head + argmax in one launch after the router
    GemvParams gu = {}, dn = {};
    int tg = 0, td = 0;
    s = moe_router_and_phases(L->moe, w.u1, L->post_norm, L->eps, H, u2, w.moe, ws, st, &gu, &dn,
                              &tg, &td);
    if (s != MTP_OK) return s;
    dn.pack_w = L->final_norm;
    dn.pack_c0 = 0;
    dn.out_xp = w.xb;
    dn.out_xs = w.xsb;
    dn.out_m = 1;
    dn.ss_out = w.ss2;
    GemvParams hd = {};
    if ((s = qmat_cached(&hd.mat[0], L->lm_head, "lm_head")) != MTP_OK) return s;
    hd.xp = w.xb;
    hd.xs = w.xsb;
    hd.m = 1;
    hd.K = H;
    hd.nseg = 1;
    hd.seg[0] = plain_seg(tiles_of(L->vocab), L->vocab, 0, nullptr, L->vocab, nullptr);
    hd.in_ss = w.ss2;
    hd.in_ss_n = ht;
    hd.in_ss_dim = H;
    hd.in_ss_eps = L->eps;
    hd.normed_src = u2;
    hd.normed_w = L->final_norm;
    hd.normed_out = out->d_hidden_out;
    hd.am_partial = w.am_partial;
    hd.am_counter = header(ws)->counters + kCntArgmax;
    hd.am_token = out->d_token;
    hd.am_value = out->d_value;
    hd.logits = out->d_logits;
    hd.err = err;
    hd.epi = kEpiArgmax;
    GemvParams ph[3] = {gu, dn, hd};
    const int tl[3] = {tg, td, tiles_of(L->vocab)};
    if ((e = launch_gemv_rows(ph, tl, 3, w.gemv, err, st)) != cudaSuccess)
      return cuda_fail(e, "experts + lm head launch");
    return MTP_OK;
  }
  if (L->moe) {
    s = enqueue_moe(L->moe, w.u1, L->post_norm, L->eps, H, u2, w.moe, ws, st);
    if (s != MTP_OK) return s;
  } else {
    // 7. f = RMSNorm(u1) * post_norm: folded into step 8
    // 8. h = silu(W_gate f) * (W_up f), packed
    const int I = L->intermediate;
    GemvParams gu = {};
    if ((s = qmat_cached(&gu.mat[0], L->ffn_gate, "ffn_gate")) != MTP_OK) return s;
    if ((s = qmat_cached(&gu.mat[1], L->ffn_up, "ffn_up")) != MTP_OK) return s;
    gu.xp = w.xb;
    gu.xs = w.xsb;
    gu.m = m;
    gu.K = H;
    gu.nseg = 1;
    gu.in_ss = w.ss1;
    gu.in_ss_n = ht;
    gu.in_ss_dim = H;
    gu.in_ss_eps = L->eps;
    gu.seg[0] = plain_seg(tiles_of(I), I, 0, nullptr, I, nullptr);
    gu.out_xp = w.xa;
    gu.out_xs = w.xsa;
    gu.out_m = m;
    gu.err = err;
    gu.epi = kEpiSwiglu;
    if (!fused_tail && (e = launch_gemv(2, nt, kEpiSwiglu, gu, tiles_of(I), w.gemv, st)) != cudaSuccess)
      return cuda_fail(e, "gate/up launch");
    // 9. u2 = u1 + W_down h
    GemvParams dn = {};
    if ((s = qmat_cached(&dn.mat[0], L->ffn_down, "ffn_down")) != MTP_OK) return s;
    dn.xp = w.xa;
    dn.xs = w.xsa;
    dn.m = m;
    dn.K = I;
    dn.nseg = 1;
    dn.seg[0] = plain_seg(tiles_of(H), H, 0, u2, H, w.u1);
    dn.err = err;
    // final RMSNorm of the last row folded into the lm_head
    dn.pack_w = L->final_norm;
    dn.pack_c0 = m - 1;
    dn.out_xp = w.xb;
    dn.out_xs = w.xsb;
    dn.out_m = 1;
    dn.ss_out = w.ss2;
    dn.epi = kEpiStore;
    if (!fused_tail && (e = launch_gemv(1, nt, kEpiStore, dn, tiles_of(H), w.gemv, st)) != cudaSuccess)
      return cuda_fail(e, "down launch");
    // 10-11. lm_head + argmax of RMSNorm(u2[m-1]) * final_norm (folded)
    GemvParams hd = {};
    if ((s = qmat_cached(&hd.mat[0], L->lm_head, "lm_head")) != MTP_OK) return s;
    hd.xp = w.xb;
    hd.xs = w.xsb;
    hd.m = 1;
    hd.K = H;
    hd.nseg = 1;
    hd.seg[0] = plain_seg(tiles_of(L->vocab), L->vocab, 0, nullptr, L->vocab, nullptr);
    hd.in_ss = w.ss2;
    hd.in_ss_n = ht;
    hd.in_ss_dim = H;
    hd.in_ss_eps = L->eps;
    hd.normed_src = u2 + (size_t)(m - 1) * H;
    hd.normed_w = L->final_norm;
    hd.normed_out = out->d_hidden_out;
    hd.am_partial = w.am_partial;
    hd.am_counter = header(ws)->counters + kCntArgmax;
    hd.am_token = out->d_token;
    hd.am_value = out->d_value;
    hd.logits = out->d_logits;
    hd.err = err;
    hd.epi = kEpiArgmax;
    if (fused_tail) {
      GemvParams ph[4] = {o, gu, dn, hd};
      const int tl[4] = {tiles_of(H), tiles_of(I), tiles_of(H), tiles_of(L->vocab)};
      if ((e = launch_gemv_rows(ph, tl, 4, w.gemv, err, st, &pre_b)) != cudaSuccess)
        return cuda_fail(e, "o_proj + gate/up + down + lm head launch");
    } else if ((e = launch_gemv(1, 1, kEpiArgmax, hd, tiles_of(L->vocab), w.gemv, st)) != cudaSuccess) {
      return cuda_fail(e, "lm head launch");
    }
    return MTP_OK;
  }

  // 10-11. final norm of the last row, lm_head + argmax
  return enqueue_head(u2 + (size_t)(m - 1) * H, L->final_norm, L->eps, H, L->lm_head,
                      out->d_token, out->d_value, out->d_logits, out->d_hidden_out, w.xa, w.xsa,
                      w.am_partial, w.gemv, ws, st);
}

mtp_status mtp_draft_forward(const mtp_layer_desc* L, const mtp_step_in* in,
                             const mtp_step_out* out, void* d_ws, size_t ws_bytes, void* stream) {
  if (!in || !out) return fail(MTP_ERR_INVALID_ARG, "mtp_draft_forward: null in/out");
  mtp_status s = check_layer(L, in->m);
  if (s != MTP_OK) return s;
  if (!in->d_hidden || !aligned16(in->d_hidden))
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_forward: hidden must be a 16-byte aligned pointer");
  if (L->embed ? !in->d_tokens : (!in->d_embed_rows || !aligned16(in->d_embed_rows)))
    return fail(MTP_ERR_INVALID_ARG,
                "mtp_draft_forward: tokens (with a table) or embedding rows are required");
  if (in->cache_len < 0 || in->pos_base < 0)
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_forward: negative cache_len or pos_base");
  if (in->cache_len + in->m > L->cache_cap)
    return fail(MTP_ERR_CAPACITY, "mtp_draft_forward: cache_len + m exceeds the cache capacity");
  if (!out->d_token || !out->d_value)
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_forward: token and value outputs are required");
  if ((out->d_hidden_out && !aligned16(out->d_hidden_out)) ||
      (out->d_u2 && !aligned16(out->d_u2)) || (out->d_logits && !aligned16(out->d_logits)))
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_forward: outputs must be 16-byte aligned");
  if (!d_ws || ws_bytes < mtp_draft_workspace_bytes(L, in->m))
    return fail(MTP_ERR_WORKSPACE, "mtp_draft_forward: workspace too small");
  return enqueue_layer(L, in, out, d_ws, static_cast<cudaStream_t>(stream));
}

mtp_status mtp_draft_chain(const mtp_layer_desc* layers, int32_t n_layers, const float* d_hidden,
                           int32_t* d_seq, const int32_t* cache_lens, int32_t m,
                           float* d_values, float* d_hidden_out, float* d_u2, float* d_logits,
                           void* d_ws, size_t ws_bytes, void* stream) {
  if (!layers || n_layers <= 0 || !d_hidden || !d_seq || !cache_lens || !d_values)
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_chain: null argument");
  size_t need = 0;
  for (int k = 0; k < n_layers; ++k) {
    mtp_status s = check_layer(&layers[k], m);
    if (s != MTP_OK) return s;
    if (!layers[k].embed) return fail(MTP_ERR_INVALID_ARG, "mtp_draft_chain: layers need an embedding table");
    if (layers[k].hidden != layers[0].hidden)
      return fail(MTP_ERR_INVALID_ARG, "mtp_draft_chain: layers must share the hidden size");
    if (d_logits && layers[k].vocab != layers[0].vocab)
      return fail(MTP_ERR_INVALID_ARG, "mtp_draft_chain: per-layer logits need one vocabulary size");
    if (cache_lens[k] < 0 || cache_lens[k] + m > layers[k].cache_cap)
      return fail(MTP_ERR_CAPACITY, "mtp_draft_chain: cache_len + m exceeds a cache capacity");
    need = std::max(need, mtp_draft_workspace_bytes(&layers[k], m));
  }
  if ((d_hidden_out && !aligned16(d_hidden_out)) || (d_u2 && !aligned16(d_u2)) ||
      (d_logits && !aligned16(d_logits)))
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_chain: outputs must be 16-byte aligned");
  if (!d_ws || ws_bytes < need) return fail(MTP_ERR_WORKSPACE, "mtp_draft_chain: workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int k = 0; k < n_layers; ++k) {
    mtp_step_in in = {};
    in.d_tokens = d_seq + k;
    in.d_hidden = d_hidden;
    in.cache_len = cache_lens[k];
    in.m = m;
    mtp_step_out out = {};
    out.d_token = d_seq + m + k;
    out.d_value = d_values + k;
    out.d_hidden_out = d_hidden_out ? d_hidden_out + (size_t)k * layers[k].hidden : nullptr;
    out.d_u2 = d_u2 ? d_u2 + (size_t)k * m * layers[k].hidden : nullptr;
    out.d_logits = d_logits ? d_logits + (size_t)k * layers[k].vocab : nullptr;
    mtp_status s = enqueue_layer(&layers[k], &in, &out, d_ws, st);
    if (s != MTP_OK) return s;
  }
  return MTP_OK;
}

mtp_status mtp_draft_steps(const mtp_layer_desc* L, int32_t k_steps, const float* d_hidden,
                           int32_t* d_tokens, int32_t cache_len, int32_t pos_base,
                           float* d_values, float* d_hidden_out, void* d_ws, size_t ws_bytes,
                           void* stream) {
  mtp_status s = check_layer(L, 1);
  if (s != MTP_OK) return s;
  if (k_steps < 1 || k_steps > 64) return fail(MTP_ERR_UNSUPPORTED, "mtp_draft_steps: k_steps must be in 1..64");
  if (!L->embed) return fail(MTP_ERR_INVALID_ARG, "mtp_draft_steps: the layer needs an embedding table");
  if (!d_hidden || !d_tokens || !d_values || !d_hidden_out)
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_steps: null argument");
  if (!aligned16(d_hidden) || !aligned16(d_hidden_out))
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_steps: hidden rows must be 16-byte aligned");
  if (cache_len < 0 || pos_base < 0)
    return fail(MTP_ERR_INVALID_ARG, "mtp_draft_steps: negative cache_len or pos_base");
  if (cache_len + k_steps > L->cache_cap)
    return fail(MTP_ERR_CAPACITY, "mtp_draft_steps: cache_len + k_steps exceeds the cache capacity");
  if (!d_ws || ws_bytes < mtp_draft_workspace_bytes(L, 1))
    return fail(MTP_ERR_WORKSPACE, "mtp_draft_steps: workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int H = L->hidden;
  for (int i = 0; i < k_steps; ++i) {
    mtp_step_in in = {};
    in.d_tokens = d_tokens + i;
    in.d_hidden = i == 0 ? d_hidden : d_hidden_out + (size_t)(i - 1) * H;
    in.cache_len = cache_len + i;
    in.m = 1;
    in.pos_base = pos_base;
    mtp_step_out out = {};
    out.d_token = d_tokens + i + 1;
    out.d_value = d_values + i;
    out.d_hidden_out = d_hidden_out + (size_t)i * H;
    if ((s = enqueue_layer(L, &in, &out, d_ws, st)) != MTP_OK) return s;
  }
  return MTP_OK;
}

mtp_status mtp_mimo_draft_round(const mtp_layer_desc* layers, int32_t n_layers,
                                mtp_mimo_layer_state* states, const float* d_hist,
                                int32_t hist_lo, int32_t hist_end, int32_t t, int32_t* d_ids,
                                int32_t ids_len, float* d_values, void* d_ws, size_t ws_bytes,
                                void* d_catch_ws, size_t catch_ws_bytes, void* stream,
                                int32_t* n_drafts) {
  if (!layers || !states || !d_hist || !d_ids || !d_values || !n_drafts || n_layers < 1 ||
      n_layers > MTP_SPEC_MAX_DEPTH)
    return fail(MTP_ERR_INVALID_ARG, "mtp_mimo_draft_round: bad arguments");
  *n_drafts = 0;
  if (!aligned16(d_hist)) return fail(MTP_ERR_INVALID_ARG, "mtp_mimo_draft_round: d_hist must be 16-byte aligned");
  // every check before any state changes or launches
  for (int l = 0; l < n_layers; ++l) {
    mtp_status s = check_layer(&layers[l], 1);
    if (s != MTP_OK) return s;
    if (!layers[l].embed) return fail(MTP_ERR_INVALID_ARG, "mtp_mimo_draft_round: layers need an embedding table");
    if (layers[l].hidden != layers[0].hidden)
      return fail(MTP_ERR_INVALID_ARG, "mtp_mimo_draft_round: layers must share the hidden size");
    if (!d_ws || ws_bytes < mtp_draft_workspace_bytes(&layers[l], 1))
      return fail(MTP_ERR_WORKSPACE, "mtp_mimo_draft_round: workspace too small");
    mtp_mimo_layer_state probe = states[l];
    int32_t start = 0;
    const int32_t n = mtp_mimo_plan_layer(&probe, l, t, hist_lo, hist_end, ids_len, &start);
    if (n <= 0) return MTP_OK;  // no draft this round (the history lacks t)
    if (t + 1 - probe.base > layers[l].cache_cap)
      return fail(MTP_ERR_CAPACITY, "mtp_mimo_draft_round: the rows exceed a layer's cache");
    if (n > 1 && (!d_catch_ws || catch_ws_bytes < mtp_kv_catch_up_workspace_bytes(&layers[l], n - 1)))
      return fail(MTP_ERR_WORKSPACE, "mtp_mimo_draft_round: catch-up workspace too small");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int H = layers[0].hidden;
  auto hist_row = [&](int pos) { return d_hist + (size_t)(pos - hist_lo) * H; };
  for (int l = 0; l < n_layers; ++l) {
    const mtp_layer_desc* L = &layers[l];
    mtp_mimo_layer_state& ls = states[l];
    int32_t start = 0;
    const int32_t n = mtp_mimo_plan_layer(&ls, l, t, hist_lo, hist_end, ids_len, &start);
    mtp_status s;
    if (n > 1) {  // positions start .. t - 1 add K/V rows only
      s = mtp_kv_catch_up(L, d_ids + start + l + 1, nullptr, n > 2 ? hist_row(start + 1) : nullptr,
                          hist_row(start), n - 1, start - ls.base, ls.base, d_catch_ws,
                          catch_ws_bytes, stream);
      if (s != MTP_OK) return s;
    }
    mtp_step_in in = {};  // position t: the layer's draft
    in.d_tokens = d_ids + t + l + 1;
    in.d_hidden = hist_row(t);
    in.cache_len = t - ls.base;
    in.m = 1;
    in.pos_base = ls.base;
    mtp_step_out out = {};
    out.d_token = d_ids + t + l + 2;
    out.d_value = d_values + l;
    if ((s = enqueue_layer(L, &in, &out, d_ws, st)) != MTP_OK) return s;
    if ((s = mtp_mimo_commit_layer(&ls, l, t, ids_len)) != MTP_OK) return s;
    *n_drafts = l + 1;
  }
  return MTP_OK;
}

}  // extern "C"

// ------------------------------------------------ attention without a workspace
namespace mtp {

// Scratch of attn_decode_sink_noalloc: the workspace header (device error
// word + completion counters) followed by the split partials.  2 MiB holds
// the partials of every geometry up to nkv * splits * (G*m) * (dv + 2)
// floats of about 520 K, e.g. 8 KV heads x 19 splits x 5 rows x 130 floats
// (395 KB) for a 40/8-head, 128-dim cache of 4096 rows.
constexpr size_t kNoallocScratchBytes = size_t(2) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];
constexpr int kNoallocMaxDevices = 64;

// Device address of the static scratch on the current device.  The first
// call on a device looks the address up and clears the header (a synchronous
// cudaMemset); later calls only read the cached address.
static mtp_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[kNoallocMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_sink_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kNoallocMaxDevices)
    return fail(MTP_ERR_UNSUPPORTED, "attn_decode_sink_noalloc: device ordinal above 63");
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_sink_noalloc: cudaGetSymbolAddress");
    e = cudaMemset(p, 0, sizeof(WsHeader));
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_sink_noalloc: clearing the scratch header");
    addr[dev] = p;
  }
  *out = addr[dev];
  return MTP_OK;
}

}  // namespace mtp

extern "C" {

// Same operation as attn_decode_sink, with the library's static scratch in
// place of a caller workspace, for callers that hold no device memory to
// lend: a host runtime whose device memory all sits in its own pools, or a
// plugin interface whose signature has no workspace argument.  It allocates
// no device memory.  The completion counters are cleared on `stream` before
// every launch; concurrent or overlapping calls on one device share the
// scratch and race, so they must be ordered (one stream, or events).
mtp_status attn_decode_sink_noalloc(const mtp_attn_geom* g, const float* d_qp, const float* d_kp,
                                    const float* d_vp, const float* d_q_norm,
                                    const float* d_k_norm, const float* d_rope,
                                    const float* d_sinks, float* d_k_cache, float* d_v_cache,
                                    int32_t cache_len, int32_t cache_cap, int32_t m,
                                    float* d_out, void* stream) {
  // every argument is checked before the scratch is set up or cleared, so an
  // invalid call does no device work
  mtp_status s = check_attn_args(g, d_qp, d_kp, d_vp, d_rope, d_k_cache, d_v_cache, cache_len,
                                 cache_cap, m, d_out, "attn_decode_sink_noalloc");
  if (s != MTP_OK) return s;
  const size_t need = attn_decode_sink_workspace_bytes(g, m, cache_len);
  if (need > kNoallocScratchBytes)
    return fail(MTP_ERR_WORKSPACE,
                "attn_decode_sink_noalloc: this geometry needs " + std::to_string(need) +
                    " bytes of scratch, the static scratch holds " +
                    std::to_string(kNoallocScratchBytes) + " (use attn_decode_sink)");
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != MTP_OK) return s;
  cudaError_t e = cudaMemsetAsync(header(scratch)->counters + kCntAttn, 0, sizeof(unsigned) * 128,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_sink_noalloc: clearing the counters");
  return attn_decode_sink(g, d_qp, d_kp, d_vp, d_q_norm, d_k_norm, d_rope, d_sinks, d_k_cache,
                          d_v_cache, cache_len, cache_cap, m, d_out, scratch,
                          kNoallocScratchBytes, stream);
}

}  // extern "C"
