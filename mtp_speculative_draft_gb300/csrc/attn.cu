// Decode attention of the draft layer over its own KV cache, fused with the
// per-head q/k RMSNorm, rotary embedding, KV append, sink logit and the
// sigmoid output gate.
//
// "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", forward_full_attention
// (apply_q_or_k_per_head_rms_norm, apply_imrope, apply_sdpa_with_kv_cache,
// apply_sigmoid_gate_multiply) and "cortiq-engine 0.8.49 src/mimo_mtp.rs"
// (sliding window, per-head sinks).
//
// Split-K over the cache, one CTA per (split, KV head), about one CTA per
// SM.  Each CTA serves all query heads of its KV head (grouped-query sharing
// of the K/V stream) for all m new rows.  The cached keys and values stream
// through a ring of shared-memory stages filled by bulk copies (one copy per
// key row into a padded row, one copy per value tile) and completed on
// mbarriers; the softmax is kept online in the log2 domain.  The m new keys
// and values are normalised/rotated in shared memory, appended to the cache
// with plain stores, and attended to by the last split from shared memory.
// The last CTA of a KV head to finish (completion counter, no spinning)
// merges the partials with precomputed split weights, adds the sink to the
// denominator, applies the gate and writes the output both as fp32 and
// packed for the o_proj GEMV.
#include "host.h"

namespace mtp {

constexpr int kAttnThreads = 512;
constexpr int kTileKeys = 32;
constexpr int kMaxQ = 16;            // query rows per KV head (heads per group x m)
constexpr float kNegBig = -1e30f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kAttnSmemMax = 200 * 1024;
constexpr int kQpt = 8;              // largest per-thread query count of the P.V split
// probability/statistics rows allocated for the padded query slices of P.V
// (up to kQpt rows per slice, at most kAttnThreads / 32 slices)
constexpr int kPadQ = kQpt * (kAttnThreads / 32);

struct AttnLayout {
  int stages;
  int kstride;       // padded K row (floats)
  size_t stage_bytes, q_off, p_off, red_off, stat_off, newk_off, newv_off, bar_off, total;
};

// Slices of the head dimension for the logits: a power of two <= 16 that
// divides dqk/4, with at most 4 float4 per slice.
__host__ __device__ inline int attn_nparts(int dqk) {
  int n = 16;
  while (n > 1 && ((dqk / 4) % n) != 0) n >>= 1;
  return n;
}

// Partials: (M, l) pairs [nkv][nsplit][QG][2], then outputs [nkv][nsplit][QG][dv]
// starting on a 16-byte boundary.
__host__ __device__ inline size_t attn_part_o_offset(int nkv, int nsplit, int QG) {
  return ((size_t)nkv * nsplit * QG * 2 + 3) / 4 * 4;
}

__host__ __device__ inline AttnLayout attn_layout(int dqk, int dv, int QG, int m) {
  AttnLayout L;
  L.kstride = dqk;  // K tiles are 128-byte-swizzled 32 x 32-float boxes (see attend_tile)
  L.stage_bytes = (size_t)kTileKeys * dqk * 4 + (size_t)kTileKeys * dv * 4;  // multiple of 4 KB
  const size_t red_bytes = (size_t)QG * attn_nparts(dqk) * kTileKeys * 4;
  const size_t fixed = (size_t)QG * dqk * 4 + (size_t)kPadQ * kTileKeys * 4 + red_bytes + 3 * kPadQ * 4 +
                       (size_t)m * (dqk + dv) * 4 + 8 * 8 + 256;
  int s = (int)((kAttnSmemMax - fixed) / L.stage_bytes);
  L.stages = s > 3 ? 3 : (s < 1 ? 1 : s);
  L.q_off = L.stages * L.stage_bytes;
  L.p_off = L.q_off + (size_t)QG * dqk * 4;
  L.red_off = L.p_off + (size_t)kPadQ * kTileKeys * 4;
  L.stat_off = L.red_off + red_bytes;
  L.newk_off = L.stat_off + 3 * kPadQ * 4;
  L.newv_off = L.newk_off + (size_t)m * dqk * 4;
  L.bar_off = (L.newv_off + (size_t)m * dv * 4 + 15) / 16 * 16;
  L.total = L.bar_off + 8 * 8 + 1024;  // + alignment slack of the swizzled stages
  return L;
}

// Per-head RMSNorm (optional) then rotary embedding of one head vector held
// in shared memory by one warp; the result is multiplied by `post_scale`.
__device__ __forceinline__ void warp_norm_rope(float* v, int d, const float* nw, float eps,
                                               const float* rope_row, int rot, float post_scale,
                                               int lane) {
  if (nw) {
    float ss = 0.f;
    for (int i = lane; i < d; i += 32) ss += v[i] * v[i];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)d + eps);
    __syncwarp();
    for (int i = lane; i < d; i += 32) v[i] = v[i] * inv * nw[i];
  }
  __syncwarp();
  const int half = rot / 2;
  for (int i = lane; i < half; i += 32) {
    const float c = rope_row[2 * i], s = rope_row[2 * i + 1];
    const float a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = a * s + b * c;
  }
  __syncwarp();
  if (post_scale != 1.f)
    for (int i = lane; i < d; i += 32) v[i] *= post_scale;
  __syncwarp();
}

// Work split of the P.V product: thread t owns output dim t % dv for the
// query rows q = t / dv + k * (kAttnThreads / dv), k < QPT (a template
// bound chosen on the host as the smallest power of two that covers QG).

// One tile of keys [key0, key0 + nk) from shared memory: logits, online
// softmax update and P.V accumulation.  Ends with the CTA synchronised.
template <int QPT>
__device__ __forceinline__ void attend_tile(const AttnParams& a, const float* Ks, bool kswz, int kstride,
                                           const float* Vs, int nk, int key0, const float* qs,
                                           float* ps, float* red, float* Ms, float* ls,
                                           float* als, float (&oacc)[QPT], int QG, int G) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int dqk = a.dqk, dv = a.dv;
  const int kq4 = dqk / 4;
  // logits: lane = key, warp = slice of the head dimension.  Each key
  // element is read from shared memory once (into registers); the query
  // slice is a warp-wide broadcast.  Slice partials meet in `red`.
  const int nparts = attn_nparts(dqk);
  const int pc4 = kq4 / nparts;  // float4 per slice
  if (warp < nparts) {
    const float4* kv = reinterpret_cast<const float4*>(Ks + lane * kstride) + warp * pc4;
    // rows past nk are not read (the new-key tile holds only m rows)
    float4 kr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < pc4 && lane < nk) {
        if (kswz) {
          // box f/8 of 32 rows x 128 bytes; 16-byte chunk c of row r at c ^ (r & 7)
          const int f = warp * pc4 + i;
          kr[i] = *reinterpret_cast<const float4*>(Ks + (f >> 3) * 1024 + lane * 32 +
                                                   (((f & 7) ^ (lane & 7)) << 2));
        } else {
          kr[i] = kv[i];
        }
      }
    }
    for (int qi = 0; qi < QG; ++qi) {
      const float4* qv = reinterpret_cast<const float4*>(qs + qi * dqk) + warp * pc4;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < pc4) {
          const float4 x = qv[i];
          acc = fmaf(x.x, kr[i].x, fmaf(x.y, kr[i].y, fmaf(x.z, kr[i].z, fmaf(x.w, kr[i].w, acc))));
        }
      }
      red[(qi * nparts + warp) * kTileKeys + lane] = acc;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < QG * kTileKeys; idx += kAttnThreads) {
    const int jj = idx & (kTileKeys - 1), qi = idx / kTileKeys;
    const int j = key0 + jj, p = a.L + qi / G;
    float l = kNegBig;
    if (jj < nk && j <= p && (a.window <= 0 || j > p - a.window)) {
      l = 0.f;
      for (int pt = 0; pt < nparts; ++pt) l += red[(qi * nparts + pt) * kTileKeys + jj];
    }
    ps[qi * kTileKeys + jj] = l;
  }
  __syncthreads();
  for (int qi = warp; qi < QG; qi += kAttnThreads / 32) {
    const float l = ps[qi * kTileKeys + lane];
    const float mold = Ms[qi];
    const float mnew = fmaxf(mold, warp_max(l));
    const float pr = l <= 0.5f * kNegBig ? 0.f : exp2f(l - mnew);
    const float s = warp_sum(pr);
    ps[qi * kTileKeys + lane] = pr;
    if (lane == 0) {
      const float alpha = exp2f(mold - mnew);
      als[qi] = alpha;
      ls[qi] = ls[qi] * alpha + s;
      Ms[qi] = mnew;
    }
  }
  __syncthreads();
  const int nsl = kAttnThreads / dv;  // query slices
  const int d = tid % dv, q0 = tid / dv;
  if (q0 < nsl) {
    // rows past QG read zero probabilities and rescale factors (padded)
#pragma unroll
    for (int k = 0; k < QPT; ++k) oacc[k] *= als[q0 + k * nsl];
    // keys four at a time: independent loads ahead of their FMAs
    int jj = 0;
    for (; jj + 4 <= nk; jj += 4) {
      const float v0 = Vs[jj * dv + d], v1 = Vs[(jj + 1) * dv + d];
      const float v2 = Vs[(jj + 2) * dv + d], v3 = Vs[(jj + 3) * dv + d];
#pragma unroll
      for (int k = 0; k < QPT; ++k) {
        const float4 pr = *reinterpret_cast<const float4*>(ps + (q0 + k * nsl) * kTileKeys + jj);
        oacc[k] = fmaf(pr.x, v0, fmaf(pr.y, v1, fmaf(pr.z, v2, fmaf(pr.w, v3, oacc[k]))));
      }
    }
    for (; jj < nk; ++jj) {
      const float v = Vs[jj * dv + d];
#pragma unroll
      for (int k = 0; k < QPT; ++k)
        oacc[k] = fmaf(ps[(q0 + k * nsl) * kTileKeys + jj], v, oacc[k]);
    }
  }
  __syncthreads();
}

template <int QPT>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const __grid_constant__ AttnParams a) {
  extern __shared__ __align__(1024) uint8_t smraw_unaligned[];
  // the swizzled K boxes need 1024-byte-aligned stages
  uint8_t* smraw = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smraw_unaligned) + 1023) & ~uintptr_t(1023));
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.nh / a.nkv;
  const int QG = G * a.m;
  const int dqk = a.dqk, dv = a.dv;
  const int q_rows = a.nh * dqk * (a.gated ? 2 : 1);
  const AttnLayout Ly = attn_layout(dqk, dv, QG, a.m);
  const int S = Ly.stages;
  float* qs = reinterpret_cast<float*>(smraw + Ly.q_off);
  float* ps = reinterpret_cast<float*>(smraw + Ly.p_off);
  float* red = reinterpret_cast<float*>(smraw + Ly.red_off);
  float* Ms = reinterpret_cast<float*>(smraw + Ly.stat_off);
  float* ls = Ms + kPadQ;
  float* als = ls + kPadQ;
  float* newk = reinterpret_cast<float*>(smraw + Ly.newk_off);
  float* newv = reinterpret_cast<float*>(smraw + Ly.newv_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smraw + Ly.bar_off);
  __shared__ bool last;

  // cached keys [kbeg, L) in whole tiles per split; new keys go to the last split
  const int L = a.L;
  const int kbeg = a.window > 0 ? max(0, L + 1 - a.window) : 0;
  const int ntiles = (L - kbeg + kTileKeys - 1) / kTileKeys;
  const int tps = (ntiles + a.nsplit - 1) / a.nsplit;
  const int t_begin = min(ntiles, split * tps);
  const int t_end = min(ntiles, t_begin + tps);
  const int my_tiles = t_end - t_begin;
  const float* vbase = a.vc + (size_t)kvh * a.cap * dv;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  const uint64_t pol = l2_policy_evict_first();
  // Warp 0 fills stage `slot` with tile `t` (relative to t_begin).
  auto issue = [&](int t, int slot) {
    const int key0 = kbeg + (t_begin + t) * kTileKeys;
    const int nk = min(kTileKeys, L - key0);
    uint8_t* st = smraw + (size_t)slot * Ly.stage_bytes;
    float* Ks = reinterpret_cast<float*>(st);
    float* Vs = Ks + kTileKeys * Ly.kstride;
    // K: dqk/32 tensor-map boxes of 32 rows (full boxes are counted even past
    // the cache end, where the copy fills zeros); V: one bulk copy of nk rows
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[slot], (uint32_t)kTileKeys * dqk * 4 + (uint32_t)nk * dv * 4);
      for (int b = 0; b < dqk / 32; ++b)
        tma_load_2d(Ks + b * 1024, &a.kmap, &bars[slot], b * 32, kvh * a.cap + key0, pol);
      bulk_load(Vs, vbase + (size_t)key0 * dv, (uint32_t)nk * dv * 4, &bars[slot], pol);
    }
  };
  if (a.prefetch_before_wait && warp == 0)
    for (int t = 0; t < S && t < my_tiles; ++t) issue(t, t);
  pdl_wait();
  pdl_launch_dependents();
  if (!a.prefetch_before_wait && warp == 0)
    for (int t = 0; t < S && t < my_tiles; ++t) issue(t, t);

  // ---- queries of this KV head: norm, rotate, pre-scale (log2 domain)
  const float qscale = a.scale * kLog2e;
  for (int qi = warp; qi < QG; qi += kAttnThreads / 32) {
    const int r = qi / G, h = kvh * G + qi % G;
    const float* src = a.qp + (size_t)r * q_rows + (size_t)h * dqk * (a.gated ? 2 : 1);
    float* dst = qs + qi * dqk;
    for (int i = lane; i < dqk; i += 32) dst[i] = src[i];
    warp_norm_rope(dst, dqk, a.qn, a.eps, a.rope + (size_t)(L + r) * a.rot, a.rot, qscale, lane);
  }
  // ---- new keys/values (last split): normalise, rotate, append to the cache
  const bool has_new = split == a.nsplit - 1;
  if (has_new) {
    for (int r = warp; r < a.m; r += kAttnThreads / 32) {
      const int pos = L + r;
      float* kn = newk + r * dqk;
      const float* ksrc = a.kp + (size_t)r * a.nkv * dqk + (size_t)kvh * dqk;
      for (int i = lane; i < dqk; i += 32) kn[i] = ksrc[i];
      warp_norm_rope(kn, dqk, a.kn, a.eps, a.rope + (size_t)pos * a.rot, a.rot, 1.f, lane);
      float* kdst = a.kc + ((size_t)kvh * a.cap + pos) * dqk;
      for (int i = lane; i < dqk; i += 32) kdst[i] = kn[i];
      float* vn = newv + r * dv;
      const float* vsrc = a.vp + (size_t)r * a.nkv * dv + (size_t)kvh * dv;
      float* vdst = a.vc + ((size_t)kvh * a.cap + pos) * dv;
      for (int i = lane; i < dv; i += 32) {
        const float v = vsrc[i];
        vn[i] = v;
        vdst[i] = v;
      }
    }
  }
  for (int i = tid; i < kPadQ; i += kAttnThreads) {
    Ms[i] = kNegBig;
    ls[i] = 0.f;
    als[i] = 0.f;
  }
  for (int i = tid; i < kPadQ * kTileKeys; i += kAttnThreads) ps[i] = 0.f;
  __syncthreads();

  float oacc[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) oacc[k] = 0.f;

  for (int t = 0; t < my_tiles; ++t) {
    const int slot = t % S;
    const bool ok = mbar_wait_bounded(&bars[slot], (uint32_t)((t / S) & 1));
    if (__syncthreads_or(!ok)) {  // the whole CTA gives up together
      if (tid == 0) set_dev_error(a.err, kErrMbarTimeout);
      return;
    }
    const float* Ks = reinterpret_cast<const float*>(smraw + (size_t)slot * Ly.stage_bytes);
    const float* Vs = Ks + kTileKeys * Ly.kstride;
    const int key0 = kbeg + (t_begin + t) * kTileKeys;
    attend_tile<QPT>(a, Ks, true, Ly.kstride, Vs, min(kTileKeys, L - key0), key0, qs, ps, red,
                     Ms, ls, als, oacc, QG, G);
    if (warp == 0 && t + S < my_tiles) issue(t + S, slot);
  }
  if (has_new)
    attend_tile<QPT>(a, newk, false, dqk, newv, a.m, L, qs, ps, red, Ms, ls, als, oacc, QG, G);

  // ---- partial of this split: (M, l) pairs and unnormalised outputs
  const size_t pidx = (size_t)(kvh * a.nsplit + split) * QG;
  float* part_o = a.part + attn_part_o_offset(a.nkv, a.nsplit, QG);
  {
    const int nsl = kAttnThreads / dv;
    const int d = tid % dv, q0 = tid / dv;
    if (q0 < nsl) {
#pragma unroll
      for (int k = 0; k < QPT; ++k) {
        const int q = q0 + k * nsl;
        if (q < QG) part_o[(pidx + q) * dv + d] = oacc[k];
      }
    }
  }
  if (tid < QG) {
    a.part[(pidx + tid) * 2 + 0] = Ms[tid];
    a.part[(pidx + tid) * 2 + 1] = ls[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.counters[kvh], 1u);
    last = (prev == (unsigned)a.nsplit - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  // ---- merge (last CTA of this KV head); the stage ring is free now
  const int ns = a.nsplit;
  float* wsm = reinterpret_cast<float*>(smraw);        // [ns][QG] split weights
  float* lsm = wsm + ns * QG;                          // [ns][QG] split denominators
  float* fin = lsm + ns * QG;                          // [QG][dv]
  const size_t base = (size_t)kvh * ns * QG;
  // all (M, l) pairs in one parallel pass, so no loop below waits on memory
  for (int i = tid; i < ns * QG; i += kAttnThreads) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part) + base + i);
    wsm[i] = ml.x;
    lsm[i] = ml.y;
  }
  __syncthreads();
  if (tid < QG) {
    const int h = kvh * G + tid % G;
    const float sinkl2 = a.sinks ? a.sinks[h] * kLog2e : kNegBig;
    float M = sinkl2;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, wsm[s * QG + tid]);
    float den = a.sinks ? exp2f(sinkl2 - M) : 0.f;
    for (int s = 0; s < ns; ++s) den += exp2f(wsm[s * QG + tid] - M) * lsm[s * QG + tid];
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int s = 0; s < ns; ++s) wsm[s * QG + tid] = exp2f(wsm[s * QG + tid] - M) * inv;
  }
  __syncthreads();
  const int dv4 = dv / 4;
  for (int it = tid; it < QG * dv4; it += kAttnThreads) {
    const int qi = it / dv4, d4 = it - qi * dv4;
    const float4* po = reinterpret_cast<const float4*>(part_o + (base + qi) * dv) + d4;
    const size_t sstride = (size_t)QG * dv4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 4 <= ns; s += 4) {
      const float4 v0 = __ldcg(po + (size_t)s * sstride);
      const float4 v1 = __ldcg(po + (size_t)(s + 1) * sstride);
      const float4 v2 = __ldcg(po + (size_t)(s + 2) * sstride);
      const float4 v3 = __ldcg(po + (size_t)(s + 3) * sstride);
      const float w0 = wsm[s * QG + qi], w1 = wsm[(s + 1) * QG + qi];
      const float w2 = wsm[(s + 2) * QG + qi], w3 = wsm[(s + 3) * QG + qi];
      acc.x += w0 * v0.x + w1 * v1.x + w2 * v2.x + w3 * v3.x;
      acc.y += w0 * v0.y + w1 * v1.y + w2 * v2.y + w3 * v3.y;
      acc.z += w0 * v0.z + w1 * v1.z + w2 * v2.z + w3 * v3.z;
      acc.w += w0 * v0.w + w1 * v1.w + w2 * v2.w + w3 * v3.w;
    }
    for (; s < ns; ++s) {
      const float4 v = __ldcg(po + (size_t)s * sstride);
      const float w = wsm[s * QG + qi];
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    float o[4] = {acc.x, acc.y, acc.z, acc.w};
    if (a.gated) {
      const int r = qi / G, h = kvh * G + qi % G;
      const float* g = a.qp + (size_t)r * q_rows + (size_t)h * dqk * 2 + dqk + d4 * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = o[e] / (1.f + __expf(-g[e]));
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) fin[qi * dv + d4 * 4 + e] = o[e];
  }
  __syncthreads();
  // fp32 output and packed copy: octets of (row, head, dims)
  const int oct_per_q = dv / 8;
  const int total_oct = QG * oct_per_q;
  for (int o0 = 0; o0 < total_oct; o0 += kAttnThreads) {
    const int oi = o0 + tid;
    float2 sum = make_float2(0.f, 0.f);
    int r = 0, k = 0;
    if (oi < total_oct) {
      const int qi = oi / oct_per_q, oc = oi - qi * oct_per_q;
      r = qi / G;
      const int h = kvh * G + qi % G;
      k = h * dv + oc * 8;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = fin[qi * dv + oc * 8 + i];
      if (a.out) {
#pragma unroll
        for (int i = 0; i < 8; ++i) a.out[(size_t)r * a.nh * dv + k + i] = v[i];
      }
      if (a.out_xp) {
        uint4 hi, lo;
        sum = pack8(v, hi, lo);
        const int g = k / kGroup, t = (k % kGroup) / 8;
        a.out_xp[xp_index(g, r, t, 0, a.m)] = hi;
        a.out_xp[xp_index(g, r, t, 1, a.m)] = lo;
      }
    }
    if (a.out_xp) {
      // the four octets of a group are adjacent (dv % 32 == 0, kAttnThreads % 4 == 0)
      sum.x += __shfl_xor_sync(0xffffffffu, sum.x, 1);
      sum.y += __shfl_xor_sync(0xffffffffu, sum.y, 1);
      sum.x += __shfl_xor_sync(0xffffffffu, sum.x, 2);
      sum.y += __shfl_xor_sync(0xffffffffu, sum.y, 2);
      if (oi < total_oct && (oi & 3) == 0) a.out_xs[(k / kGroup) * a.m + r] = sum;
    }
  }
  if (tid == 0) a.counters[kvh] = 0u;
}

int attn_splits(int nkv, int keys) {
  const int target = sm_count();  // about one CTA per SM
  int ns = (target + nkv - 1) / nkv;
  const int max_by_tiles = (keys + kTileKeys - 1) / kTileKeys;  // at least one tile per split
  if (ns > max_by_tiles) ns = max_by_tiles;
  if (ns < 1) ns = 1;
  return ns;
}

size_t attn_part_bytes(int nkv, int nsplit, int q_per_kv, int dv) {
  return (attn_part_o_offset(nkv, nsplit, q_per_kv) + (size_t)nkv * nsplit * q_per_kv * dv) *
         sizeof(float);
}

template <int QPT>
static cudaError_t launch_attn_t(const AttnParams& a, size_t smem, cudaStream_t st) {
  static_assert(sizeof(AttnParams) <= 4096, "kernel parameters fit the classic limit");
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<QPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kAttnSmemMax + 1024);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.nkv);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<QPT>, a);
}

cudaError_t launch_attn(const AttnParams& a_in, cudaStream_t st) {
  AttnParams a = a_in;
  cudaError_t ke = encode_f32_tile_map(&a.kmap, a.kc, (uint64_t)a.nkv * a.cap, (uint64_t)a.dqk);
  if (ke != cudaSuccess) return ke;
  const int QG = (a.nh / a.nkv) * a.m;
  const AttnLayout Ly = attn_layout(a.dqk, a.dv, QG, a.m);
  // the merge reuses the stage ring: split weights and the finished rows
  const size_t merge = (size_t)a.nsplit * QG * 8 + (size_t)QG * a.dv * 4;
  const size_t smem = Ly.total > merge ? Ly.total : merge;
  if (smem > (size_t)kAttnSmemMax + 1024) return cudaErrorInvalidValue;
  const int nsl = kAttnThreads / a.dv;
  const int need = (QG + nsl - 1) / nsl;
  if (need <= 1) return launch_attn_t<1>(a, smem, st);
  if (need <= 2) return launch_attn_t<2>(a, smem, st);
  if (need <= 4) return launch_attn_t<4>(a, smem, st);
  return launch_attn_t<8>(a, smem, st);
}

}  // namespace mtp
