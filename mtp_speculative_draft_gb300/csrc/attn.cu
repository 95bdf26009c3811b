// Decode attention of the draft layer over its own KV cache, fused with the
// per-head q/k RMSNorm, rotary embedding, KV append, sink logit and the
// sigmoid output gate.
//
// "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", forward_full_attention
// (apply_q_or_k_per_head_rms_norm, apply_imrope, apply_sdpa_with_kv_cache,
// apply_sigmoid_gate_multiply) and "cortiq-engine 0.8.49 src/mimo_mtp.rs"
// (sliding window, per-head sinks).
//
// Split-K over the cache (one CTA per (split, KV head)): each CTA serves all
// query heads of its KV head (grouped-query sharing of the K/V stream) for all
// m new rows, keeps an online softmax in the log2 domain, and writes an
// unnormalised partial.  The last CTA of a KV head (completion counter, no
// spinning) merges the partials, adds the sink to the denominator, applies
// the gate and writes the output both as fp32 and packed for the o_proj GEMV.
#include "host.h"

namespace mtp {

constexpr int kAttnThreads = 128;
constexpr int kTileKeys = 32;
constexpr int kMaxQ = 16;            // query rows per KV head (heads per group x m)
constexpr float kNegBig = -1e30f;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnSmem {
  static size_t bytes(int dqk, int dv, int QG) {
    return (size_t)kTileKeys * (dqk + 4) * 4 + (size_t)kTileKeys * dv * 4 +
           (size_t)QG * dqk * 4 + (size_t)QG * kTileKeys * 4 + 4 * kMaxQ * 4 + 64;
  }
};

// Per-head RMSNorm (optional) then rotary embedding of one head vector held
// in shared memory by one warp.
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

__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnParams a) {
  extern __shared__ __align__(16) float sm[];
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.nh / a.nkv;
  const int QG = G * a.m;
  const int dqk = a.dqk, dv = a.dv;
  const int q_rows = a.nh * dqk * (a.gated ? 2 : 1);

  float* Ks = sm;                                   // [TK][dqk+4]
  float* Vs = Ks + kTileKeys * (dqk + 4);           // [TK][dv]
  float* qs = Vs + kTileKeys * dv;                  // [QG][dqk]
  float* ps = qs + QG * dqk;                        // [QG][TK]
  float* Ms = ps + QG * kTileKeys;                  // [kMaxQ]
  float* ls = Ms + kMaxQ;
  float* als = ls + kMaxQ;
  __shared__ bool last;

  const int L = a.L;
  const int kbeg = a.window > 0 ? max(0, L - a.window + 1) : 0;
  const int kend = L + a.m;
  const int chunk = (kend - kbeg + a.nsplit - 1) / a.nsplit;
  const int c0 = min(kend, kbeg + split * chunk);
  const int c1 = min(kend, c0 + chunk);

  pdl_wait();
  pdl_launch_dependents();

  // ---- queries of this KV head: norm, rotate, pre-scale (log2 domain)
  const float qscale = a.scale * kLog2e;
  for (int qi = warp; qi < QG; qi += kAttnThreads / 32) {
    const int r = qi / G, h = kvh * G + qi % G;
    const float* src = a.qp + (size_t)r * q_rows + (size_t)h * dqk * (a.gated ? 2 : 1);
    float* dst = qs + qi * dqk;
    for (int i = lane; i < dqk; i += 32) dst[i] = src[i];
    warp_norm_rope(dst, dqk, a.qn, a.eps, a.rope + (size_t)(L + r) * a.rot, a.rot, qscale, lane);
  }
  // ---- new keys/values whose positions fall in this CTA's chunk: append
  for (int r = warp; r < a.m; r += kAttnThreads / 32) {
    const int pos = L + r;
    if (pos < c0 || pos >= c1) continue;
    float* kdst = a.kc + ((size_t)kvh * a.cap + pos) * dqk;
    const float* ksrc = a.kp + (size_t)r * a.nkv * dqk + (size_t)kvh * dqk;
    // normalise + rotate in the K tile area of shared memory, then store
    float* tmp = Ks + warp * (dqk + 4);
    for (int i = lane; i < dqk; i += 32) tmp[i] = ksrc[i];
    warp_norm_rope(tmp, dqk, a.kn, a.eps, a.rope + (size_t)pos * a.rot, a.rot, 1.f, lane);
    for (int i = lane; i < dqk; i += 32) kdst[i] = tmp[i];
    float* vdst = a.vc + ((size_t)kvh * a.cap + pos) * dv;
    const float* vsrc = a.vp + (size_t)r * a.nkv * dv + (size_t)kvh * dv;
    for (int i = lane; i < dv; i += 32) vdst[i] = vsrc[i];
  }
  if (tid < kMaxQ) {
    Ms[tid] = kNegBig;
    ls[tid] = 0.f;
  }
  __syncthreads();

  float oacc[kMaxQ][2];
#pragma unroll
  for (int q = 0; q < kMaxQ; ++q) oacc[q][0] = oacc[q][1] = 0.f;

  const float* kbase = a.kc + (size_t)kvh * a.cap * dqk;
  const float* vbase = a.vc + (size_t)kvh * a.cap * dv;
  for (int t0 = c0; t0 < c1; t0 += kTileKeys) {
    const int nk = min(kTileKeys, c1 - t0);
    // load K and V tiles
    const int kq4 = dqk / 4, vq4 = dv / 4;
    for (int i = tid; i < kTileKeys * kq4; i += kAttnThreads) {
      const int jj = i / kq4, d4 = i - jj * kq4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (jj < nk) v = *reinterpret_cast<const float4*>(kbase + (size_t)(t0 + jj) * dqk + d4 * 4);
      *reinterpret_cast<float4*>(Ks + jj * (dqk + 4) + d4 * 4) = v;
    }
    for (int i = tid; i < kTileKeys * vq4; i += kAttnThreads) {
      const int jj = i / vq4, d4 = i - jj * vq4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (jj < nk) v = *reinterpret_cast<const float4*>(vbase + (size_t)(t0 + jj) * dv + d4 * 4);
      *reinterpret_cast<float4*>(Vs + jj * dv + d4 * 4) = v;
    }
    __syncthreads();
    // logits
    for (int pi = tid; pi < QG * kTileKeys; pi += kAttnThreads) {
      const int jj = pi & (kTileKeys - 1), qi = pi / kTileKeys;
      const int j = t0 + jj, r = qi / G, p = L + r;
      float l = kNegBig;
      const bool ok = jj < nk && j <= p && (a.window <= 0 || j > p - a.window);
      if (ok) {
        const float4* qv = reinterpret_cast<const float4*>(qs + qi * dqk);
        const float4* kv = reinterpret_cast<const float4*>(Ks + jj * (dqk + 4));
        float acc = 0.f;
        for (int d4 = 0; d4 < kq4; ++d4) {
          const float4 x = qv[d4], y = kv[d4];
          acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
        }
        l = acc;
      }
      ps[qi * kTileKeys + jj] = l;
    }
    __syncthreads();
    // online softmax update, one warp per query row
    for (int qi = warp; qi < QG; qi += kAttnThreads / 32) {
      const float l = ps[qi * kTileKeys + lane];
      const float tmax = warp_max(l);
      const float mold = Ms[qi];
      const float mnew = fmaxf(mold, tmax);
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
    // o = alpha * o + P V
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q) {
      if (q < QG) {
        const float al = als[q];
        oacc[q][0] *= al;
        oacc[q][1] *= al;
      }
    }
    for (int jj = 0; jj < nk; ++jj) {
      const float v0 = tid < dv ? Vs[jj * dv + tid] : 0.f;
      const float v1 = tid + kAttnThreads < dv ? Vs[jj * dv + tid + kAttnThreads] : 0.f;
#pragma unroll
      for (int q = 0; q < kMaxQ; ++q) {
        if (q < QG) {
          const float pr = ps[q * kTileKeys + jj];
          oacc[q][0] = fmaf(pr, v0, oacc[q][0]);
          oacc[q][1] = fmaf(pr, v1, oacc[q][1]);
        }
      }
    }
    __syncthreads();
  }

  // ---- partial of this split
  const int pstride = dv + 2;
  float* mypart = a.part + ((size_t)(kvh * a.nsplit + split) * QG) * pstride;
#pragma unroll
  for (int q = 0; q < kMaxQ; ++q) {
    if (q < QG) {
      if (tid < dv) mypart[q * pstride + 2 + tid] = oacc[q][0];
      if (tid + kAttnThreads < dv) mypart[q * pstride + 2 + tid + kAttnThreads] = oacc[q][1];
    }
  }
  if (tid < QG) {
    mypart[tid * pstride + 0] = Ms[tid];
    mypart[tid * pstride + 1] = ls[tid];
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

  // ---- merge (last CTA of this KV head)
  float* fin = Ks;  // [QG][dv]
  const float* kvpart = a.part + (size_t)kvh * a.nsplit * QG * pstride;
  for (int qi = warp; qi < QG; qi += kAttnThreads / 32) {
    const int h = kvh * G + qi % G;
    float M = kNegBig;
    for (int s = lane; s < a.nsplit; s += 32) M = fmaxf(M, __ldcg(kvpart + ((size_t)s * QG + qi) * pstride));
    M = warp_max(M);
    const float sinkl2 = a.sinks ? a.sinks[h] * kLog2e : kNegBig;
    M = fmaxf(M, sinkl2);
    float den = 0.f;
    for (int s = lane; s < a.nsplit; s += 32) {
      const float* pp = kvpart + ((size_t)s * QG + qi) * pstride;
      den += exp2f(__ldcg(pp) - M) * __ldcg(pp + 1);
    }
    den = warp_sum(den);
    if (a.sinks) den += exp2f(sinkl2 - M);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int d = lane; d < dv; d += 32) {
      float o = 0.f;
      for (int s = 0; s < a.nsplit; ++s) {
        const float* pp = kvpart + ((size_t)s * QG + qi) * pstride;
        o = fmaf(exp2f(__ldcg(pp) - M), __ldcg(pp + 2 + d), o);
      }
      o *= inv;
      if (a.gated) {
        const int r = qi / G;
        const float g = a.qp[(size_t)r * q_rows + (size_t)h * dqk * 2 + dqk + d];
        o = o / (1.f + __expf(-g));
      }
      fin[qi * dv + d] = o;
    }
  }
  __syncthreads();
  // fp32 output and packed copy: octets of (row, head, dims)
  const int oct_per_q = dv / 8;
  const int total_oct = QG * oct_per_q;
  for (int o0 = 0; o0 < total_oct; o0 += kAttnThreads) {
    const int oi = o0 + tid;
    float sum = 0.f;
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
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      if (oi < total_oct && (oi & 3) == 0) a.out_xs[(k / kGroup) * a.m + r] = sum;
    }
  }
  if (tid == 0) a.counters[kvh] = 0u;
}

int attn_splits(int nkv, int keys) {
  const int target = 2 * sm_count();  // about two CTAs per SM
  int ns = (target + nkv - 1) / nkv;
  const int max_by_keys = (keys + kTileKeys - 1) / kTileKeys;  // at least one tile per split
  if (ns > max_by_keys) ns = max_by_keys;
  if (ns < 1) ns = 1;
  return ns;
}

size_t attn_part_bytes(int nkv, int nsplit, int q_per_kv, int dv) {
  return (size_t)nkv * nsplit * q_per_kv * (dv + 2) * sizeof(float);
}

cudaError_t launch_attn(const AttnParams& a, cudaStream_t st) {
  const int QG = (a.nh / a.nkv) * a.m;
  const size_t smem = AttnSmem::bytes(a.dqk, a.dv, QG);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
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
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel, a);
}

}  // namespace mtp
