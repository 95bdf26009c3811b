// RMSNorm (+ residual, + embedding gather) with packing of the result into the
// tensor-core activation layout, and the rotary-table initialiser.
//
// RMSNorm: x / sqrt(mean(x^2) + eps) * w ("hf2q 0.1.13
// src/inference/models/qwen35/mtp.rs", rms_norm_with_weight and
// dispatch_fused_residual_norm_f32).
#include "host.h"

namespace mtp {

struct NormPackArgs {
  NormSeg seg[2];
  int nseg;
  int m;
  uint4* xp;
  float2* xs;
  int* err;
};

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

__device__ __forceinline__ const float* seg_row(const NormSeg& s, int c, int* err) {
  if (s.table) {
    int tok = s.tokens[c];
    if (tok < 0 || tok >= s.vocab) {
      set_dev_error(err, kErrBadToken);
      tok = 0;
    }
    return s.table + (size_t)tok * s.dim;
  }
  return s.src + (size_t)c * s.src_ld;
}

__global__ void __launch_bounds__(kNormThreads) norm_pack_kernel(const NormPackArgs a) {
  __shared__ float red[kNormThreads / 32];
#ifndef MTP_NORM_EARLY_TRIGGER
#define MTP_NORM_EARLY_TRIGGER 0
#endif
#if MTP_NORM_EARLY_TRIGGER
  // Lets the projection that follows launch (and start streaming weights)
  // right away; measured slower on the draft step, so off by default.
  pdl_launch_dependents();
  pdl_wait();
#else
  pdl_wait();
  pdl_launch_dependents();
#endif
  // grid = (slices, m): every CTA of row c computes the row's norms and
  // writes octets [slice * per, (slice + 1) * per) of the packed output
  const int c = blockIdx.y;
  float inv[2] = {1.f, 1.f};
  for (int si = 0; si < a.nseg; ++si) {
    const NormSeg& s = a.seg[si];
    if (!s.w) continue;
    const float* row = seg_row(s, c, a.err);
    const float* dl = s.delta ? s.delta + (size_t)c * s.src_ld : nullptr;
    float ss = 0.f;
#pragma unroll 4
    for (int k = threadIdx.x * 4; k < s.dim; k += kNormThreads * 4) {  // loads issued together
      float4 v = *reinterpret_cast<const float4*>(row + k);
      if (dl) {
        const float4 d = *reinterpret_cast<const float4*>(dl + k);
        v.x += d.x; v.y += d.y; v.z += d.z; v.w += d.w;
      }
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum(ss, red);
    inv[si] = rsqrtf(ss / (float)s.dim + s.eps);
  }
  // pass 2: octets of the concatenation
  const int K = a.seg[0].dim + (a.nseg > 1 ? a.seg[1].dim : 0);
  const int octets = K / 8;
  // slices hold whole groups (4 octets) so the group sums stay in one CTA
  const int per = (octets / 4 + gridDim.x - 1) / gridDim.x * 4;
  const int o_begin = blockIdx.x * per;
  const int o_end = min(octets, o_begin + per);
  for (int o0 = o_begin; o0 < o_end; o0 += kNormThreads) {
    const int o = o0 + threadIdx.x;
    const bool valid = o < o_end;
    const int k = o * 8;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) {
      const int si = (a.nseg > 1 && k >= a.seg[0].dim) ? 1 : 0;
      const NormSeg& s = a.seg[si];
      const int kk = k - (si ? a.seg[0].dim : 0);
      const float* row = seg_row(s, c, a.err);
      const float* dl = s.delta ? s.delta + (size_t)c * s.src_ld : nullptr;
      const float4 v0 = *reinterpret_cast<const float4*>(row + kk);
      const float4 v1 = *reinterpret_cast<const float4*>(row + kk + 4);
      v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
      v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
      if (dl) {
        const float4 d0 = *reinterpret_cast<const float4*>(dl + kk);
        const float4 d1 = *reinterpret_cast<const float4*>(dl + kk + 4);
        v[0] += d0.x; v[1] += d0.y; v[2] += d0.z; v[3] += d0.w;
        v[4] += d1.x; v[5] += d1.y; v[6] += d1.z; v[7] += d1.w;
      }
      if (s.out_sum) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s.out_sum[(size_t)c * s.dim + kk + i] = v[i];
      }
      if (s.w) {
        const float4 w0 = *reinterpret_cast<const float4*>(s.w + kk);
        const float4 w1 = *reinterpret_cast<const float4*>(s.w + kk + 4);
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = v[i] * inv[si] * wv[i];
      }
      if (s.out_norm) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s.out_norm[(size_t)c * s.dim + kk + i] = v[i];
      }
    }
    if (a.xp) {
      // octets o..o+3 of one group sit in adjacent lanes (kNormThreads % 4 == 0)
      uint4 hi, lo;
      const float2 gx = pack8_group(v, valid, hi, lo);
      if (valid) {
        const int g = k / kGroup, t = (k % kGroup) / 8;
        a.xp[xp_index(g, c, t, 0, a.m)] = hi;
        a.xp[xp_index(g, c, t, 1, a.m)] = lo;
        if ((o & 3) == 0) a.xs[(o / 4) * a.m + c] = gx;
      }
    }
  }
}

cudaError_t launch_norm_pack(const NormSeg* segs, int nseg, int m, uint4* xp, float2* xs,
                             int* err, cudaStream_t st) {
  NormPackArgs a = {};
  a.seg[0] = segs[0];
  if (nseg > 1) a.seg[1] = segs[1];
  a.nseg = nseg;
  a.m = m;
  a.xp = xp;
  a.xs = xs;
  a.err = err;
  // a few CTAs per row so one row's octets are packed in parallel
  const int K = segs[0].dim + (nseg > 1 ? segs[1].dim : 0);
  int slices = (K / 8 + kNormThreads - 1) / kNormThreads;
  if (slices > 8) slices = 8;
  if (m > 4) slices = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(slices, m);
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, norm_pack_kernel, a);
}

// --------------------------------------------------------------- rotary table
__global__ void rope_table_kernel(float* __restrict__ d, int max_pos, int rot, double theta) {
  const int half = rot / 2;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)max_pos * half) return;
  const int p = (int)(i / half);
  const int j = (int)(i % half);
  const double ang = (double)p * pow(theta, -2.0 * (double)j / (double)rot);
  double sn, cs;
  sincos(ang, &sn, &cs);
  d[2 * i] = (float)cs;
  d[2 * i + 1] = (float)sn;
}

cudaError_t launch_rope_table(float* d, int max_pos, int rot, double theta, cudaStream_t st) {
  const long long n = (long long)max_pos * (rot / 2);
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads);
  rope_table_kernel<<<blocks, threads, 0, st>>>(d, max_pos, rot, theta);
  return cudaGetLastError();
}

}  // namespace mtp
