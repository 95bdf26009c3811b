// MoE router of the draft layer: RMSNorm of the residual row, float32 router
// projection, softmax, top-k (lowest index among equal logits), renormalised
// weights, and the sigmoid gate of the shared expert.
//
// "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", MtpFfnWeightsGpu::Moe
// (router ffn_gate_inp, stacked experts, four shared-expert tensors).
//
// Every CTA normalises the row itself (it is only `hidden` floats) and owns
// a slice of the experts; the last CTA to finish (completion counter, no
// spinning) ranks the logits.
#include "host.h"

namespace mtp {

constexpr int kRouterThreads = 256;
constexpr int kRouterRowsPerCta = 8;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;

__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterParams r) {
  extern __shared__ __align__(16) float fsm[];  // [H] normalised row
  __shared__ float red[kRouterThreads / 32];
  __shared__ bool last;
  __shared__ unsigned long long kred[kRouterThreads / 32];
  __shared__ float lg[kMaxExperts];
  __shared__ float gate_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = r.H;
  pdl_wait();
  pdl_launch_dependents();

  float ss = 0.f;
  for (int k = tid; k < H; k += kRouterThreads) {
    const float v = r.u1[k];
    ss += v * v;
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < kRouterThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)H + r.eps);
  for (int k = tid; k < H; k += kRouterThreads) fsm[k] = r.u1[k] * inv * r.post_norm[k];
  __syncthreads();

  // CTA 0 also packs the normalised row for the expert projections
  if (blockIdx.x == 0 && r.xp) {
    for (int o0 = 0; o0 < H / 8; o0 += kRouterThreads) {
      const int o = o0 + tid;
      const bool valid = o < H / 8;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (valid)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = fsm[o * 8 + i];
      uint4 hi, lo;
      const float2 gx = pack8_group(v, valid, hi, lo);
      if (valid) {
        const int g = o / 4, t = o & 3;
        r.xp[xp_index(g, 0, t, 0, 1)] = hi;
        r.xp[xp_index(g, 0, t, 1, 1)] = lo;
        if (t == 0) r.xs[g] = gx;
      }
    }
  }

  // router logits for this CTA's experts
  const int e0 = blockIdx.x * kRouterRowsPerCta;
  for (int e = e0 + warp; e < min(r.E, e0 + kRouterRowsPerCta); e += kRouterThreads / 32) {
    const float* wr = r.router + (size_t)e * H;
    float acc = 0.f;
    for (int k = lane * 4; k < H; k += 128) {
      const float4 w = *reinterpret_cast<const float4*>(wr + k);
      acc = fmaf(w.x, fsm[k], fmaf(w.y, fsm[k + 1], fmaf(w.z, fsm[k + 2], fmaf(w.w, fsm[k + 3], acc))));
    }
    acc = warp_sum(acc);
    if (lane == 0) r.logits[e] = acc;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(r.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();

  // shared expert gate
  if (r.sh_gate_inp) {
    float g = 0.f;
    for (int k = tid; k < H; k += kRouterThreads) g = fmaf(r.sh_gate_inp[k], fsm[k], g);
    g = warp_sum(g);
    __syncthreads();
    if (lane == 0) red[warp] = g;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kRouterThreads / 32; ++w) t += red[w];
      gate_s = 1.f / (1.f + expf(-t));
    }
  }
  for (int e = tid; e < r.E; e += kRouterThreads) lg[e] = __ldcg(r.logits + e);
  __syncthreads();
  // top-k by repeated block argmax over the logits (softmax is monotone)
  float selv[kMaxTopK];
  int seli[kMaxTopK];
  for (int k = 0; k < r.top_k; ++k) {
    unsigned long long best = 0ull;
    for (int e = tid; e < r.E; e += kRouterThreads) {
      const unsigned long long key = argmax_key(lg[e], e);
      best = key > best ? key : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    if (lane == 0) kred[warp] = best;
    __syncthreads();
    unsigned long long b = kred[0];
    for (int w = 1; w < kRouterThreads / 32; ++w) b = kred[w] > b ? kred[w] : b;
    const int idx = argmax_key_index(b);
    selv[k] = argmax_key_value(b);
    seli[k] = idx;
    __syncthreads();
    if (tid == 0) lg[idx] = -INFINITY;
    __syncthreads();
  }
  if (tid == 0) {
    const float mx = selv[0];
    float den = 0.f;
    for (int k = 0; k < r.top_k; ++k) den += expf(selv[k] - mx);
    for (int k = 0; k < r.top_k; ++k) {
      r.sel[k] = seli[k];
      r.weight[k] = expf(selv[k] - mx) / den;
    }
    r.weight[r.top_k] = r.sh_gate_inp ? gate_s : 0.f;
    *r.counter = 0u;
  }
}

cudaError_t launch_router(const RouterParams& r, cudaStream_t st) {
  const int grid = (r.E + kRouterRowsPerCta - 1) / kRouterRowsPerCta;
  const size_t smem = (size_t)r.H * sizeof(float);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, router_kernel, r);
}

}  // namespace mtp
