// MoE router of the draft layer: RMSNorm of the residual row, float32 router
// projection, softmax, top-k (lowest index among equal logits), renormalised
// weights, and the sigmoid gate of the shared expert.
//
// "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", MtpFfnWeightsGpu::Moe
// (router ffn_gate_inp, stacked experts, four shared-expert tensors).
//
// Each CTA owns a few expert rows, one warp each: the rows do not depend on
// the previous kernel, so they are bulk-copied into shared memory before the
// wait on it.  Every CTA normalises the row itself (`hidden` floats); CTA 0
// also packs it for the expert projections and computes the shared-expert
// gate.  The last CTA to finish (completion counter, no spinning) ranks the
// logits with one warp.
#include "host.h"

namespace mtp {

constexpr int kRouterThreads = 128;  // one warp per expert row of the CTA
constexpr int kRouterMaxRows = kRouterThreads / 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr size_t kRouterSmemLimit = 200 * 1024;

__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterParams r) {
  extern __shared__ __align__(16) float smem[];  // [rows][H] router rows, [H] normalised row, [H] gate
  __shared__ float red[kRouterThreads / 32];
  __shared__ bool last;
  __shared__ float lg[kMaxExperts];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = r.H;
  const int e0 = blockIdx.x * r.rows_per_cta;
  const int nrows = min(r.rows_per_cta, r.E - e0);
  float* wsm = smem;
  float* fsm = smem + (size_t)r.rows_per_cta * H;
  float* gsm = fsm + H;  // CTA 0: the shared-expert gate vector
  const bool gate_copy = blockIdx.x == 0 && r.sh_gate_inp &&
                         (reinterpret_cast<uintptr_t>(r.sh_gate_inp) & 15) == 0;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)((nrows + (gate_copy ? 1 : 0)) * H * 4));
    for (int i = 0; i < nrows; ++i)
      bulk_load(wsm + (size_t)i * H, r.router + (size_t)(e0 + i) * H, (uint32_t)(H * 4), &bar,
                l2_policy_evict_first());
    if (gate_copy) bulk_load(gsm, r.sh_gate_inp, (uint32_t)(H * 4), &bar, l2_policy_evict_first());
  }
  pdl_wait();
  pdl_launch_dependents();

  float ss = 0.f;
#pragma unroll 4
  for (int k = tid * 4; k < H; k += kRouterThreads * 4) {  // loads issued together
    const float4 v = __ldcg(reinterpret_cast<const float4*>(r.u1 + k));
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < kRouterThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)H + r.eps);
#pragma unroll 8
  for (int k = tid; k < H; k += kRouterThreads) fsm[k] = __ldcg(r.u1 + k) * inv * r.post_norm[k];
  __syncthreads();

  if (blockIdx.x == 0) {
    // the packed normalised row for the expert projections
    if (r.xp) {
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
    // shared expert gate (from the copy when it was aligned for one)
    float gsum = 0.f;
    if (gate_copy) {
      if (mbar_wait_bounded(&bar, 0))
        for (int k = tid; k < H; k += kRouterThreads) gsum = fmaf(gsm[k], fsm[k], gsum);
      else if (tid == 0)
        set_dev_error(r.err, kErrMbarTimeout);
    } else if (r.sh_gate_inp) {
      for (int k = tid; k < H; k += kRouterThreads) gsum = fmaf(r.sh_gate_inp[k], fsm[k], gsum);
    }
    gsum = warp_sum(gsum);
    __syncthreads();
    if (lane == 0) red[warp] = gsum;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kRouterThreads / 32; ++w) t += red[w];
      r.weight[r.top_k] = r.sh_gate_inp ? 1.f / (1.f + expf(-t)) : 0.f;
    }
  }

  // router logits of this CTA's rows (from shared memory)
  bool ok = true;
  if (nrows > 0 || gate_copy) ok = mbar_wait_bounded(&bar, 0);
  if (!ok) {
    if (tid == 0) set_dev_error(r.err, kErrMbarTimeout);
  } else if (warp < nrows) {
    const float* wr = wsm + (size_t)warp * H;
    float acc0 = 0.f, acc1 = 0.f;
    int k = lane * 4;
    for (; k + 128 + 3 < H; k += 256) {  // two independent chains
      const float4 w0 = *reinterpret_cast<const float4*>(wr + k);
      const float4 x0 = *reinterpret_cast<const float4*>(fsm + k);
      const float4 w1 = *reinterpret_cast<const float4*>(wr + k + 128);
      const float4 x1 = *reinterpret_cast<const float4*>(fsm + k + 128);
      acc0 = fmaf(w0.x, x0.x, fmaf(w0.y, x0.y, fmaf(w0.z, x0.z, fmaf(w0.w, x0.w, acc0))));
      acc1 = fmaf(w1.x, x1.x, fmaf(w1.y, x1.y, fmaf(w1.z, x1.z, fmaf(w1.w, x1.w, acc1))));
    }
    for (; k + 3 < H; k += 128) {  // H is a multiple of 4
      const float4 w0 = *reinterpret_cast<const float4*>(wr + k);
      const float4 x0 = *reinterpret_cast<const float4*>(fsm + k);
      acc0 = fmaf(w0.x, x0.x, fmaf(w0.y, x0.y, fmaf(w0.z, x0.z, fmaf(w0.w, x0.w, acc0))));
    }
    const float acc = warp_sum(acc0 + acc1);
    if (lane == 0) r.logits[e0 + warp] = acc;
  }
  __syncthreads();  // the CTA's logits (and CTA 0's gate), then one release
  if (tid == 0) last = atom_add_acq_rel_gpu(r.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last || warp != 0) return;
  asm volatile("fence.acq_rel.gpu;" ::: "memory");  // every CTA's logits, for this warp

  // top-k by repeated warp argmax over the logits (softmax is monotone)
  for (int e = lane; e < r.E; e += 32) lg[e] = __ldcg(r.logits + e);
  __syncwarp();
  float selv[kMaxTopK];
  int seli[kMaxTopK];
  for (int k = 0; k < r.top_k; ++k) {
    unsigned long long best = 0ull;
    for (int e = lane; e < r.E; e += 32) {
      const unsigned long long key = argmax_key(lg[e], e);
      best = key > best ? key : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int idx = argmax_key_index(best);
    selv[k] = argmax_key_value(best);
    seli[k] = idx;
    if (lane == (idx & 31)) lg[idx] = -INFINITY;
    __syncwarp();
  }
  if (lane == 0) {
    const float mx = selv[0];
    float den = 0.f;
    for (int k = 0; k < r.top_k; ++k) den += expf(selv[k] - mx);
    for (int k = 0; k < r.top_k; ++k) {
      r.sel[k] = seli[k];
      r.weight[k] = expf(selv[k] - mx) / den;
    }
    *r.counter = 0u;
  }
}

cudaError_t launch_router(const RouterParams& r_in, cudaStream_t st) {
  RouterParams r = r_in;
  // as many rows per CTA (one warp each) as fit beside the normalised row
  int rows = kRouterMaxRows;
  while (rows > 1 && (size_t)(rows + 2) * r.H * sizeof(float) > kRouterSmemLimit) --rows;
  if ((size_t)(rows + 2) * r.H * sizeof(float) > kRouterSmemLimit) return cudaErrorInvalidValue;
  r.rows_per_cta = rows;
  const int grid = (r.E + rows - 1) / rows;
  const size_t smem = (size_t)(rows + 2) * r.H * sizeof(float);  // + the normalised row, the gate
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRouterSmemLimit);
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
