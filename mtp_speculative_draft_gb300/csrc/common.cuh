// Shared device helpers of the draft-layer kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mtp {

constexpr int kGroup = 32;               // affine quantisation group
constexpr unsigned kWaitLimit = 2000;     // bounded device-side waits (polls of at most 1 ms)

// Workspace header shared by every entry point that takes a workspace.
// word 0: device error code; word 1: poll limit of the cross-CTA waits (0:
// the compiled default; set by mtp_workspace_set_wait_limit); then the
// completion counters.
struct WsHeader {
  int err;
  int wait_limit;
  int pad[30];
  unsigned counters[224];
};
static_assert(sizeof(WsHeader) == 1024, "workspace header is 1 KB");

// Device error word of a workspace (first error wins).
enum DevErr : int {
  kErrNone = 0,
  kErrMbarTimeout = 1,   // a wait for a TMA copy gave up
  kErrBadToken = 2,      // a token id outside [0, vocab) (row 0 used instead)
  kErrPhaseTimeout = 3,  // a wait for the previous phase of a one-row launch gave up
  kErrSplitTimeout = 4,  // a wait of the attention splits of a KV head for each other gave up
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  // The hint lets the hardware suspend the thread (up to 1 ms) until the
  // phase completes instead of spinning on issue slots.
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of `bar`; gives up after kWaitLimit polls (each
// suspends at most 1 ms) and returns false (the caller records the error).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (unsigned it = 0; it < kWaitLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 2-D tiled load of box (x = inner coordinate, y = row) into shared memory,
// completion signalled on `bar` (complete_tx bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- tensor core
// D = A(16x16 f16, row) * B(16x8 f16, col) + D, f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// 4-bit codes -> f16x2 as subnormal halves: a half with a zero exponent
// field is mantissa * 2^-24, so masking alone gives exact values with no
// offset.  Bits 0..3 and 16..19 of `w` give (c * 2^-24, c' * 2^-24); bits
// 4..7 and 20..23 give (16c * 2^-24, 16c' * 2^-24).  One LOP3 each; the
// 2^24 is restored in f32 after the tensor-core sums.
constexpr float kCodeScale = 16777216.f;   // 2^24
constexpr float kCodeUnscale = 1.f / 16777216.f;
__device__ __forceinline__ uint32_t codes_lo_f16x2(uint32_t w) { return w & 0x000F000Fu; }
__device__ __forceinline__ uint32_t codes_hi_f16x2(uint32_t w) { return w & 0x00F000F0u; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Orders this thread's earlier (acquired) view of global memory before its
// later bulk-copy (async proxy) reads of it.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses of shared memory (and,
// after a warp barrier, its warp's) before its later bulk copies into it.
__device__ __forceinline__ void fence_proxy_async_shared_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// GPU-scope counters: a barrier (bar.sync / bar.warp.sync) makes the block's
// or warp's earlier stores precede the releasing thread's operation, whose
// release then publishes them (the barrier-then-release pattern).
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned r;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "r"(v) : "memory");
  return r;
}
__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void set_dev_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Poll limit of a cross-CTA wait: the workspace header's override (the word
// after the error word) when it is positive, else `dflt`.
__device__ __forceinline__ unsigned wait_polls(const int* err, unsigned dflt) {
  const int v = err ? __ldcg(err + 1) : 0;
  return v > 0 ? (unsigned)v : dflt;
}

// One head vector (d <= 256) read by one warp (global or shared memory): per-head
// RMSNorm (when nw is given), rotary embedding of the first rot dims (pairs
// i, i + rot/2), times post_scale; the result goes to v in shared memory.
// All global loads are issued before any arithmetic.
__device__ __forceinline__ void warp_norm_rope(float* v, const float* src, int d, const float* nw,
                                               float eps, const float* rope_row, int rot,
                                               float post_scale, int lane) {
  float x[8], w[8], cs[4], sn[4];
  const int half = rot / 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = lane + 32 * j;
    x[j] = i < d ? src[i] : 0.f;
    w[j] = (nw && i < d) ? nw[i] : 1.f;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = lane + 32 * j;
    cs[j] = i < half ? rope_row[2 * i] : 1.f;
    sn[j] = i < half ? rope_row[2 * i + 1] : 0.f;
  }
  float inv = 1.f;
  if (nw) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += x[j] * x[j];
    inv = rsqrtf(warp_sum(ss) / (float)d + eps);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = lane + 32 * j;
    if (i < d) v[i] = x[j] * inv * w[j];
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      const float a = v[i], b = v[i + half];
      v[i] = a * cs[j] - b * sn[j];
      v[i + half] = a * sn[j] + b * cs[j];
    }
  }
  __syncwarp();
  if (post_scale != 1.f)
    for (int i = lane; i < d; i += 32) v[i] *= post_scale;
  __syncwarp();
}

}  // namespace mtp
