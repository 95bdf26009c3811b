// KV catch-up of a target batch on the 5th-generation tensor cores.
//
// "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", process_target_batch and
// append_attention_kv: for seq rows at once, the draft layer's K/V rows are
// computed from the embedding rows and the target's hidden rows shifted one
// row right (row 0 reads the pending hidden, or zeros for a cold prompt):
//   u = eh_proj [RMSNorm(e)*enorm ; RMSNorm(h)*hnorm]   (eps 1e-6)
//   x = RMSNorm(u)*attn_norm;  k = W_k x (+ per-head k RMSNorm), v = W_v x
//   k rotated at its position, both appended to the cache.
// No attention, FFN or head runs.
//
// With seq in the hundreds the projections are a dense contraction, so they
// run on tcgen05 (bf16 operands, f32 accumulators in tensor memory) instead
// of the weight-streaming GEMV kernels, and every weight is read once per
// tile of activation rows.  Accuracy: the dequantised weight s*q + b and the
// activations are each split into bf16 hi + lo parts, and each K16 step
// issues hi*hi + hi*lo + lo*hi (the dropped lo*lo term is ~2^-17 relative).
//
// Launches (programmatic dependent launch between them):
//   1. pack:   rows of [RMSNorm(e)*enorm ; RMSNorm(h)*hnorm] as bf16 hi/lo
//   2. GEMM:   u = eh_proj x1 (split-K partials in f32)
//   3. pack:   x2 = RMSNorm(u)*attn_norm as bf16 hi/lo (sums the partials)
//   4. GEMM:   [k | v] = [W_k ; W_v] x2 (one launch over both matrices)
//   5. append: sums the partials, per-head k RMSNorm, RoPE, cache rows.
#include <cuda_bf16.h>

#include "host.h"
#include "tc5.cuh"

namespace mtp {

// ------------------------------------------------------------------ GEMM
// out[split][r][col0 + n] = sum over this split's K of x[r][k] * w[n][k],
// w[n][k] = s[n][k/32] * code + b[n][k/32].  CTA tile: 128 weight rows x BN
// activation rows; K in stages of 64 (one 128-byte swizzle row of bf16).
struct TcSeg {
  const uint32_t* q;   // [N][K/8]
  const float* s;      // [N][K/32]
  const float* b;
  int N;
  int tiles;           // ceil(N / 128)
  int out_col0;
};

struct TcGemmParams {
  CUtensorMap xh, xl;  // bf16 [rows][K] hi / lo parts, box 64 x BN, 128-byte swizzle
  TcSeg seg[2];
  int nseg;
  int K;
  int rows;
  int ks_per_split;    // 64-wide K stages per split (grid.z splits)
  float* out;          // [nsplit][rows][ldo]
  int ldo;
  size_t split_stride; // floats between splits
  int* err;
};

template <int BN>
struct TcCfg {
  static constexpr int kA = 128 * 128;  // one operand tile: 128 rows x 128 bytes
  static constexpr int kB = BN * 128;
  static constexpr int kStage = 2 * kA + 2 * kB;
  static constexpr int kStages = BN >= 128 ? 3 : 4;
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr int kSmem = kStages * kStage + 1024 + 256;  // + alignment, barriers
};

// One 16-byte chunk (8 consecutive k) of a weight row: codes of word w,
// group scale and bias folded as s16 = 16 s, bb = b - 16 s so that
// s * c + b = s16 * (1 + c / 16) + bb with 1 + c/16 built from the bits.
__device__ __forceinline__ void dequant_chunk(uint32_t w, float s16, float bb, uint4& hi,
                                              uint4& lo) {
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t bits = 0x3F800000u | (((w >> (4 * e)) & 0xFu) << 19);
    v[e] = fmaf(s16, __uint_as_float(bits), bb);
  }
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 hp = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    const float2 hf = __bfloat1622float2(hp);
    const __nv_bfloat162 lp = __floats2bfloat162_rn(v[2 * j] - hf.x, v[2 * j + 1] - hf.y);
    h[j] = *reinterpret_cast<const uint32_t*>(&hp);
    l[j] = *reinterpret_cast<const uint32_t*>(&lp);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

template <int BN>
__global__ void __launch_bounds__(256, 1) tc_affine_gemm_kernel(const __grid_constant__ TcGemmParams p) {
  using Cf = TcCfg<BN>;
  constexpr int S = Cf::kStages;
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + S * Cf::kStage);
  uint64_t* empty = full + S;
  uint64_t* accb = empty + S;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int tile = blockIdx.x, si = 0;
  if (p.nseg > 1 && tile >= p.seg[0].tiles) {
    tile -= p.seg[0].tiles;
    si = 1;
  }
  const TcSeg& sg = p.seg[si];
  const int n0 = tile * 128;
  const int r0 = blockIdx.y * BN;
  const int KS = p.K / 64;
  const int ks0 = blockIdx.z * p.ks_per_split;
  const int nks = min(p.ks_per_split, KS - ks0);  // >= 1 (host)

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1 + 4);  // the activation copy + one arrival per dequant warp
      mbar_init(&empty[i], 1);     // the MMA commit
    }
    mbar_init(accb, 1);
    mbar_fence_init();
  }
  if (warp == 1) tc5::alloc(tslot, Cf::kTmemCols);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = *tslot;
  pdl_launch_dependents();

  auto a_hi = [&](int s) { return sm + s * Cf::kStage; };
  auto a_lo = [&](int s) { return sm + s * Cf::kStage + Cf::kA; };
  auto b_hi = [&](int s) { return sm + s * Cf::kStage + 2 * Cf::kA; };
  auto b_lo = [&](int s) { return sm + s * Cf::kStage + 2 * Cf::kA + Cf::kB; };

  if (warp == 0) {
    // activation producer: the activations come from the previous launch
    if (lane == 0) {
      tma_prefetch_desc(&p.xh);
      tma_prefetch_desc(&p.xl);
      pdl_wait();
      const uint64_t pol = l2_policy_evict_last();  // re-read by every weight tile
      for (int it = 0; it < nks; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
          set_dev_error(p.err, kErrMbarTimeout);
          break;
        }
        mbar_arrive_expect_tx(&full[s], 2u * Cf::kB);
        const int kx = (ks0 + it) * 64;
        tma_load_2d(b_hi(s), &p.xh, &full[s], kx, r0, pol);
        tma_load_2d(b_lo(s), &p.xl, &full[s], kx, r0, pol);
      }
    }
  } else if (warp == 1) {
    // MMA issuer (one thread); the commit to accb follows every MMA it issued
    if (lane == 0) {
      constexpr uint32_t idesc = tc5::idesc_bf16_f32(128, BN);
      for (int it = 0; it < nks; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait_bounded(&full[s], ph)) {
          set_dev_error(p.err, kErrMbarTimeout);
          break;
        }
        tc5::fence_after_sync();
        const uint64_t ah = tc5::desc_k_sw128(smem_u32(a_hi(s)));
        const uint64_t al = tc5::desc_k_sw128(smem_u32(a_lo(s)));
        const uint64_t bh = tc5::desc_k_sw128(smem_u32(b_hi(s)));
        const uint64_t bl = tc5::desc_k_sw128(smem_u32(b_lo(s)));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t o = (uint64_t)(2 * kk);  // 32 bytes of K per K16 step
          tc5::mma_bf16(tmem, ah + o, bh + o, idesc, (it | kk) != 0 ? 1u : 0u);
          tc5::mma_bf16(tmem, ah + o, bl + o, idesc, 1u);
          tc5::mma_bf16(tmem, al + o, bh + o, idesc, 1u);
        }
        tc5::commit(&empty[s]);
      }
      tc5::commit(accb);
    }
  } else if (warp >= 4) {
    // dequantising producers: thread i writes weight row n0 + i of every stage
    const int i = tid - 128;
    const int n = n0 + i;
    const bool row_ok = n < sg.N;
    const size_t nr = row_ok ? (size_t)n : 0;
    const uint4* qrow = reinterpret_cast<const uint4*>(sg.q + nr * (size_t)(p.K / 8));
    const float2* srow = reinterpret_cast<const float2*>(sg.s + nr * (size_t)(p.K / 32));
    const float2* brow = reinterpret_cast<const float2*>(sg.b + nr * (size_t)(p.K / 32));
    const uint32_t rbase = (uint32_t)i * 128u, rx = (uint32_t)(i & 7);
    auto load = [&](int it, uint4& w0, uint4& w1, float2& sv, float2& bv) {
      if (row_ok && it < nks) {
        const int ks = ks0 + it;  // words 8 ks .. 8 ks + 7, groups 2 ks and 2 ks + 1
        w0 = __ldg(qrow + 2 * ks);
        w1 = __ldg(qrow + 2 * ks + 1);
        sv = __ldg(srow + ks);
        bv = __ldg(brow + ks);
      } else {
        w0 = w1 = make_uint4(0u, 0u, 0u, 0u);
        sv = bv = make_float2(0.f, 0.f);
      }
    };
    bool ok = true;
    auto stage = [&](int it, const uint4& w0, const uint4& w1, const float2& sv, const float2& bv) {
      const int s = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
        if (lane == 0) set_dev_error(p.err, kErrMbarTimeout);
        ok = false;
        return;
      }
      uint8_t* ah = a_hi(s) + rbase;
      uint8_t* al = a_lo(s) + rbase;
      const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const float s16[2] = {16.f * sv.x, 16.f * sv.y};
      const float bb[2] = {bv.x - 16.f * sv.x, bv.y - 16.f * sv.y};
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 hi, lo;
        dequant_chunk(words[c], s16[c >> 2], bb[c >> 2], hi, lo);
        const uint32_t off = ((uint32_t)c ^ rx) << 4;
        *reinterpret_cast<uint4*>(ah + off) = hi;
        *reinterpret_cast<uint4*>(al + off) = lo;
      }
      tc5::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc5::mbar_arrive(&full[s]);
    };
    // two stages of weights in flight in registers
    uint4 a0, a1, b0, b1;
    float2 as, ab, bs, bb;
    load(0, a0, a1, as, ab);
    load(1, b0, b1, bs, bb);
    for (int it = 0; it < nks && ok; it += 2) {
      {
        const uint4 w0 = a0, w1 = a1;
        const float2 sv = as, bv = ab;
        load(it + 2, a0, a1, as, ab);
        stage(it, w0, w1, sv, bv);
      }
      if (it + 1 < nks && ok) {
        const uint4 w0 = b0, w1 = b1;
        const float2 sv = bs, bv = bb;
        load(it + 3, b0, b1, bs, bb);
        stage(it + 1, w0, w1, sv, bv);
      }
    }
    // epilogue: TMEM lanes 32 q .. 32 q + 31 hold weight rows n0 + 32 q + lane
    if (!mbar_wait_bounded(accb, 0u) && lane == 0) set_dev_error(p.err, kErrMbarTimeout);
    tc5::fence_after_sync();
    const int q = warp - 4;
    const int nrow = n0 + 32 * q + lane;
    float* out = p.out + (size_t)blockIdx.z * p.split_stride + sg.out_col0 + nrow;
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
      uint32_t v[16];
      tc5::ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c, v);
      tc5::ld_wait();
      if (nrow < sg.N) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = r0 + c + j;
          if (r < p.rows) out[(size_t)r * p.ldo] = __uint_as_float(v[j]);
        }
      }
    }
    tc5::fence_before_sync();
  }
  __syncthreads();
  if (warp == 1) {
    tc5::fence_after_sync();
    tc5::dealloc(tmem, Cf::kTmemCols);
  }
}

// ------------------------------------------------------------------ packing
constexpr int kCatchThreads = 256;

__device__ __forceinline__ float block_sum_ct(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kCatchThreads / 32; ++w) t += red[w];
  return t;
}

// Four values as bf16 hi and lo parts (two 8-byte stores).
__device__ __forceinline__ void store_hilo4(__nv_bfloat16* xh, __nv_bfloat16* xl, size_t off,
                                            float4 v) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(v.z, v.w);
  const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
  const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
  const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
  uint2 hh, ll;
  hh.x = *reinterpret_cast<const uint32_t*>(&h0);
  hh.y = *reinterpret_cast<const uint32_t*>(&h1);
  ll.x = *reinterpret_cast<const uint32_t*>(&l0);
  ll.y = *reinterpret_cast<const uint32_t*>(&l1);
  *reinterpret_cast<uint2*>(xh + off) = hh;
  *reinterpret_cast<uint2*>(xl + off) = ll;
}

struct CatchPack1Args {
  const float* table;    // [vocab][H] or null (rows given)
  const int* tokens;
  int vocab;
  const float* rows;     // [seq][H]
  const float* target;   // [seq][H]: row i - 1 feeds row i
  const float* pending;  // [H] feeds row 0, or null (zeros)
  const float* enorm;
  const float* hnorm;
  int H;
  __nv_bfloat16* xh;     // [seq][2H]
  __nv_bfloat16* xl;
  int* err;
};

// Row i: [RMSNorm(e_i) * enorm ; RMSNorm(h_i) * hnorm] (eps 1e-6), h_i the
// shifted target hidden, as bf16 hi/lo parts.
__global__ void __launch_bounds__(kCatchThreads) catchup_pack1_kernel(const CatchPack1Args a) {
  __shared__ float red[kCatchThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x, H = a.H;
  const float* e;
  if (a.table) {
    int tok = a.tokens[i];
    if (tok < 0 || tok >= a.vocab) {
      if (threadIdx.x == 0) set_dev_error(a.err, kErrBadToken);
      tok = 0;
    }
    e = a.table + (size_t)tok * H;
  } else {
    e = a.rows + (size_t)i * H;
  }
  const float* h = i > 0 ? a.target + (size_t)(i - 1) * H : a.pending;  // null: zeros
  float se = 0.f, sh = 0.f;
  for (int k = threadIdx.x * 4; k < H; k += kCatchThreads * 4) {
    const float4 ev = *reinterpret_cast<const float4*>(e + k);
    se += ev.x * ev.x + ev.y * ev.y + ev.z * ev.z + ev.w * ev.w;
    if (h) {
      const float4 hv = *reinterpret_cast<const float4*>(h + k);
      sh += hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w;
    }
  }
  se = block_sum_ct(se, red);
  sh = block_sum_ct(sh, red);
  const float re = rsqrtf(se / (float)H + 1e-6f), rh = rsqrtf(sh / (float)H + 1e-6f);
  const size_t row = (size_t)i * 2 * H;
  for (int k = threadIdx.x * 4; k < H; k += kCatchThreads * 4) {
    const float4 ev = *reinterpret_cast<const float4*>(e + k);
    const float4 ew = *reinterpret_cast<const float4*>(a.enorm + k);
    store_hilo4(a.xh, a.xl, row + k,
                make_float4(ev.x * re * ew.x, ev.y * re * ew.y, ev.z * re * ew.z, ev.w * re * ew.w));
    float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h) hv = *reinterpret_cast<const float4*>(h + k);
    const float4 hw = *reinterpret_cast<const float4*>(a.hnorm + k);
    store_hilo4(a.xh, a.xl, row + H + k,
                make_float4(hv.x * rh * hw.x, hv.y * rh * hw.y, hv.z * rh * hw.z, hv.w * rh * hw.w));
  }
}

struct CatchPack2Args {
  const float* upart;    // [nsplit][seq][H]
  int nsplit;
  size_t split_stride;
  const float* w;        // attn_norm
  float eps;
  int H;
  __nv_bfloat16* xh;     // [seq][H]
  __nv_bfloat16* xl;
};

// Row i: RMSNorm(u_i) * attn_norm as bf16 hi/lo, u_i the sum of the split
// partials in split order.
__global__ void __launch_bounds__(kCatchThreads) catchup_pack2_kernel(const CatchPack2Args a) {
  __shared__ float red[kCatchThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x, H = a.H;
  const float* u0 = a.upart + (size_t)i * H;
  auto urow = [&](int k) {
    float4 t = *reinterpret_cast<const float4*>(u0 + k);
    for (int sp = 1; sp < a.nsplit; ++sp) {
      const float4 v = *reinterpret_cast<const float4*>(u0 + sp * a.split_stride + k);
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    return t;
  };
  float ss = 0.f;
  for (int k = threadIdx.x * 4; k < H; k += kCatchThreads * 4) {
    const float4 v = urow(k);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum_ct(ss, red);
  const float r = rsqrtf(ss / (float)H + a.eps);
  for (int k = threadIdx.x * 4; k < H; k += kCatchThreads * 4) {
    const float4 v = urow(k);
    const float4 w = *reinterpret_cast<const float4*>(a.w + k);
    store_hilo4(a.xh, a.xl, (size_t)i * H + k,
                make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w));
  }
}

struct CatchAppendArgs {
  const float* kvpart;   // [nsplit][seq][nkv*dqk + nkv*dv]
  int nsplit;
  size_t split_stride;
  int nkv, dqk, dv, rot;
  const float* k_norm;   // [dqk] or null
  float eps;
  const float* rope;     // [pos][rot/2] (cos, sin)
  int pos0;              // rope position of row 0
  float* kc;             // [nkv][cap][dqk]
  float* vc;             // [nkv][cap][dv]
  int cap;
  int row0;              // cache row of batch row 0
};

// One warp per (row, KV head): K = per-head RMSNorm (when given) then RoPE,
// V as projected; both written to the cache.
__global__ void catchup_append_kernel(const CatchAppendArgs a) {
  extern __shared__ float kbuf[];  // [warps][dqk]
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int width = a.nkv * (a.dqk + a.dv);
  float* kb = kbuf + (size_t)h * a.dqk;
  const float* src = a.kvpart + (size_t)i * width;
  for (int d = lane; d < a.dqk; d += 32) {
    float t = 0.f;
    for (int sp = 0; sp < a.nsplit; ++sp) t += src[sp * a.split_stride + h * a.dqk + d];
    kb[d] = t;
  }
  __syncwarp();
  warp_norm_rope(kb, kb, a.dqk, a.k_norm, a.eps, a.rope + (size_t)(a.pos0 + i) * a.rot, a.rot, 1.f,
                 lane);
  float* kdst = a.kc + ((size_t)h * a.cap + a.row0 + i) * a.dqk;
  for (int d = lane; d < a.dqk; d += 32) kdst[d] = kb[d];
  float* vdst = a.vc + ((size_t)h * a.cap + a.row0 + i) * a.dv;
  const float* vs = src + a.nkv * a.dqk + h * a.dv;
  for (int d = lane; d < a.dv; d += 32) {
    float t = 0.f;
    for (int sp = 0; sp < a.nsplit; ++sp) t += vs[sp * a.split_stride + d];
    vdst[d] = t;
  }
}

// ------------------------------------------------------------------ host side
static cudaLaunchAttribute pdl_attr_ct() {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  return at;
}

static int tc_bn_for_rows(int rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128; }

// Split-K count (at least 8 stages per split).  One CTA runs per SM, so the
// GEMM takes ceil(CTAs / SMs) waves of one split's K stages plus a fixed
// cost per wave (TMEM allocation, pipeline fill, epilogue: about 4 stages);
// each further split also writes (and the next kernel reads) one more f32
// partial of rows x N, counted in waves of one K stage (about 4.8 MB of HBM
// traffic each, as measured at 128 x 128 tiles).  The split count with the
// lowest total wins (eh_proj at 512 rows: 4 splits in 5 waves of 40 stages
// instead of 2 waves of 160).
#ifndef MTP_CATCH_WAVE_COST
#define MTP_CATCH_WAVE_COST 4  // fixed cost of a wave, in K stages (tuning knob)
#endif
static int tc_splits(int tiles, int rows, int K) {
  const int bn = tc_bn_for_rows(rows);
  const int ctas = tiles * ((rows + bn - 1) / bn);
  const int KS = K / 64;
  const int cap = KS / 8 > 1 ? KS / 8 : 1;
  const int sms = sm_count();
  const double split_cost = (double)rows * tiles * 128 * 8.0 / 4.8e6;
  int best = 1;
  double best_cost = 1e300;
  for (int ns = 1; ns <= cap; ++ns) {
    const int per = (KS + ns - 1) / ns;
    const int n = (KS + per - 1) / per;  // no empty split
    const long long waves = ((long long)ctas * n + sms - 1) / sms;
    const double cost = (double)waves * (per + MTP_CATCH_WAVE_COST) + (n - 1) * split_cost;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = n;
    }
  }
  return best;
}

template <int BN>
static cudaError_t launch_tc_t(const TcGemmParams& p, dim3 grid, cudaStream_t st) {
  using Cf = TcCfg<BN>;
  static thread_local int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(tc_affine_gemm_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute at = pdl_attr_ct();
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, tc_affine_gemm_kernel<BN>, p);
}

// x: bf16 hi/lo [rows][K]; weights: one or two segments stacked along the
// output columns; out: [nsplit][rows][ldo] f32 partials.
static cudaError_t launch_tc_gemm(const __nv_bfloat16* xh, const __nv_bfloat16* xl, int rows,
                                  int K, const mtp_affine4* w, int nw, float* out, int ldo,
                                  int nsplit, int* err, cudaStream_t st) {
  TcGemmParams p = {};
  const int bn = tc_bn_for_rows(rows);
  cudaError_t e = encode_bf16_rows_map(&p.xh, xh, (uint64_t)rows, (uint64_t)K, bn);
  if (e == cudaSuccess) e = encode_bf16_rows_map(&p.xl, xl, (uint64_t)rows, (uint64_t)K, bn);
  if (e != cudaSuccess) return e;
  int tiles = 0, col = 0;
  for (int s = 0; s < nw; ++s) {
    p.seg[s].q = w[s].q;
    p.seg[s].s = w[s].s;
    p.seg[s].b = w[s].b;
    p.seg[s].N = w[s].n;
    p.seg[s].tiles = (w[s].n + 127) / 128;
    p.seg[s].out_col0 = col;
    col += w[s].n;
    tiles += p.seg[s].tiles;
  }
  p.nseg = nw;
  p.K = K;
  p.rows = rows;
  const int KS = K / 64;
  p.ks_per_split = (KS + nsplit - 1) / nsplit;
  p.out = out;
  p.ldo = ldo;
  p.split_stride = (size_t)rows * ldo;
  p.err = err;
  const dim3 grid(tiles, (rows + bn - 1) / bn, nsplit);
  switch (bn) {
    case 16: return launch_tc_t<16>(p, grid, st);
    case 32: return launch_tc_t<32>(p, grid, st);
    case 64: return launch_tc_t<64>(p, grid, st);
    default: return launch_tc_t<128>(p, grid, st);
  }
}

template <class K, class A>
static cudaError_t launch_small(K kern, const A& args, dim3 grid, dim3 block, size_t smem,
                                cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at = pdl_attr_ct();
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, kern, args);
}

struct CatchWs {
  __nv_bfloat16 *x1h, *x1l, *x2h, *x2l;
  float *upart, *kvpart;
  int ns1, ns2;
};

static size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: 1 KB header, x1 hi/lo [seq][2H], u partials [ns1][seq][H],
// x2 hi/lo [seq][H], k/v partials [ns2][seq][nkv (dqk + dv)].
static size_t carve_catch(uint8_t* base, const mtp_layer_desc* L, int seq, CatchWs* w) {
  const int H = L->hidden;
  const mtp_attn_geom& g = L->attn;
  const int nkv = g.n_kv_heads, width = nkv * (g.head_dim_qk + g.head_dim_v);
  w->ns1 = tc_splits((H + 127) / 128, seq, 2 * H);
  w->ns2 = tc_splits((nkv * g.head_dim_qk + 127) / 128 + (nkv * g.head_dim_v + 127) / 128, seq, H);
  size_t off = 1024;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off = a256(off + bytes);
    return p;
  };
  w->x1h = reinterpret_cast<__nv_bfloat16*>(take((size_t)seq * 2 * H * 2));
  w->x1l = reinterpret_cast<__nv_bfloat16*>(take((size_t)seq * 2 * H * 2));
  w->upart = reinterpret_cast<float*>(take((size_t)w->ns1 * seq * H * 4));
  w->x2h = reinterpret_cast<__nv_bfloat16*>(take((size_t)seq * H * 2));
  w->x2l = reinterpret_cast<__nv_bfloat16*>(take((size_t)seq * H * 2));
  w->kvpart = reinterpret_cast<float*>(take((size_t)w->ns2 * seq * width * 4));
  return off + 256;
}

}  // namespace mtp

using namespace mtp;

extern "C" {

size_t mtp_kv_catch_up_workspace_bytes(const mtp_layer_desc* L, int32_t seq) {
  if (!L || seq <= 0 || L->hidden <= 0 || L->attn.n_kv_heads <= 0) return 0;
  CatchWs w;
  return carve_catch(nullptr, L, seq, &w);
}

mtp_status mtp_kv_catch_up(const mtp_layer_desc* L, const int32_t* d_tokens,
                           const float* d_embed_rows, const float* d_target,
                           const float* d_pending, int32_t seq, int32_t cache_len,
                           int32_t pos_base, void* d_ws, size_t ws_bytes, void* stream) {
  if (!L) return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: null layer");
  const int H = L->hidden;
  if (H <= 0 || H % 128) return fail(MTP_ERR_UNSUPPORTED, "mtp_kv_catch_up: hidden % 128 != 0");
  if (seq < 1 || seq > 65535) return fail(MTP_ERR_UNSUPPORTED, "mtp_kv_catch_up: seq must be in 1..65535");
  const mtp_attn_geom& g = L->attn;
  if (g.n_kv_heads <= 0 || g.n_kv_heads > 32 || g.head_dim_qk <= 0 || g.head_dim_qk % 32 ||
      g.head_dim_qk > 256 || g.head_dim_v <= 0 || g.head_dim_v % 32 || g.head_dim_v > 256)
    return fail(MTP_ERR_UNSUPPORTED, "mtp_kv_catch_up: 1..32 KV heads, head dims multiples of 32 up to 256");
  if (g.rot_dim < 0 || g.rot_dim % 2 || g.rot_dim > g.head_dim_qk)
    return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: rot_dim must be even and <= head_dim_qk");
  if (!(L->eps >= 0.f) || !(g.eps >= 0.f)) return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: eps must be >= 0");
  mtp_status s;
  if ((s = check_affine(&L->eh_proj, H, 2 * H, "eh_proj", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->wk, g.n_kv_heads * g.head_dim_qk, H, "wk", true)) != MTP_OK) return s;
  if ((s = check_affine(&L->wv, g.n_kv_heads * g.head_dim_v, H, "wv", true)) != MTP_OK) return s;
  const float* norms[] = {L->enorm, L->hnorm, L->attn_norm};
  for (const float* p : norms)
    if (!p || !aligned16(p))
      return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: norm weights must be non-null and 16-byte aligned");
  if (!L->rope || !L->k_cache || !L->v_cache || L->cache_cap <= 0)
    return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: rope table and KV cache are required");
  if (!aligned16(L->k_cache) || !aligned16(L->v_cache))
    return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: caches must be 16-byte aligned");
  if (L->embed ? !d_tokens : (!d_embed_rows || !aligned16(d_embed_rows)))
    return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: tokens (with a table) or embedding rows are required");
  if (L->embed && !aligned16(L->embed))
    return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: embedding table must be 16-byte aligned");
  if ((seq > 1 && !d_target) || (d_target && !aligned16(d_target)) || (d_pending && !aligned16(d_pending)))
    return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: target rows (seq > 1) must be 16-byte aligned");
  if (cache_len < 0 || pos_base < 0) return fail(MTP_ERR_INVALID_ARG, "mtp_kv_catch_up: negative position");
  if (cache_len + seq > L->cache_cap)
    return fail(MTP_ERR_CAPACITY, "mtp_kv_catch_up: cache_len + seq exceeds the cache capacity");
  if (!d_ws || ws_bytes < mtp_kv_catch_up_workspace_bytes(L, seq))
    return fail(MTP_ERR_WORKSPACE, "mtp_kv_catch_up: workspace too small");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CatchWs w;
  carve_catch(static_cast<uint8_t*>(d_ws), L, seq, &w);
  int* err = static_cast<int*>(d_ws);  // the workspace header's error word
  const int nkv = g.n_kv_heads, width = nkv * (g.head_dim_qk + g.head_dim_v);

  CatchPack1Args p1 = {};
  p1.table = L->embed;
  p1.tokens = d_tokens;
  p1.vocab = L->vocab;
  p1.rows = d_embed_rows;
  p1.target = d_target;
  p1.pending = d_pending;
  p1.enorm = L->enorm;
  p1.hnorm = L->hnorm;
  p1.H = H;
  p1.xh = w.x1h;
  p1.xl = w.x1l;
  p1.err = err;
  cudaError_t e = launch_small(catchup_pack1_kernel, p1, dim3(seq), dim3(kCatchThreads), 0, st);
  if (e != cudaSuccess) return cuda_fail(e, "catch-up pack launch");

  e = launch_tc_gemm(w.x1h, w.x1l, seq, 2 * H, &L->eh_proj, 1, w.upart, H, w.ns1, err, st);
  if (e != cudaSuccess) return cuda_fail(e, "catch-up eh_proj launch");

  CatchPack2Args p2 = {};
  p2.upart = w.upart;
  p2.nsplit = w.ns1;
  p2.split_stride = (size_t)seq * H;
  p2.w = L->attn_norm;
  p2.eps = L->eps;
  p2.H = H;
  p2.xh = w.x2h;
  p2.xl = w.x2l;
  e = launch_small(catchup_pack2_kernel, p2, dim3(seq), dim3(kCatchThreads), 0, st);
  if (e != cudaSuccess) return cuda_fail(e, "catch-up attention-norm launch");

  const mtp_affine4 kv[2] = {L->wk, L->wv};
  e = launch_tc_gemm(w.x2h, w.x2l, seq, H, kv, 2, w.kvpart, width, w.ns2, err, st);
  if (e != cudaSuccess) return cuda_fail(e, "catch-up k/v launch");

  CatchAppendArgs ap = {};
  ap.kvpart = w.kvpart;
  ap.nsplit = w.ns2;
  ap.split_stride = (size_t)seq * width;
  ap.nkv = nkv;
  ap.dqk = g.head_dim_qk;
  ap.dv = g.head_dim_v;
  ap.rot = g.rot_dim;
  ap.k_norm = L->k_norm;
  ap.eps = g.eps;
  ap.rope = L->rope;
  ap.pos0 = pos_base + cache_len;
  ap.kc = L->k_cache;
  ap.vc = L->v_cache;
  ap.cap = L->cache_cap;
  ap.row0 = cache_len;
  e = launch_small(catchup_append_kernel, ap, dim3(seq), dim3(32 * nkv),
                   sizeof(float) * nkv * g.head_dim_qk, st);
  if (e != cudaSuccess) return cuda_fail(e, "catch-up append launch");
  return MTP_OK;
}

}  // extern "C"
