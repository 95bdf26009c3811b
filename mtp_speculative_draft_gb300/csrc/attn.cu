// Decode attention of the draft layer over its own KV cache, fused with the
// per-head q/k RMSNorm, rotary embedding, KV append, sink logit and the
// sigmoid output gate.
//
// "hf2q 0.1.13 src/inference/models/qwen35/mtp.rs", forward_full_attention
// (apply_q_or_k_per_head_rms_norm, apply_imrope, apply_sdpa_with_kv_cache,
// apply_sigmoid_gate_multiply) and "cortiq-engine 0.8.49 src/mimo_mtp.rs"
// (sliding window, per-head sinks).
//
// Split-K over the cache, at most one CTA per SM.  A CTA serves every query
// row of its KV head (grouped-query sharing of the K/V stream: G heads x m
// new rows).  It owns `nbuf` tile buffers of 16 keys; each buffer is read by
// `qgroups` warps, each of which holds a slice of the query rows.  Warps work
// on their buffer's tiles alone, with no CTA-wide barrier in the loop:
//   * the tile arrives by TMA (K as 128-byte-swizzled boxes of 16 rows x 32
//     floats, V as one bulk copy) and completes on the buffer's mbarrier;
//   * logits with lane = (key, half of the head dims): a lane reads its half
//     of the key row once and keeps one accumulator per query row; query
//     chunks are shared-memory broadcasts; one shuffle adds the halves;
//   * online softmax per query row in the log2 domain (half-warp shuffles);
//   * P.V with lane = output dims; probabilities go through a per-warp row
//     of shared memory and are read back four keys at a time.
// The buffers' states meet once in shared memory and the CTA writes one
// partial.  The m new keys and values are normalised/rotated, appended to the
// cache by the last split and attended to from shared memory.  The splits of
// a KV head then wait (bounded) for each other's partials and each merges a
// slice of whole 32-dim groups: adds the sink to the denominator, applies the
// gate and writes the output as fp32 and packed for the o_proj GEMV.
#include "host.h"

namespace mtp {

constexpr int kTileKeys = 16;  // keys per tile: a half-warp of lanes, one key each
constexpr float kNegBig = -1e30f;
constexpr float kLog2e = 1.4426950408889634f;
#ifndef MTP_ATTN_MAX_WARPS
#define MTP_ATTN_MAX_WARPS 12
#endif
// L2 policy of the cached K/V tiles (tuning knob).  Evict-first: keeping
// the 33.5 MB cache of the 40/8-head, 4096-row layer resident with
// evict-last measured 10 us slower per draft step (it crowds the weights).
#ifndef MTP_ATTN_KV_POLICY
#define MTP_ATTN_KV_POLICY l2_policy_evict_first
#endif
#ifndef MTP_ATTN_MIN_QGROUPS
#define MTP_ATTN_MIN_QGROUPS 1
#endif
constexpr int kAttnMaxWarps = MTP_ATTN_MAX_WARPS;  // warps per CTA (tuning knob)
constexpr int kAttnQMax = 8;                     // query rows per warp (template bound)
constexpr size_t kAttnSmemLimit = 226 * 1024;     // dynamic shared memory of one CTA (227 KB less static)
constexpr size_t kAttnSlack = 1024;               // alignment of the swizzled K boxes
constexpr int kAttnWq = 18;                       // per query row: <= 16 buffer weights, M, l

// Partials: (M, l) pairs [nkv][nsplit][QG][2], then outputs [nkv][nsplit][QG][dv]
// starting on a 16-byte boundary.
__host__ __device__ inline size_t attn_part_o_offset(int nkv, int nsplit, int QG) {
  return ((size_t)nkv * nsplit * QG * 2 + 3) / 4 * 4;
}

__host__ __device__ inline size_t attn_tile_bytes(int dqk, int dv) {
  return (size_t)kTileKeys * (dqk + dv) * 4;  // a multiple of 2 KB (dims are multiples of 32)
}

struct AttnLayout {
  size_t q_off, newk_off, newv_off, ps_off, bar_off, total;
};

// [nbuf tile buffers][query slots qslots x dqk][new keys m x dqk][new values m x dv]
// [probability rows: warps x kAttnQMax x 32][mbarriers].  Query slots: each
// group of query rows owns QM slots; slots past the group's rows hold zeros.
__host__ __device__ inline AttnLayout attn_layout(int dqk, int dv, int qslots, int m, int nbuf,
                                                  int warps) {
  AttnLayout L;
  L.q_off = (size_t)nbuf * attn_tile_bytes(dqk, dv);
  L.newk_off = L.q_off + (size_t)qslots * dqk * 4;
  L.newv_off = L.newk_off + (size_t)m * dqk * 4;
  L.ps_off = L.newv_off + (size_t)m * dv * 4;
  L.bar_off = L.ps_off + (size_t)warps * kAttnQMax * kTileKeys * 4;
  L.total = L.bar_off + (size_t)nbuf * 8;
  return L;
}

// Waits (one thread, bounded) until *cnt >= target; acquire.
__device__ __forceinline__ bool wait_count_cta(const unsigned* cnt, unsigned target,
                                               unsigned polls) {
  for (unsigned i = 0; i < polls; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    __nanosleep(128);
  }
  return false;
}

// Named-barrier AND-reduction over `count` threads (all of them arrive).
__device__ __forceinline__ bool bar_and(bool v, int id, int count) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bar_named(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Retires an mbarrier before its shared memory is reused for other data.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Output dims held by a lane: DV = dv / 32 values, in vectors of VW floats;
// vector c of lane holds dims VW * (lane + 32 c) + [0, VW).
template <int DV>
struct LaneDims {
  static constexpr int VW = DV % 4 == 0 ? 4 : (DV % 2 == 0 ? 2 : 1);
  static constexpr int NV = DV / VW;
  __device__ static int dim(int lane, int c) { return VW * (lane + 32 * c); }
};

template <int DV>
__device__ __forceinline__ void load_dims(const float* row, int lane, float (&v)[DV]) {
  using LD = LaneDims<DV>;
#pragma unroll
  for (int c = 0; c < LD::NV; ++c) {
    const float* p = row + LD::dim(lane, c);
    if constexpr (LD::VW == 4) {
      const float4 t = *reinterpret_cast<const float4*>(p);
      v[4 * c] = t.x; v[4 * c + 1] = t.y; v[4 * c + 2] = t.z; v[4 * c + 3] = t.w;
    } else if constexpr (LD::VW == 2) {
      const float2 t = *reinterpret_cast<const float2*>(p);
      v[2 * c] = t.x; v[2 * c + 1] = t.y;
    } else {
      v[c] = *p;
    }
  }
}

// Running softmax state of one warp for its query rows.
template <int QM, int DV>
struct WarpState {
  float M[QM], l[QM], o[QM][DV];
};

// One tile of nk keys starting at absolute key index key0, for the warp's QM
// query slots (query rows q0 .. q0 + QM - 1; slots past the group's rows are
// zero vectors whose results are never used, so no row is branched on).
// `swz`: K in swizzled boxes (cached tiles), else plain rows of dqk floats
// (the new keys).
template <int QM, int DV>
__device__ __forceinline__ void warp_tile(const AttnParams& a, WarpState<QM, DV>& st,
                                          const float* Ks, bool swz, const float* Vs, int nk,
                                          int key0, const float* qrow, int q0, int G, float* ps,
                                          int lane) {
  const int dqk = a.dqk, dv = a.dv;
  const int kq4 = dqk / 4;
  // ---- logits: lane = (key, half); half h takes the 16-byte chunks 2i + h
  // of every 32-dim block (so the two halves' query broadcasts fall in
  // different banks), and one shuffle adds the halves
  const int key = lane & (kTileKeys - 1), half = lane >> 4;
  float acc[QM];
#pragma unroll
  for (int q = 0; q < QM; ++q) acc[q] = 0.f;
  if (key < nk) {
    // 32-dim blocks: the key's 4 chunks of a block (all loads in flight)
    const int l7 = key & 7;
    for (int bx = 0; bx < kq4 / 8; ++bx) {
      float4 k[4];
      if (swz) {  // box bx: row key, 16-byte chunk c at c ^ (key & 7)
        const float* kb = Ks + bx * (kTileKeys * 32) + key * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          k[i] = *reinterpret_cast<const float4*>(kb + (((2 * i + half) ^ l7) << 2));
      } else {
        const float* kb = Ks + key * dqk + bx * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i] = *reinterpret_cast<const float4*>(kb + 4 * (2 * i + half));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < QM; ++q) {
          const float4 x =
              *reinterpret_cast<const float4*>(qrow + q * dqk + bx * 32 + 4 * (2 * i + half));
          acc[q] = fmaf(x.x, k[i].x, fmaf(x.y, k[i].y, fmaf(x.z, k[i].z, fmaf(x.w, k[i].w, acc[q]))));
        }
    }
  }
#pragma unroll
  for (int q = 0; q < QM; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], 16);
  // ---- online softmax per query row (both halves hold every key's logit:
  // reductions over 16 lanes); probabilities to the warp's rows
  const int j = key0 + key;
#pragma unroll
  for (int q = 0; q < QM; ++q) {
    const int p = a.L + (q0 + q) / G;
    const bool ok = key < nk && j <= p && (a.window <= 0 || j > p - a.window);
    const float l = ok ? acc[q] : kNegBig;
    float mx = l;
#pragma unroll
    for (int o = kTileKeys / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mnew = fmaxf(st.M[q], mx);
    const float pr = ok ? exp2f(l - mnew) : 0.f;
    const float alpha = exp2f(st.M[q] - mnew);
    float sm = pr;
#pragma unroll
    for (int o = kTileKeys / 2; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    st.l[q] = st.l[q] * alpha + sm;
    st.M[q] = mnew;
    if (half == 0) ps[q * kTileKeys + key] = pr;
#pragma unroll
    for (int i = 0; i < DV; ++i) st.o[q][i] *= alpha;
  }
  __syncwarp();
  // ---- P.V: lane = output dims, four keys per step (rows past nk hold p = 0
  // and are read only from the V rows the copy filled)
  int jj = 0;
  for (; jj + 4 <= nk; jj += 4) {
    float v[4][DV];
#pragma unroll
    for (int u = 0; u < 4; ++u) load_dims<DV>(Vs + (size_t)(jj + u) * dv, lane, v[u]);
#pragma unroll
    for (int q = 0; q < QM; ++q) {
      const float4 p4 = *reinterpret_cast<const float4*>(ps + q * kTileKeys + jj);
#pragma unroll
      for (int i = 0; i < DV; ++i)
        st.o[q][i] = fmaf(p4.x, v[0][i],
                          fmaf(p4.y, v[1][i], fmaf(p4.z, v[2][i], fmaf(p4.w, v[3][i], st.o[q][i]))));
    }
  }
  for (; jj < nk; ++jj) {
    float v[DV];
    load_dims<DV>(Vs + (size_t)jj * dv, lane, v);
#pragma unroll
    for (int q = 0; q < QM; ++q) {
      const float p = ps[q * kTileKeys + jj];
#pragma unroll
      for (int i = 0; i < DV; ++i) st.o[q][i] = fmaf(p, v[i], st.o[q][i]);
    }
  }
  __syncwarp();
}

// ------------------------------------------------ tensor-core tile path
// For 128-dim heads and at most 8 query rows per KV head: logits and P.V as
// mma.sync m16n8k8 TF32 products, each operand split into a TF32 "big" part
// and the remainder (three products, the small x small one dropped: about
// 2^-21 relative error per product, float32 accumulation).  One warp owns a
// 16-key tile and all 8 query slots:
//   S^T[key][q] = K . Q^T: M = keys, N = query slots, K = dims, with the dims
//     of k-step (block b, step s) permuted so lane (gid, tq) reads dims
//     32b + 8tq + [0, 8) of key rows gid and gid + 8 (two conflict-free
//     16-byte loads per row from the swizzled K box) and holds the same dims
//     of query slot gid in registers;
//   O^T[dim][q] += V^T . P^T: M = dims with row r of m-tile mt standing for
//     dim 16 (r mod 8) + 2 mt + r / 8, so lane gid's A elements of all eight
//     m-tiles are dims 16 gid + [0, 16) of its two key rows; P goes through
//     the warp's row of shared memory from the logits' layout to the B layout.
// The accumulator layouts of both products put query slots 2tq, 2tq + 1 in
// lane (gid, tq), so the online-softmax rescale needs no data movement.
constexpr int kTcNB = 4;   // 32-dim blocks of the 128-dim q/k heads
constexpr int kTcNMT = 8;  // 16-dim m-tiles of the 128-dim v heads
// unrolling of the tile's dim-block and key-step loops (tuning knob: the
// code size of one tile against the loop overhead)
#ifndef MTP_ATTN_TC_UNROLL
#define MTP_ATTN_TC_UNROLL 1
#endif
constexpr int kTcUnrollB = MTP_ATTN_TC_UNROLL;
constexpr int kTcUnrollK = MTP_ATTN_TC_UNROLL > 2 ? 2 : MTP_ATTN_TC_UNROLL;

__device__ __forceinline__ void tf32_split(float x, uint32_t& big, uint32_t& small) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(big) : "f"(x));
  small = __float_as_uint(x - __uint_as_float(big));  // truncated to TF32 by the tensor core
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d += A B with A = a (four f32 values, split here) and B given split
__device__ __forceinline__ void mma_tf32x3(float (&d)[4], const float (&a)[4], uint32_t bb0,
                                           uint32_t bs0, uint32_t bb1, uint32_t bs1) {
  uint32_t ab[4], as[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) tf32_split(a[i], ab[i], as[i]);
  mma_tf32(d, as, bb0, bb1);
  mma_tf32(d, ab, bs0, bs1);
  mma_tf32(d, ab, bb0, bb1);
}

struct TcState {
  float M[2], l[2];         // query slots 2tq, 2tq + 1
  float o[kTcNMT][4];       // O^T fragments
};

__device__ __forceinline__ void load8(float (&v)[8], const float* p0, const float* p1) {
  const float4 x = *reinterpret_cast<const float4*>(p0);
  const float4 y = *reinterpret_cast<const float4*>(p1);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}

// One tile of nk <= 16 keys from key0 on.  swz: K in swizzled boxes (cached
// tiles), else plain rows of 128 floats (the new keys); V plain rows of 128
// floats.  Rows at or past nk are not read.
__device__ __forceinline__ void warp_tile_tc(const AttnParams& a, TcState& st, const float* Ks,
                                             bool swz, const float* Vs, int nk, int key0,
                                             const float* qrow, int G, int QG, float* ps,
                                             int lane) {
  const int gid = lane >> 2, tq = lane & 3;
  // two accumulators (even and odd dim blocks) halve the dependent MMA chain
  float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll kTcUnrollB
  for (int b = 0; b < kTcNB; ++b) {
    float k0[8], k1[8];  // key rows gid and gid + 8, dims 32b + 8tq + [0, 8)
    if (swz) {
      const float* kb = Ks + b * (kTileKeys * 32);
      const int c0 = ((2 * tq) ^ (gid & 7)) << 2, c1 = ((2 * tq + 1) ^ (gid & 7)) << 2;
      load8(k0, kb + gid * 32 + c0, kb + gid * 32 + c1);
      load8(k1, kb + (gid + 8) * 32 + c0, kb + (gid + 8) * 32 + c1);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) k0[i] = k1[i] = 0.f;
      const int off = 32 * b + 8 * tq;
      if (gid < nk) load8(k0, Ks + gid * 128 + off, Ks + gid * 128 + off + 4);
      if (gid + 8 < nk) load8(k1, Ks + (gid + 8) * 128 + off, Ks + (gid + 8) * 128 + off + 4);
    }
    float q[8];  // query slot gid, the same dims
    load8(q, qrow + gid * 128 + 32 * b + 8 * tq, qrow + gid * 128 + 32 * b + 8 * tq + 4);
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      uint32_t bb0, bs0, bb1, bs1;
      tf32_split(q[2 * s2], bb0, bs0);
      tf32_split(q[2 * s2 + 1], bb1, bs1);
      const float av[4] = {k0[2 * s2], k1[2 * s2], k0[2 * s2 + 1], k1[2 * s2 + 1]};
      mma_tf32x3((b & 1) ? d2 : d, av, bb0, bs0, bb1, bs1);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] += d2[i];
  // online softmax per query slot column (d[2 hh + c]: key gid + 8 hh, slot 2tq + c)
  float p[4], alpha[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int qi = 2 * tq + c;
    const int pos = a.L + qi / G;
    bool ok[2];
    float mx = kNegBig;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int key = gid + 8 * hh, j = key0 + key;
      ok[hh] = qi < QG && key < nk && j <= pos && (a.window <= 0 || j > pos - a.window);
      if (ok[hh]) mx = fmaxf(mx, d[2 * hh + c]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mnew = fmaxf(st.M[c], mx);
    const float p0 = ok[0] ? exp2f(d[c] - mnew) : 0.f;
    const float p1 = ok[1] ? exp2f(d[2 + c] - mnew) : 0.f;
    float sm = p0 + p1;
    sm += __shfl_xor_sync(0xffffffffu, sm, 4);
    sm += __shfl_xor_sync(0xffffffffu, sm, 8);
    sm += __shfl_xor_sync(0xffffffffu, sm, 16);
    alpha[c] = exp2f(st.M[c] - mnew);
    st.l[c] = st.l[c] * alpha[c] + sm;
    st.M[c] = mnew;
    p[c] = p0;
    p[2 + c] = p1;
  }
#pragma unroll
  for (int mt = 0; mt < kTcNMT; ++mt) {
    st.o[mt][0] *= alpha[0];
    st.o[mt][2] *= alpha[0];
    st.o[mt][1] *= alpha[1];
    st.o[mt][3] *= alpha[1];
  }
  // probabilities as [slot][key] in the warp's row of shared memory
  ps[(2 * tq) * kTileKeys + gid] = p[0];
  ps[(2 * tq + 1) * kTileKeys + gid] = p[1];
  ps[(2 * tq) * kTileKeys + gid + 8] = p[2];
  ps[(2 * tq + 1) * kTileKeys + gid + 8] = p[3];
  __syncwarp();
#pragma unroll kTcUnrollK
  for (int ks = 0; ks < 2; ++ks) {
    const int ka = 8 * ks + tq, kb2 = ka + 4;
    uint32_t bb0, bs0, bb1, bs1;
    tf32_split(ps[gid * kTileKeys + ka], bb0, bs0);
    tf32_split(ps[gid * kTileKeys + kb2], bb1, bs1);
    float va[16], vb[16];  // key rows ka, kb2, dims 16 gid + [0, 16) (zero past nk)
#pragma unroll
    for (int i = 0; i < 16; ++i) va[i] = vb[i] = 0.f;
    // swz: dims 16 gid + [0, 16) of key row k sit in box gid / 2, 16-byte
    // chunks 4 (gid & 1) + c4 at position chunk ^ (k & 7) (conflict-free)
    auto vrow = [&](int k, float (&v)[16]) {
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float* src = swz ? Vs + (gid >> 1) * (kTileKeys * 32) + k * 32 +
                                     (((4 * (gid & 1) + c4) ^ (k & 7)) << 2)
                               : Vs + k * 128 + 16 * gid + 4 * c4;
        const float4 x = *reinterpret_cast<const float4*>(src);
        v[4 * c4] = x.x; v[4 * c4 + 1] = x.y; v[4 * c4 + 2] = x.z; v[4 * c4 + 3] = x.w;
      }
    };
    if (ka < nk) vrow(ka, va);
    if (kb2 < nk) vrow(kb2, vb);
#pragma unroll
    for (int mt = 0; mt < kTcNMT; ++mt) {
      const float av[4] = {va[2 * mt], va[2 * mt + 1], vb[2 * mt], vb[2 * mt + 1]};
      mma_tf32x3(st.o[mt], av, bb0, bs0, bb1, bs1);
    }
  }
  __syncwarp();  // the probability row is rewritten by the next tile
}

template <int QM, int DV, bool TC>
__global__ void __launch_bounds__(kAttnMaxWarps * 32, 1)
    attn_decode_kernel(const __grid_constant__ AttnParams a) {
  extern __shared__ __align__(1024) uint8_t smraw_unaligned[];
  // the swizzled K boxes need 1024-byte-aligned buffers
  uint8_t* smraw = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smraw_unaligned) + 1023) & ~uintptr_t(1023));
  using LD = LaneDims<DV>;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nthreads = blockDim.x, nw = nthreads >> 5;
  const int G = a.nh / a.nkv;
  const int QG = G * a.m;
  const int dqk = a.dqk, dv = a.dv;
  const int q_rows = a.nh * dqk * (a.gated ? 2 : 1);
  const int nbuf = a.nbuf, qgroups = a.qgroups;
  const int qpw = (QG + qgroups - 1) / qgroups;      // query rows per warp (<= QM)
  const int qslots = qgroups * QM;
  const AttnLayout Ly = attn_layout(dqk, dv, qslots, a.m, nbuf, nw);
  const size_t tile_bytes = attn_tile_bytes(dqk, dv);
  float* qs = reinterpret_cast<float*>(smraw + Ly.q_off);
  float* newk = reinterpret_cast<float*>(smraw + Ly.newk_off);
  float* newv = reinterpret_cast<float*>(smraw + Ly.newv_off);
  float* ps = reinterpret_cast<float*>(smraw + Ly.ps_off) + (size_t)warp * kAttnQMax * kTileKeys;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smraw + Ly.bar_off);
  __shared__ bool arrived;

  // this warp: buffer b, query rows [q0, q0 + nq) in slots [qgi * QM, qgi * QM + QM)
  const int b = warp / qgroups, qgi = warp % qgroups;
  const int q0 = qgi * qpw;
  const int nq = max(0, min(qpw, QG - q0));
  const float* qrow = nullptr;  // set once the slots are filled
  const bool leader = qgi == 0 && lane == 0;
  float* Kb = reinterpret_cast<float*>(smraw + (size_t)b * tile_bytes);
  float* Vb = Kb + kTileKeys * dqk;

  // cached keys [kbeg, L) in whole tiles per split; the new keys go to the last split
  const int L = a.L;
  const int kbeg = a.window > 0 ? max(0, L + 1 - a.window) : 0;
  const int ntiles = (L - kbeg + kTileKeys - 1) / kTileKeys;
  const int tps = (ntiles + a.nsplit - 1) / a.nsplit;
  const int t_begin = min(ntiles, split * tps);
  const int t_end = min(ntiles, t_begin + tps);
  const float* vbase = a.vc + (size_t)kvh * a.cap * dv;

  if (tid < nbuf) {
    mbar_init(&bars[tid], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const uint64_t pol = MTP_ATTN_KV_POLICY();
  // the buffer's leader lane fills it with tile t (absolute index)
  auto issue = [&](int t) {
    const int key0 = kbeg + t * kTileKeys;
    const int nk = min(kTileKeys, L - key0);
    if constexpr (TC) {  // V in swizzled boxes as well (whole boxes; rows past nk unused)
      mbar_arrive_expect_tx(&bars[b], (uint32_t)kTileKeys * (dqk + dv) * 4);
      for (int bx = 0; bx < dv / 32; ++bx)
        tma_load_2d(Vb + bx * (kTileKeys * 32), &a.vmap, &bars[b], bx * 32, kvh * a.cap + key0, pol);
    } else {
      mbar_arrive_expect_tx(&bars[b], (uint32_t)kTileKeys * dqk * 4 + (uint32_t)nk * dv * 4);
      bulk_load(Vb, vbase + (size_t)key0 * dv, (uint32_t)nk * dv * 4, &bars[b], pol);
    }
    for (int bx = 0; bx < dqk / 32; ++bx)
      tma_load_2d(Kb + bx * (kTileKeys * 32), &a.kmap, &bars[b], bx * 32, kvh * a.cap + key0, pol);
  };
  const int t_first = t_begin + b;
  if (a.prefetch_before_wait && leader && t_first < t_end) issue(t_first);
  pdl_wait();
  pdl_launch_dependents();
  if (!a.prefetch_before_wait && leader && t_first < t_end) issue(t_first);

  // ---- query slots of this KV head: norm, rotate, pre-scale (log2 domain);
  // slots past a group's rows are zeroed
  const float qscale = a.scale * kLog2e;
  for (int sl = warp; sl < qslots; sl += nw) {
    const int g = sl / QM, l = sl - g * QM;
    const int qi = g * qpw + l;
    float* dst = qs + (size_t)sl * dqk;
    if (l < qpw && qi < QG) {
      const int r = qi / G, h = kvh * G + qi % G;
      const float* src = a.qp + (size_t)r * q_rows + (size_t)h * dqk * (a.gated ? 2 : 1);
      warp_norm_rope(dst, src, dqk, a.qn, a.eps, a.rope + (size_t)(a.pos_base + L + r) * a.rot, a.rot, qscale,
                     lane);
    } else {
      for (int i = lane; i < dqk; i += 32) dst[i] = 0.f;
    }
  }
  qrow = qs + (size_t)qgi * QM * dqk;
  // ---- new keys/values (last split): normalise, rotate, append to the cache
  const bool has_new = split == a.nsplit - 1;
  if (has_new) {
    for (int r = warp; r < a.m; r += nw) {
      const int pos = L + r;
      float* kn = newk + r * dqk;
      const float* ksrc = a.kp + (size_t)r * a.nkv * dqk + (size_t)kvh * dqk;
      warp_norm_rope(kn, ksrc, dqk, a.kn, a.eps, a.rope + (size_t)(a.pos_base + pos) * a.rot, a.rot,
                     1.f, lane);
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
  __syncthreads();

  WarpState<QM, DV> st;
  TcState tc;
  if constexpr (TC) {
    tc.M[0] = tc.M[1] = kNegBig;
    tc.l[0] = tc.l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < kTcNMT; ++mt) tc.o[mt][0] = tc.o[mt][1] = tc.o[mt][2] = tc.o[mt][3] = 0.f;
  } else {
#pragma unroll
    for (int q = 0; q < QM; ++q) {
      st.M[q] = kNegBig;
      st.l[q] = 0.f;
#pragma unroll
      for (int i = 0; i < DV; ++i) st.o[q][i] = 0.f;
    }
  }
  // ---- the buffer's tiles: t_first, t_first + nbuf, ...
  const int bar_id = 1 + b, bar_cnt = qgroups * 32;
  bool dead = false;
  uint32_t phase = 0;
  for (int t = t_first; t < t_end; t += nbuf) {
    const bool ok = mbar_wait_bounded(&bars[b], phase);
    __syncwarp();
    if (!bar_and(ok, bar_id, bar_cnt)) {  // the buffer's warps give up together
      if (leader) set_dev_error(a.err, kErrMbarTimeout);
      dead = true;
      break;
    }
    phase ^= 1u;
    const int key0 = kbeg + t * kTileKeys;
    if constexpr (TC)
      warp_tile_tc(a, tc, Kb, true, Vb, min(kTileKeys, L - key0), key0, qrow, G, QG, ps, lane);
    else if (nq > 0)
      warp_tile<QM, DV>(a, st, Kb, true, Vb, min(kTileKeys, L - key0), key0, qrow, q0, G, ps,
                        lane);
    if (t + nbuf < t_end) {
      bar_named(bar_id, bar_cnt);  // every reader of the buffer is done with it
      if (leader) issue(t + nbuf);
    }
  }
  if (has_new && b == nbuf - 1) {
    if constexpr (TC)
      warp_tile_tc(a, tc, newk, false, newv, a.m, L, qrow, G, QG, ps, lane);
    else if (nq > 0)
      warp_tile<QM, DV>(a, st, newk, false, newv, a.m, L, qrow, q0, G, ps, lane);
  }
  if (__syncthreads_or(dead)) return;
  if (tid < nbuf) mbar_inval(&bars[tid]);
  __syncthreads();

  // ---- the buffers' states meet in shared memory (the tile buffers are free)
  float* wstat = reinterpret_cast<float*>(smraw);                 // [nw][QM][2]
  float* wout = wstat + (size_t)kAttnMaxWarps * kAttnQMax * 2;    // [nw][QM][ldw]
  const int ldw = dv + 4;  // padded rows: the tensor-core fragments store with 2-way conflicts at most
  if constexpr (TC) {
    const int gid = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int q = 2 * tq + c;
      if (q < nq && gid == 0) {
        wstat[(warp * QM + q) * 2] = tc.M[c];
        wstat[(warp * QM + q) * 2 + 1] = tc.l[c];
      }
    }
    // slot 2tq + c holds dims 16 gid + [0, 16): fragments (mt, c) and (mt, c + 2)
    // are dims 16 gid + 2 mt and + 1
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int q = 2 * tq + c;
      if (q < nq)
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4)
          *reinterpret_cast<float4*>(wout + ((size_t)warp * QM + q) * ldw + 16 * gid + 4 * j4) =
              make_float4(tc.o[2 * j4][c], tc.o[2 * j4][c + 2], tc.o[2 * j4 + 1][c],
                          tc.o[2 * j4 + 1][c + 2]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < QM; ++q) {
      if (q < nq) {
        if (lane == 0) {
          wstat[(warp * QM + q) * 2] = st.M[q];
          wstat[(warp * QM + q) * 2 + 1] = st.l[q];
        }
#pragma unroll
        for (int c = 0; c < LD::NV; ++c)
#pragma unroll
          for (int e = 0; e < LD::VW; ++e)
            wout[((size_t)warp * QM + q) * ldw + LD::dim(lane, c) + e] = st.o[q][c * LD::VW + e];
      }
    }
  }
  __syncthreads();
  const size_t pidx = (size_t)(kvh * a.nsplit + split) * QG;
  float* part_o = a.part + attn_part_o_offset(a.nkv, a.nsplit, QG);
  // each query row's buffer weights exp2(M_b - M) once (a warp per row,
  // lanes over the buffers), then the weighted sums of the outputs
  float* wq = wout + (size_t)nw * QM * ldw;  // [QG][kAttnWq]: weights, then M and l
  for (int q = warp; q < QG; q += nw) {
    const int g = q / qpw, ql = q - g * qpw;
    const float mb = lane < nbuf ? wstat[((lane * qgroups + g) * QM + ql) * 2] : kNegBig;
    const float lb = lane < nbuf ? wstat[((lane * qgroups + g) * QM + ql) * 2 + 1] : 0.f;
    const float M = warp_max(mb);
    const float f = lane < nbuf ? exp2f(mb - M) : 0.f;
    const float l = warp_sum(f * lb);
    if (lane < nbuf) wq[q * kAttnWq + lane] = f;
    if (lane == 0) {
      wq[q * kAttnWq + kAttnWq - 2] = M;
      wq[q * kAttnWq + kAttnWq - 1] = l;
    }
  }
  __syncthreads();
  for (int it = tid; it < QG * dv; it += nthreads) {
    const int q = it / dv, d = it - q * dv;
    const int g = q / qpw, ql = q - g * qpw;
    const float* fq = wq + q * kAttnWq;
    const float* src = wout + (size_t)(g * QM + ql) * ldw + d;  // buffer bb at + bb * bstride
    const size_t bstride = (size_t)qgroups * QM * ldw;
    float o0 = 0.f, o1 = 0.f;
    int bb = 0;
    for (; bb + 2 <= nbuf; bb += 2) {  // two independent chains
      o0 = fmaf(fq[bb], src[bb * bstride], o0);
      o1 = fmaf(fq[bb + 1], src[(bb + 1) * bstride], o1);
    }
    if (bb < nbuf) o0 = fmaf(fq[bb], src[bb * bstride], o0);
    part_o[(pidx + q) * dv + d] = o0 + o1;
    if (d == 0) {
      a.part[(pidx + q) * 2 + 0] = fq[kAttnWq - 2];
      a.part[(pidx + q) * 2 + 1] = fq[kAttnWq - 1];
    }
  }
  // ---- all splits of this KV head publish their partials, then each merges
  // one slice of the head's output (whole 32-dim groups, for the packed copy)
  const int ns = a.nsplit;
  if (!a.merge_in_kernel) return;  // the next launch merges the partials
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    atomicAdd(&a.counters[kvh], 1u);
    arrived = wait_count_cta(&a.counters[kvh], (unsigned)ns, wait_polls(a.err, 4u << 20));
    if (!arrived) set_dev_error(a.err, kErrSplitTimeout);
  }
  __syncthreads();
  if (!arrived) return;
  const size_t base = (size_t)kvh * ns * QG;
  const int gpq = dv / kGroup;                 // 32-dim groups per query row
  const int ngroups = QG * gpq;
  const int g0 = split * ngroups / ns, g1 = (split + 1) * ngroups / ns;
  const int nit = (g1 - g0) * 8;               // float4 items of the slice
  // smem: split weights [ns][QG], denominators [ns][QG], partial outputs of
  // the slice [ns][nit] float4, merged slice [nit] float4 (tile buffers are free)
  float* wsm = reinterpret_cast<float*>(smraw);
  float* lsm = wsm + ns * QG;
  float4* osm = reinterpret_cast<float4*>(smraw + (((size_t)2 * ns * QG * 4 + 15) / 16) * 16);
  float4* fsm = osm + (size_t)ns * nit;
  // one round trip: (M, l) pairs and the slice's partials, all loads in flight
  for (int i2 = tid; i2 < ns * QG; i2 += nthreads) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part) + base + i2);
    wsm[i2] = ml.x;
    lsm[i2] = ml.y;
  }
  for (int i2 = tid; i2 < ns * nit; i2 += nthreads) {
    const int sp2 = i2 / nit, it = i2 - sp2 * nit;
    const int gg = g0 + it / 8;                // group of the head's output
    const int qi = gg / gpq, d4 = (gg - qi * gpq) * 8 + (it & 7);
    osm[i2] = __ldcg(reinterpret_cast<const float4*>(part_o + ((size_t)(kvh * ns + sp2) * QG + qi) * dv) + d4);
  }
  __syncthreads();
  // split weights of the slice's rows: one warp per row, lanes over the splits
  const int q_lo = (g0 * kGroup) / dv, q_hi = g1 > g0 ? ((g1 - 1) * kGroup) / dv : q_lo - 1;
  for (int q = q_lo + warp; q <= q_hi; q += nw) {
    const int h = kvh * G + q % G;
    const float sinkl2 = a.sinks ? a.sinks[h] * kLog2e : kNegBig;
    float M = sinkl2;
    for (int s2 = lane; s2 < ns; s2 += 32) M = fmaxf(M, wsm[s2 * QG + q]);
    M = warp_max(M);
    float den = 0.f;
    for (int s2 = lane; s2 < ns; s2 += 32) den += exp2f(wsm[s2 * QG + q] - M) * lsm[s2 * QG + q];
    den = warp_sum(den) + (a.sinks ? exp2f(sinkl2 - M) : 0.f);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __syncwarp();
    for (int s2 = lane; s2 < ns; s2 += 32) wsm[s2 * QG + q] = exp2f(wsm[s2 * QG + q] - M) * inv;
  }
  __syncthreads();
  for (int it = tid; it < nit; it += nthreads) {
    const int gg = g0 + it / 8;
    const int qi = gg / gpq, d4 = (gg - qi * gpq) * 8 + (it & 7);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s2 = 0; s2 < ns; ++s2) {  // k order: deterministic
      const float w = wsm[s2 * QG + qi];
      const float4 v = osm[s2 * nit + it];
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (a.gated) {
      const int r = qi / G, h = kvh * G + qi % G;
      const float4 g = *reinterpret_cast<const float4*>(a.qp + (size_t)r * q_rows +
                                                        (size_t)h * dqk * 2 + dqk + d4 * 4);
      acc.x = acc.x / (1.f + __expf(-g.x));
      acc.y = acc.y / (1.f + __expf(-g.y));
      acc.z = acc.z / (1.f + __expf(-g.z));
      acc.w = acc.w / (1.f + __expf(-g.w));
    }
    fsm[it] = acc;
  }
  __syncthreads();
  // fp32 output and packed copy: octets (two float4 items) of the slice
  const int noct = nit / 2;
  for (int o0 = 0; o0 < noct; o0 += nthreads) {
    const int oi = o0 + tid;
    const bool valid = oi < noct;
    int r = 0, k = 0;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) {
      const int gg = g0 + oi / 4;
      const int qi = gg / gpq;
      r = qi / G;
      const int h = kvh * G + qi % G;
      k = h * dv + (gg - qi * gpq) * kGroup + (oi & 3) * 8;
      const float4 v0 = fsm[2 * oi], v1 = fsm[2 * oi + 1];
      v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
      v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
      if (a.out) {
        float4* dst = reinterpret_cast<float4*>(a.out + (size_t)r * a.nh * dv + k);
        dst[0] = v0;
        dst[1] = v1;
      }
    }
    if (a.out_xp) {
      // the four octets of a group are adjacent lanes (groups start at multiples of 4)
      uint4 hi, lo;
      const float2 gx = pack8_group(v, valid, hi, lo);
      if (valid) {
        const int g = k / kGroup, t = (k % kGroup) / 8;
        a.out_xp[xp_index(g, r, t, 0, a.m)] = hi;
        a.out_xp[xp_index(g, r, t, 1, a.m)] = lo;
        if ((oi & 3) == 0) a.out_xs[g * a.m + r] = gx;
      }
    }
  }
  // leave the counters cleared once every split has read the arrivals
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.counters[a.nkv + kvh], 1u);
    if (prev == (unsigned)ns - 1) {
      a.counters[kvh] = 0u;
      a.counters[a.nkv + kvh] = 0u;
    }
  }
}

// ------------------------------------------------------------------ host side
static int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Upper bound of the split count for `cached` keys in the window (sizes the
// partials); attn_splits never exceeds it and it grows with `cached`.  At
// most one CTA per SM: the splits of a KV head wait for each other.
int attn_splits_bound(int nkv, int cached) {
  const int ntiles = ceil_div(cached, kTileKeys);
  int ns = sm_count() / nkv;
  if (ns > ntiles) ns = ntiles;
  return ns < 1 ? 1 : ns;
}

// Splits: as many as the SMs allow (one CTA per SM), but never fewer tiles
// per split than a CTA has buffers while that still leaves a quarter of the
// SMs a CTA: the MoE layer's 2048-key cache of 256-dim heads (6 buffers per
// CTA) then takes 22 splits per KV head instead of 64, and the next launch
// merges 22 partials (measured -1.9 us per step); short caches (a 128-key
// window, a 64-key cache) keep one tile per split, which measured faster.
static void attn_groups(int QG, int dqk, int dv, int* qgroups, int* qm);
int attn_splits(int nkv, int cached, int QG, int dqk, int dv, int m) {
  const int ntiles = ceil_div(cached, kTileKeys);
  const int bound = attn_splits_bound(nkv, cached);
  if (ntiles == 0) return 1;
  int tps = ceil_div(ntiles, bound);
  int qg = 0, qm = 0;
  attn_groups(QG, dqk, dv, &qg, &qm);
  int nb = std::min(kAttnMaxWarps / qg, 15);
  while (nb > 1 && attn_layout(dqk, dv, qg * qm, m, nb, nb * qg).total + kAttnSlack > kAttnSmemLimit)
    --nb;
  // one tile per buffer while that still gives a quarter of the SMs a CTA
  if (tps < nb && ceil_div(ntiles, nb) * nkv >= sm_count() / 4) tps = nb;
  return ceil_div(ntiles, tps);  // no split without cached tiles
}

const float* attn_part_outputs(const float* part, int nkv, int nsplit, int q_per_kv) {
  return part + attn_part_o_offset(nkv, nsplit, q_per_kv);
}

size_t attn_part_bytes(int nkv, int nsplit, int q_per_kv, int dv) {
  return (attn_part_o_offset(nkv, nsplit, q_per_kv) + (size_t)nkv * nsplit * q_per_kv * dv) *
         sizeof(float);
}

// Query rows per warp (the kernel's template bound): at most kAttnQMax and
// at most 32 state floats per lane.
static int attn_qmax(int dv) { return dv <= 128 ? kAttnQMax : 4; }

// Query groups per buffer and the slots per group (the kernel's QM: the
// smallest instantiated size that holds a group's rows).
// The tensor-core tile path: 128-dim q/k and v heads, at most 8 query rows
// per KV head (one warp holds all of them as the MMA's 8 columns).
#ifndef MTP_ATTN_TC
#define MTP_ATTN_TC 1
#endif
static bool attn_use_tc(int QG, int dqk, int dv) {
  return MTP_ATTN_TC && dqk == 128 && dv == 128 && QG <= 8;
}

static void attn_groups(int QG, int dv, int* qgroups, int* qm) {
  *qgroups = ceil_div(QG, attn_qmax(dv));
  // more warps per buffer (fewer rows each) shorten the per-tile chains
  if (*qgroups < MTP_ATTN_MIN_QGROUPS) *qgroups = MTP_ATTN_MIN_QGROUPS < QG ? MTP_ATTN_MIN_QGROUPS : QG;
  const int qpw = ceil_div(QG, *qgroups);
  *qm = qpw <= 2 ? 2 : qpw <= 4 ? 4 : qpw <= 6 ? 6 : 8;
}
static void attn_groups(int QG, int dqk, int dv, int* qgroups, int* qm) {
  if (attn_use_tc(QG, dqk, dv)) {
    *qgroups = 1;
    *qm = 8;
    return;
  }
  attn_groups(QG, dv, qgroups, qm);
}

bool attn_supported(int QG, int dqk, int dv, int m) {
  int qg, qm;
  attn_groups(QG, dqk, dv, &qg, &qm);
  if (qg > kAttnMaxWarps) return false;
  const AttnLayout Ly = attn_layout(dqk, dv, qg * qm, m, 1, qg);
  return Ly.total + kAttnSlack <= kAttnSmemLimit;
}

template <int QM, int DV, bool TC = false>
static cudaError_t launch_attn_t(const AttnParams& a, size_t smem, cudaStream_t st) {
  static_assert(sizeof(AttnParams) <= 4096, "kernel parameters fit the classic limit");
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<QM, DV, TC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kAttnSmemLimit);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.nkv);
  cfg.blockDim = dim3(a.nbuf * a.qgroups * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<QM, DV, TC>, a);
}

template <int DV>
static cudaError_t launch_attn_qm(const AttnParams& a, int qm, size_t smem, cudaStream_t st) {
  switch (qm) {
    case 2: return launch_attn_t<2, DV>(a, smem, st);
    case 4: return launch_attn_t<4, DV>(a, smem, st);
    case 6: if constexpr (DV <= 4) return launch_attn_t<6, DV>(a, smem, st); else break;
    case 8: if constexpr (DV <= 4) return launch_attn_t<8, DV>(a, smem, st); else break;
    default: break;
  }
  return cudaErrorInvalidValue;
}

// Slots per query group: up to 8 for head_dim_v <= 128, else 4 (at most 32
// state floats per lane).
static cudaError_t launch_attn_dv(const AttnParams& a, int qm, size_t smem, cudaStream_t st) {
  switch (a.dv / 32) {
    case 1: return launch_attn_qm<1>(a, qm, smem, st);
    case 2: return launch_attn_qm<2>(a, qm, smem, st);
    case 3: return launch_attn_qm<3>(a, qm, smem, st);
    case 4: return launch_attn_qm<4>(a, qm, smem, st);
    case 5: return launch_attn_qm<5>(a, qm, smem, st);
    case 6: return launch_attn_qm<6>(a, qm, smem, st);
    case 7: return launch_attn_qm<7>(a, qm, smem, st);
    case 8: return launch_attn_qm<8>(a, qm, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn(const AttnParams& a_in, cudaStream_t st) {
  AttnParams a = a_in;
  cudaError_t ke =
      encode_f32_tile_map(&a.kmap, a.kc, (uint64_t)a.nkv * a.cap, (uint64_t)a.dqk, kTileKeys);
  if (ke == cudaSuccess && attn_use_tc((a.nh / a.nkv) * a.m, a.dqk, a.dv))
    ke = encode_f32_tile_map(&a.vmap, a.vc, (uint64_t)a.nkv * a.cap, (uint64_t)a.dv, kTileKeys);
  if (ke != cudaSuccess) return ke;
  const int QG = (a.nh / a.nkv) * a.m;
  // warps per buffer: the fewest that keep each warp within attn_qmax rows
  int qm = 0;
  attn_groups(QG, a.dqk, a.dv, &a.qgroups, &qm);
  const int qslots = a.qgroups * qm;
  // buffers: as many as the split has tiles, within the warp and smem limits
  const int kbeg = a.window > 0 ? (a.L + 1 - a.window > 0 ? a.L + 1 - a.window : 0) : 0;
  const int ntiles = ceil_div(a.L - kbeg, kTileKeys);
  const int tps = ntiles > 0 ? ceil_div(ntiles, a.nsplit) : 1;
  int nbuf = tps;
  // at least one warp per query slot and new row for the prologue (its norm
  // and rotation are a dependent round trip per row), within the warp limit
#ifndef MTP_ATTN_PROLOGUE_WARPS
#define MTP_ATTN_PROLOGUE_WARPS 1
#endif
  if (MTP_ATTN_PROLOGUE_WARPS) {
    const int want = std::min(kAttnMaxWarps, qslots + a.m);
    if (nbuf * a.qgroups < want) nbuf = std::max(nbuf, want / a.qgroups);
  }
  if (nbuf > kAttnMaxWarps / a.qgroups) nbuf = kAttnMaxWarps / a.qgroups;
  if (nbuf > 15) nbuf = 15;  // named barriers 1..15 (0 is the CTA barrier)
  while (nbuf > 1 &&
         attn_layout(a.dqk, a.dv, qslots, a.m, nbuf, nbuf * a.qgroups).total + kAttnSlack >
             kAttnSmemLimit)
    --nbuf;
  if (nbuf < 1) nbuf = 1;
  a.nbuf = nbuf;
  const int nw = nbuf * a.qgroups;
  const AttnLayout Ly = attn_layout(a.dqk, a.dv, qslots, a.m, nbuf, nw);
  // the tile buffers are reused for the buffers' states, then the merge
  const size_t combine =
      ((size_t)kAttnMaxWarps * kAttnQMax * 2 + (size_t)nw * qm * (a.dv + 4) + (size_t)QG * kAttnWq) * 4;
  // the merge of one split: weights and denominators [ns][QG], its slice's
  // partials [ns][items] and merged items (float4 items, 8 per 32-dim group)
  const int ngroups = QG * a.dv / kGroup;
  const size_t items = (size_t)ceil_div(ngroups, a.nsplit) * 8;
  const size_t merge = ((size_t)2 * a.nsplit * QG * 4 + 15) / 16 * 16 + (a.nsplit + 1) * items * 16;
  size_t smem = Ly.total;
  if (combine > smem) smem = combine;
  if (merge > smem) smem = merge;
  smem += kAttnSlack;
  if (smem > kAttnSmemLimit) return cudaErrorInvalidValue;
  if (attn_use_tc(QG, a.dqk, a.dv)) return launch_attn_t<8, 4, true>(a, smem, st);
  return launch_attn_dv(a, qm, smem, st);
}

}  // namespace mtp
