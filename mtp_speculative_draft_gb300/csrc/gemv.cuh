// Affine 4-bit group-32 skinny GEMM y[m][N] = x[m][K] . W^T for m <= 16.
//
// Weight format ("hf2q 0.1.1 src/serve/forward_mlx_shared.rs", MlxAffineExtra):
// codes uint32 [N][K/8] (column 8j+i in bits 4i..4i+3 of word j), float32
// scales/biases [N][K/32], w = s*code + b.
//
// Design (GB300): the layer is HBM-bound (0.75 byte per weight), so the
// kernel is a persistent weight stream.  Every warp owns a private TMA
// pipeline of S stages; a stage is a 32-row x 256-column slab of one
// matrix: 4 KB of codes (128-byte swizzled tile) plus 1 KB of scales and
// 1 KB of biases.  Codes go shared -> registers with ldmatrix, which hands
// lane (g, t) word t of a group for rows g and g+8 -- exactly the
// m16n8k16 A-fragment slots once the k order inside a group is permuted.
// Codes become f16x2 registers with one mask (LOP3) each and no shift for
// two of the four nibble pairs of a word: kept in place with a zero exponent
// field they are exact subnormal halves, c * 2^-24 (bits 0-3/16-19) and
// 16c * 2^-24 (bits 4-7/20-23), so the tensor pipe accumulates
// 2^-24 * sum(code * x) with no offset term.  The activations are split into
// f16 hi + lo parts (about 22 bits), the slots that meet a 16c code carry
// x/16, and the products run on the tensor pipe with f32 accumulation.  The
// per-group scale and bias are applied in f32 after each group, with the
// group sums pre-scaled by 2^-24:  y' += s * D' + b * 2^-24 sum(x), and the
// finished tile is multiplied by 2^24 (exact).
// Activations arrive pre-packed ("xpack") in the B-fragment order with the
// per-group sums precomputed by the producer kernel.
#pragma once

#include "common.cuh"

namespace mtp {

// ------------------------------------------------------------------ xpack
// For activations X[m][K]: xp is uint4 [G8][m][4][2] and xs float2 [G8][m]
// (G8 = K/32 rounded up to whole stages of 8 groups).  Entry (g, c, t, hl):
// hl = 0 holds the f16 "hi" parts, 1 the "lo" parts, of the eight values
// x[c][32g + 8t + p] as f16x2 words (first element in the low half):
//   word 0: (p0, p4)   word 1: (p1/16, p5/16)   word 2: (p2, p6)   word 3: (p3/16, p7/16)
// xs[g][c] = (2^-24 * sum of the represented x over the group, 2^e): the
// sum meets the bias b at the scale of the tensor-core sums (see above), and
// the parts hold x * 2^-e, with e = 0 while the group's largest |x| is below
// 2^15, else the e that brings it into [2^14, 2^15).  The consumer multiplies
// the group's weight scale by 2^e, so any finite activation is represented
// (to the split's 22 bits; elements more than 2^-100 below their group's
// largest may flush to zero).
__host__ __device__ inline int xpack_groups(int K) { return (K / kGroup + 7) / 8 * 8; }
__host__ __device__ inline size_t xpack_xs_offset(int m, int K) {
  return (size_t)xpack_groups(K) * m * 128;
}
// Buffers hold whole stages of 8 groups; groups past K/32 are read by the
// GEMV (with zero weights) and must hold finite values (they start zeroed).
__host__ __device__ inline size_t xpack_bytes(int m, int K) {
  return xpack_xs_offset(m, K) + (size_t)xpack_groups(K) * m * 8;
}
__device__ __forceinline__ int xp_index(int g, int c, int t, int hl, int m) {
  return ((g * m + c) * 4 + t) * 2 + hl;
}

// f32 -> (hi, lo) f16 split; returns hi + lo as f32.
__device__ __forceinline__ float split_f16(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  const float h = __half2float(hi);
  lo = __float2half_rn(x - h);
  return h + __half2float(lo);
}

// Power-of-two scale 2^e of a group whose largest |x| is amax: 1 below 2^15
// (and for inf or NaN, which then propagate), else amax * 2^-e in [2^14, 2^15).
__device__ __forceinline__ float xpack_group_scale(float amax) {
  if (!(amax >= 32768.f) || isinf(amax)) return 1.f;
  const unsigned ex = (__float_as_uint(amax) >> 23) & 0xffu;  // biased exponent, >= 142
  return __uint_as_float((ex - 14u) << 23);
}
// 1 / s for a power of two s in [1, 2^113] (exact).
__device__ __forceinline__ float pow2_inverse(float s) {
  return __uint_as_float((254u << 23) - __float_as_uint(s));
}

// Packs the eight values of (g, c, t) times inv (the group's 2^-e); returns
// their contribution to the group's sum (2^-24 * represented x).
__device__ __forceinline__ float pack8(const float v[8], float inv, float scale, uint4& hi,
                                       uint4& lo) {
  __half h[8], l[8];
  float sa = 0.f, sb = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool bslot = (i & 1) != 0;  // elements 1, 3, 5, 7 meet a 16*code
    const float r = split_f16((bslot ? v[i] * 0.0625f : v[i]) * inv, h[i], l[i]);
    if (bslot) sb += r; else sa += r;
  }
  auto pk = [](__half a, __half b) -> uint32_t {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
  };
  hi = make_uint4(pk(h[0], h[4]), pk(h[1], h[5]), pk(h[2], h[6]), pk(h[3], h[7]));
  lo = make_uint4(pk(l[0], l[4]), pk(l[1], l[5]), pk(l[2], l[6]), pk(l[3], l[7]));
  return (sa + 16.f * sb) * scale * kCodeUnscale;
}

// One octet of a group held by four adjacent lanes (octet t in lane t of the
// four); every lane of the warp calls it (valid = false: no octet, v unused).
// Packs the octet with the group's scale and returns the group's xs entry.
__device__ __forceinline__ float2 pack8_group(const float v[8], bool valid, uint4& hi, uint4& lo) {
  float amax = 0.f;
  if (valid)
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float sc = xpack_group_scale(amax);
  float sum = valid ? pack8(v, pow2_inverse(sc), sc, hi, lo) : 0.f;
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  return make_float2(sum, sc);
}

// Stores element p (0..7) of an (g, c, t) octet times inv (the group's
// 2^-e): word p % 4, half p / 4.  Returns its contribution to the group's
// sum (2^-24 * represented x).
__device__ __forceinline__ float xp_store_elem(uint4* xp, int m, int g, int c, int t, int p,
                                               float v, float inv, float scale) {
  const bool bslot = (p & 1) != 0;
  __half h, l;
  const float r = split_f16((bslot ? v * 0.0625f : v) * inv, h, l);
  unsigned short* base = reinterpret_cast<unsigned short*>(xp);
  const size_t w_hi = (size_t)xp_index(g, c, t, 0, m) * 8 + (p & 3) * 2 + (p >> 2);
  const size_t w_lo = (size_t)xp_index(g, c, t, 1, m) * 8 + (p & 3) * 2 + (p >> 2);
  base[w_hi] = __half_as_ushort(h);
  base[w_lo] = __half_as_ushort(l);
  return (bslot ? 16.f * r : r) * scale * kCodeUnscale;
}

// A group held one element per lane (element `lane`, v = 0 where store is
// false); every lane of the warp calls it.  Returns the group's xs entry.
__device__ __forceinline__ float2 xp_store_group(uint4* xp, int m, int g, int c, int lane,
                                                 float v, bool store = true) {
  float amax = store ? fabsf(v) : 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = xpack_group_scale(amax);
  float sum = store ? xp_store_elem(xp, m, g, c, lane >> 3, lane & 7, v, pow2_inverse(sc), sc) : 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  return make_float2(sum, sc);
}

// ------------------------------------------------------------------ params
struct alignas(64) QMat {
  CUtensorMap q;  // uint32 [rows][K/8], box 32 x 32 words, 128B swizzle
  CUtensorMap s;  // float  [rows][K/32], box 32 x 8
  CUtensorMap b;  // float  [rows][K/32], box 32 x 8
};

struct GemvSeg {
  int tile_end;     // cumulative tile count (exclusive) up to and including this segment
  int n;            // rows of the segment (stores are guarded by row < n)
  int mat;          // matrix slot (two-matrix epilogues use mat and mat + 1)
  int sel_idx;      // >= 0: row offset = rowsel[sel_idx] * row_mult
  int row_mult;
  int w_idx;        // >= 0: SwiGLU output scaled by segw[w_idx]
  int out_col0;     // column offset of this segment in the output
  int ld;           // leading dimension of out / res
  float* out;       // fp32 output (may be null for pack-only epilogues)
  const float* res; // residual added before the store, or null
};

enum : int { kEpiStore = 0, kEpiSwiglu = 1, kEpiArgmax = 2 };

constexpr int kMaxSeg = 10;

struct GemvParams {
  QMat mat[4];
  const uint4* xp;
  const float2* xs;
  int m;
  int K;                 // reduction length (concatenated length in K-segment mode)
  int nseg;
  GemvSeg seg[kMaxSeg];
  const int* rowsel;     // routed expert ids (device), or null
  const float* segw;     // routed weights (device), or null
  int rowsel_after_wait; // 1: rowsel is produced by the previous kernel
  int epi;               // one-row kernel: kEpiStore / kEpiSwiglu / kEpiArgmax
  int sbf_mask;          // one-row kernel: bit i set when slot i's scales/biases are bfloat16
  int um;                // one-row kernel: 2 when gate (mat) and up (mat + 1) are separate units
  int wq;                // one-row kernel: warps gw < wq take units gw, gw + wq, ... (same count each)
  // K-segment mode (MoE down projection): K = nkseg * kseg_len
  int kseg_len;          // 0: off
  int nkseg;
  int kseg_row_mult;
  int kseg_last_mat;     // < 0: every K segment is routed; else the last one reads this slot
  // SwiGLU pack target
  uint4* out_xp;
  float2* out_xs;
  int out_m;
  // argmax
  unsigned long long* am_partial;  // [gridDim.x]
  unsigned* am_counter;
  int* am_token;
  float* am_value;
  float* logits;                    // optional fp32 logits
  // split-K over units of `spu` stages: partial fragments and per-tile counters
  int ksplit;
  int spu;
  float* part;
  unsigned* tile_cnt;
  int* err;
  // RMSNorm folded into the projection: the input rows x' = u * w are packed
  // unnormalised and the outputs of row c are scaled by
  // r[c] = rsqrt(sum_{i < in_ss_n} in_ss[i * m + c] / in_ss_dim + in_ss_eps).
  const float* in_ss;    // per-tile sums of u^2 written by the producer, or null
  int in_ss_n;
  int in_ss_dim;
  float in_ss_eps;
  // Store epilogue (one segment): also packs rows c >= pack_c0 of the stored
  // value v, times pack_w[row], into out_xp/out_xs (column c - pack_c0 of
  // out_m) and writes the tile's sum of v^2 per packed row to ss_out[tile * out_m + c'].
  const float* pack_w;
  int pack_c0;
  float* ss_out;
  // Argmax epilogue: tiles t < K / 32 also write normed_out[k] = normed_src[k] * r[0] * normed_w[k]
  // for k in [32 t, 32 t + 32)
  const float* normed_src;
  const float* normed_w;
  float* normed_out;
};

// Sum over i < n of part[i * m + c], taken by the whole warp in a fixed order
// (every lane gets the same value).
__device__ __forceinline__ float warp_col_sum(const float* part, int n, int m, int c) {
  float s = 0.f;
  for (int i = threadIdx.x & 31; i < n; i += 32) s += __ldcg(part + (size_t)i * m + c);
  return warp_sum(s);
}

constexpr int kStageMatBytes = 6144;  // 4 KB codes + 1 KB scales + 1 KB biases
// Warps per GEMV CTA (compile-time tuning knob).
#ifndef MTP_GEMV_WARPS
#define MTP_GEMV_WARPS 4
#endif
constexpr int kGemvWarps = MTP_GEMV_WARPS;
constexpr int kXChunk = 1088;         // staged activations per column: 8 groups x (128 + 8) bytes

// Bytes of staged activations per stage, padded so every tensor-map
// destination stays 128-byte aligned.
template <int XM>
__host__ __device__ constexpr int gemv_xchunk_bytes() {
  return (XM * kXChunk + 127) / 128 * 128;
}
// Per-stage shared-memory footprint: NMAT weight slabs plus, when XM > 0, the
// activation fragments of the stage's 8 groups for up to XM columns.
template <int NMAT, int XM>
__host__ __device__ constexpr int gemv_stage_bytes() {
  return NMAT * kStageMatBytes + gemv_xchunk_bytes<XM>();
}
template <int NMAT, int S, int XM>
__host__ __device__ constexpr int gemv_smem_bytes() {
  return kGemvWarps * S * gemv_stage_bytes<NMAT, XM>() + 2048;  // + barriers + alignment slack
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ float argmax_key_value(unsigned long long k) {
  uint32_t u = (uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu));
}

__device__ __forceinline__ int find_seg(const GemvParams& p, int tile) {
  int s = 0;
#pragma unroll 1
  while (s < p.nseg - 1 && tile >= p.seg[s].tile_end) ++s;
  return s;
}

// Position of a warp in its sequence of work units.  A unit is (tile,
// k-chunk): 32 output rows over stages [ks, ke) of the reduction.  The
// segment, matrix slot and first weight row of the unit are resolved once
// when the unit starts, so advancing by a stage costs a compare.
struct Cursor {
  int u, ks, ke, tile, seg, mat, row, mi;
  // um = 2 when a tile's gate and up matrices are separate units (SwiGLU)
  __device__ __forceinline__ void start(const GemvParams& p, int u0, int units, int ksplit,
                                        int spu, int KS, int um = 1) {
    u = u0;
    if (u < units) {
      tile = u / (um * ksplit);
      const int rem = u - tile * (um * ksplit);
      mi = rem / ksplit;
      const int kc = rem - mi * ksplit;
      ks = kc * spu;
      ke = min(KS, ks + spu);
      seg = find_seg(p, tile);
      const GemvSeg& sg = p.seg[seg];
      const int lt = tile - (seg ? p.seg[seg - 1].tile_end : 0);
      mat = sg.mat + mi;
      row = (sg.sel_idx >= 0 ? p.rowsel[sg.sel_idx] * sg.row_mult : 0) + lt * 32;
    }
  }
  // returns true when the unit just finished
  __device__ __forceinline__ bool advance(const GemvParams& p, int W, int units, int ksplit,
                                          int spu, int KS, int um = 1) {
    if (++ks < ke) return false;
    start(p, u + W, units, ksplit, spu, KS, um);
    return true;
  }
  // weight coordinates of the current stage (GS groups of 32 columns per stage)
  template <int GS = 8>
  __device__ __forceinline__ void coords(const GemvParams& p, int& m_out, int& r_out, int& kx,
                                         int& sx) const {
    if (p.kseg_len > 0) {
      const int spk = p.kseg_len / (GS * kGroup);
      const int kj = ks / spk;
      const int kin = ks - kj * spk;
      const int lt = row;  // row holds lt * 32 in this mode (no sel on the segment)
      if (p.kseg_last_mat < 0 || kj < p.nkseg - 1) {
        m_out = mat;
        r_out = p.rowsel[kj] * p.kseg_row_mult + lt;
      } else {
        m_out = p.kseg_last_mat;
        r_out = lt;
      }
      kx = kin * GS * 4;
      sx = kin * GS;
    } else {
      m_out = mat;
      r_out = row;
      kx = ks * GS * 4;
      sx = ks * GS;
    }
  }
};

// ------------------------------------------------------------ shared parts
// Accumulator fragments of one weight matrix: [row tile rt][column tile nt][e],
// e = 0: (row gid, column 2tq), 1: (gid, 2tq + 1), 2: (gid + 8, 2tq), 3: (gid + 8, 2tq + 1)
// of the m16n8 tile; rows are output rows, columns activation rows.

// Per-lane output scales of a folded input RMSNorm for the activation rows
// this lane's fragments hold (column c = nt*8 + 2tq + e); with `one_row`
// every fragment holds activation row 0.
template <int NT>
__device__ __forceinline__ void row_scales(const GemvParams& p, int m, int tq, bool one_row,
                                           float (&rsc)[NT][2]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) rsc[nt][0] = rsc[nt][1] = 1.f;
  if (!p.in_ss) return;
  for (int c = 0; c < m; ++c) {
    const float ss = warp_col_sum(p.in_ss, p.in_ss_n, m, c);
    const float r = rsqrtf(ss / (float)p.in_ss_dim + p.in_ss_eps);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (one_row || nt * 8 + 2 * tq + e == c) rsc[nt][e] = r;
  }
}

// Deterministic split-K (and SwiGLU gate/up pairing): the unit stores its
// NACC-float fragment partial and clears `acc`; the last of the tile's
// um * ksplit units to finish sums the partials in k order into fin[um] and
// returns true.
template <int NACC, int UMAX>
__device__ __forceinline__ bool splitk_finish(const GemvParams& p, int unit, int tile, int um,
                                              int ksplit, float* acc, float (&fin)[UMAX][NACC],
                                              int lane) {
  float4* mine = reinterpret_cast<float4*>(p.part) + ((size_t)unit * 32 + lane) * (NACC / 4);
#pragma unroll
  for (int q = 0; q < NACC / 4; ++q)
    mine[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  __threadfence();
  __syncwarp();
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(p.tile_cnt + tile, 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
#pragma unroll
  for (int q = 0; q < NACC; ++q) acc[q] = 0.f;
  if (prev != (unsigned)(um * ksplit) - 1) return false;
  __threadfence();
  // k order is fixed (deterministic); loads of four partials are issued
  // together so their L2 latencies overlap
  const size_t pstride = (size_t)32 * (NACC / 4);
#pragma unroll
  for (int u2 = 0; u2 < UMAX; ++u2) {
    if (u2 >= um) break;
    float* aw = fin[u2];
#pragma unroll
    for (int q = 0; q < NACC; ++q) aw[q] = 0.f;
    const float4* src0 = reinterpret_cast<const float4*>(p.part) +
                         ((size_t)(tile * um + u2) * ksplit * 32 + lane) * (NACC / 4);
    int s2 = 0;
    for (; s2 + 4 <= ksplit; s2 += 4) {
      float4 v[4][NACC / 4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < NACC / 4; ++q) v[u][q] = __ldcg(src0 + (s2 + u) * pstride + q);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < NACC / 4; ++q) {
          aw[4 * q] += v[u][q].x;
          aw[4 * q + 1] += v[u][q].y;
          aw[4 * q + 2] += v[u][q].z;
          aw[4 * q + 3] += v[u][q].w;
        }
    }
    for (; s2 < ksplit; ++s2) {
#pragma unroll
      for (int q = 0; q < NACC / 4; ++q) {
        const float4 v = __ldcg(src0 + s2 * pstride + q);
        aw[4 * q] += v.x;
        aw[4 * q + 1] += v.y;
        aw[4 * q + 2] += v.z;
        aw[4 * q + 3] += v.w;
      }
    }
  }
  if (lane == 0) p.tile_cnt[tile] = 0u;  // leave the counter cleared
  return true;
}

// Store epilogue: out = f (+ res); optionally packs the stored rows times
// pack_w into out_xp/out_xs and writes the tile's sums of squares (a folded
// RMSNorm of the next projection).
template <int NT>
__device__ __forceinline__ void epi_store(const GemvParams& p, const GemvSeg& sg, int lt, int m,
                                          const float (&f)[2][NT][4], int gid, int tq) {
  const int rbase = lt * 32;
  const bool packing = p.pack_w != nullptr;  // full tiles, one segment (checked by the host)
  const int g_out = (sg.out_col0 + rbase) / kGroup;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // a group (32 rows of column c) is the 8 lanes of one tq, 4 values each
    float pv[2][4];
    bool pk[2][4];
    float amax[2] = {0.f, 0.f}, ssq[2] = {0.f, 0.f};
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rloc = rt * 16 + gid + ((e & 2) ? 8 : 0);
        const int row = rbase + rloc;
        const int c = nt * 8 + 2 * tq + (e & 1);
        pk[rt][e] = false;
        pv[rt][e] = 0.f;
        if (row < sg.n && c < m) {
          const size_t o = (size_t)c * sg.ld + sg.out_col0 + row;
          float v = f[rt][nt][e];
          if (sg.res) v += __ldcg(sg.res + o);
          sg.out[o] = v;
          if (packing && c >= p.pack_c0) {
            pk[rt][e] = true;
            pv[rt][e] = v * p.pack_w[sg.out_col0 + row];
            amax[e & 1] = fmaxf(amax[e & 1], fabsf(pv[rt][e]));
            ssq[e & 1] = fmaf(v, v, ssq[e & 1]);
          }
        }
      }
    if (packing) {
      float sc[2], sum[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1)
          amax[e] = fmaxf(amax[e], __shfl_xor_sync(0xffffffffu, amax[e], o));
        sc[e] = xpack_group_scale(amax[e]);
      }
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (pk[rt][e]) {
            const int rloc = rt * 16 + gid + ((e & 2) ? 8 : 0);
            const int c = nt * 8 + 2 * tq + (e & 1);
            sum[e & 1] += xp_store_elem(p.out_xp, p.out_m, g_out, c - p.pack_c0, rloc >> 3,
                                        rloc & 7, pv[rt][e], pow2_inverse(sc[e & 1]), sc[e & 1]);
          }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = sum[e];
        float q2 = ssq[e];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          v += __shfl_xor_sync(0xffffffffu, v, o);
          q2 += __shfl_xor_sync(0xffffffffu, q2, o);
        }
        const int c = nt * 8 + 2 * tq + e;
        if (gid == 0 && c < m && c >= p.pack_c0) {
          p.out_xs[g_out * p.out_m + (c - p.pack_c0)] = make_float2(v, sc[e]);
          p.ss_out[lt * p.out_m + (c - p.pack_c0)] = q2;
        }
      }
    }
  }
}

// SwiGLU epilogue: h = silu(gate) * up (times the routed weight), packed
// for the next projection (and optionally stored).
template <int NT>
__device__ __forceinline__ void epi_swiglu(const GemvParams& p, const GemvSeg& sg, int lt,
                                           const float (&g)[2][NT][4], const float (&u)[2][NT][4],
                                           int gid, int tq) {
  const int rbase = lt * 32;
  const float scale = sg.w_idx >= 0 ? p.segw[sg.w_idx] : 1.f;
  const int g_out = (sg.out_col0 + rbase) / kGroup;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float hv[2][4];
    float amax[2] = {0.f, 0.f};
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rloc = rt * 16 + gid + ((e & 2) ? 8 : 0);
        const int c = nt * 8 + 2 * tq + (e & 1);
        const float gv = g[rt][nt][e], uv = u[rt][nt][e];
        hv[rt][e] = gv / (1.f + __expf(-gv)) * uv * scale;
        if (c < p.out_m) {
          amax[e & 1] = fmaxf(amax[e & 1], fabsf(hv[rt][e]));
          if (sg.out) sg.out[(size_t)c * sg.ld + sg.out_col0 + rbase + rloc] = hv[rt][e];
        }
      }
    float sc[2], sum[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1)
        amax[e] = fmaxf(amax[e], __shfl_xor_sync(0xffffffffu, amax[e], o));
      sc[e] = xpack_group_scale(amax[e]);
    }
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rloc = rt * 16 + gid + ((e & 2) ? 8 : 0);
        const int c = nt * 8 + 2 * tq + (e & 1);
        if (c < p.out_m)
          sum[e & 1] += xp_store_elem(p.out_xp, p.out_m, g_out, c, rloc >> 3, rloc & 7, hv[rt][e],
                                      pow2_inverse(sc[e & 1]), sc[e & 1]);
      }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = sum[e];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      const int c = nt * 8 + 2 * tq + e;
      if (gid == 0 && c < p.out_m) p.out_xs[g_out * p.out_m + c] = make_float2(v, sc[e]);
    }
  }
}

// Argmax epilogue over activation row 0: logits (optional) and the lane's best key.
__device__ __forceinline__ void epi_argmax(const GemvParams& p, const GemvSeg& sg, int lt,
                                           const float (&f)[2][1][4], int gid, int tq,
                                           unsigned long long& best) {
  const int rbase = lt * 32;
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int row = rbase + rt * 16 + gid + ((e & 2) ? 8 : 0);
      if (tq == 0 && row < sg.n) {
        const float v = f[rt][0][e];
        if (p.logits) p.logits[row] = v;
        const unsigned long long key = argmax_key(v, row);
        best = key > best ? key : best;
      }
    }
}

// CTA-wide argmax, then the grid's: the last CTA to finish writes the token
// and value.  Every thread of every CTA calls this once.
__device__ __forceinline__ void argmax_finish(const GemvParams& p, unsigned long long best) {
  __shared__ unsigned long long red[kGemvWarps];
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
    best = other > best ? other : best;
  }
  if (lane == 0) red[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = red[0];
    for (int w2 = 1; w2 < kGemvWarps; ++w2) b = red[w2] > b ? red[w2] : b;
    p.am_partial[blockIdx.x] = b;
    const unsigned prev = atom_add_acq_rel_gpu(p.am_counter, 1u);  // releases the partial
    last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (last) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");  // every CTA's partial, for all threads
    unsigned long long b = 0ull;
    for (int i2 = threadIdx.x; i2 < (int)gridDim.x; i2 += blockDim.x) {
      const unsigned long long v = __ldcg(p.am_partial + i2);
      b = v > b ? v : b;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, b, o);
      b = other > b ? other : b;
    }
    if (lane == 0) red[warp] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long bb = red[0];
      for (int w2 = 1; w2 < kGemvWarps; ++w2) bb = red[w2] > bb ? red[w2] : bb;
      *p.am_token = argmax_key_index(bb);
      *p.am_value = argmax_key_value(bb);
      *p.am_counter = 0u;  // leave the workspace cleared for the next call
    }
  }
}

// ------------------------------------------------------- several activation rows
// m in 2..16: the m16n8 tiles' columns are activation rows (NT tiles of 8).
// PC (m <= 4, one tile of columns): the eight columns are (activation row,
// hi/lo part) pairs instead, so one product covers both parts of four rows:
// half the MMAs and activation fragments per stage; lane (gid, tq) sums the
// two parts of row tq and applies that row's group scale and sum.  At a
// unit's end the per-lane results move (shuffles) to the column layout the
// epilogues share.
// With staged activations the paired-column kernel fits two CTAs per SM, and
// may first move a whole stage into registers, release its slot for the next
// copy and then compute (tuning knob: 1 releases early, 0 after the stage).
#ifndef MTP_TC_PC_EARLY
#define MTP_TC_PC_EARLY 1
#endif
constexpr bool kTcPcEarly = MTP_TC_PC_EARLY != 0;

template <int NMAT, int NT, int EPI, int S, int XM, bool PAIRED = false, bool PC = false>
__global__ void __launch_bounds__(kGemvWarps * 32,
                                  (NMAT == 1 && NT == 1 && !(PC && XM > 0)) ? 4 : 2)
    gemv_tc_kernel(const __grid_constant__ GemvParams p) {
  static_assert(!PC || NT == 1, "paired columns: one column tile");
  // PAIRED: the SwiGLU gate and up matrices of a tile are separate work
  // units (one matrix in flight per warp); their partial sums meet in the
  // split-K reduction.
  constexpr int UM = PAIRED ? 2 : 1;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of each codes tile is required by the 128B swizzle.
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;
  const int tq = lane & 3;

  constexpr int kCode = NMAT * 4096;                   // codes per stage (1 KB aligned)
  constexpr int kRest = NMAT * 2048 + gemv_xchunk_bytes<XM>();  // scales, biases, activations
  uint8_t* code_base = smem + warp * S * kCode;
  uint8_t* rest_base = smem + kGemvWarps * S * kCode + warp * S * kRest;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + kGemvWarps * S * (kCode + kRest)) + warp * S;

  const int m = p.m;
  const int G = p.K / kGroup;
  const int KS = (G + 7) / 8;
  const int ksplit = p.ksplit, spu = p.spu;
  const int W = gridDim.x * kGemvWarps;
  const int gw = warp * gridDim.x + blockIdx.x;
  const int total_tiles = p.seg[p.nseg - 1].tile_end;
  const int units = total_tiles * UM * ksplit;

  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncwarp();

  const uint64_t pol_w = l2_policy_evict_first();
  const uint64_t pol_x = l2_policy_evict_last();
  auto issue_w = [&](const Cursor& c, int slot) {
    int mat, row, kx, sx;
    c.coords(p, mat, row, kx, sx);
    uint8_t* cd = code_base + slot * kCode;
    uint8_t* rs = rest_base + slot * kRest;
    uint32_t bytes = NMAT * kStageMatBytes;
    if (XM > 0) bytes += (uint32_t)8 * m * (128 + 8);
    mbar_arrive_expect_tx(&bars[slot], bytes);
#pragma unroll
    for (int mi = 0; mi < NMAT; ++mi) {
      const QMat& mt = p.mat[mat + mi];
      tma_load_2d(cd + mi * 4096, &mt.q, &bars[slot], kx, row, pol_w);
      tma_load_2d(rs + mi * 2048, &mt.s, &bars[slot], sx, row, pol_w);
      tma_load_2d(rs + mi * 2048 + 1024, &mt.b, &bars[slot], sx, row, pol_w);
    }
  };
  auto issue_x = [&](const Cursor& c, int slot) {
    if constexpr (XM > 0) {
      uint8_t* rs = rest_base + slot * kRest + NMAT * 2048;
      const int g0 = c.ks * 8;
      bulk_load(rs, p.xp + (size_t)g0 * m * 8, (uint32_t)8 * m * 128, &bars[slot], pol_x);
      bulk_load(rs + XM * 1024, p.xs + (size_t)g0 * m, (uint32_t)8 * m * 8, &bars[slot], pol_x);
    }
  };

  // Weights never depend on the previous kernel: start streaming them before
  // waiting on it, unless the rows to stream are chosen by it (then even the
  // cursor, which resolves those rows, starts after the wait).
  Cursor pc, cc;
  int pre = 0;
  Cursor pre_c[S];
  if (!p.rowsel_after_wait) {
    pc.start(p, gw, units, ksplit, spu, KS, UM);
    cc = pc;
    if (lane == 0) {
      for (; pre < S && pc.u < units; ++pre) {
        pre_c[pre] = pc;
        issue_w(pc, pre);
        pc.advance(p, W, units, ksplit, spu, KS, UM);
      }
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  if (p.rowsel_after_wait) {
    pc.start(p, gw, units, ksplit, spu, KS, UM);
    cc = pc;
  }
  if (lane == 0) {
    for (int i = 0; i < pre; ++i) issue_x(pre_c[i], i);
    for (; pre < S && pc.u < units; ++pre) {
      issue_w(pc, pre);
      issue_x(pc, pre);
      pc.advance(p, W, units, ksplit, spu, KS, UM);
    }
  }
  // (after the first activation copies are in flight: these loads wait on L2)
  float rsc[NT][2];
  row_scales<NT>(p, m, tq, false, rsc);

  float acc[NMAT][2][NT][4];
  float accp[NMAT][2][2];  // PC: [mi][rt][row gid, gid + 8] for activation row tq
#pragma unroll
  for (int mi = 0; mi < NMAT; ++mi) accp[mi][0][0] = accp[mi][0][1] = accp[mi][1][0] = accp[mi][1][1] = 0.f;
#pragma unroll
  for (int mi = 0; mi < NMAT; ++mi)
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][rt][nt][e] = 0.f;

  // ldmatrix addressing: lane supplies row ri + 8*(mtx&1) of a 16-row tile
  // and group 2*jp + (mtx>>1).  With the 128-byte swizzle that group's chunk
  // sits at ((2*jp + (mtx>>1)) ^ ri) << 4 = (jp << 5) ^ (((mtx>>1) ^ ri) << 4),
  // because 2*jp and mtx>>1 occupy different bits.
  const int ri = lane & 7, mtx = lane >> 3;
  const uint32_t ld_lane = smem_u32(code_base) + (uint32_t)(ri + 8 * (mtx & 1)) * 128;
  const uint32_t ld_c = (uint32_t)(((mtx >> 1) ^ ri) << 4);
  const int sb_lane = gid * 8;  // float offset of row gid in a [32][8] scale tile

  uint4 bh[2][NT], bl[2][NT];      // activation fragments of the next pair of groups
  float2 xs0[2][NT], xs1[2][NT];
  bool b_ready = false;
  for (int i = 0; cc.u < units; ++i) {
    const int slot = i % S;
    if (!mbar_wait_bounded(&bars[slot], (uint32_t)((i / S) & 1))) {
      // give up on the remaining work of this warp
      if (lane == 0) set_dev_error(p.err, kErrMbarTimeout);
      break;
    }
    const uint32_t cd = ld_lane + slot * kCode;
    const uint8_t* rs = rest_base + slot * kRest;
    const int gbase = cc.ks * 8;

    // B fragments (activations) of a pair of groups and their group sums.
    auto load_b_at = [&](int gb, int jp, uint4 (&bh)[2][NT], uint4 (&bl)[2][NT],
                         float2 (&x0)[2][NT], float2 (&x1)[2][NT]) {
      const uint4* xp_st = p.xp + (size_t)(gb * m) * 8;
      const float2* xs_st = p.xs + (size_t)gb * m;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * jp + h;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          bh[h][nt] = make_uint4(0, 0, 0, 0);
          bl[h][nt] = make_uint4(0, 0, 0, 0);
          x0[h][nt] = make_float2(0.f, 0.f);
          x1[h][nt] = make_float2(0.f, 0.f);
          const int c = nt * 8 + gid;
          const int c0 = nt * 8 + 2 * tq;
          if constexpr (XM > 0) {
            const uint4* xps = reinterpret_cast<const uint4*>(rs + NMAT * 2048);
            const float2* xss = reinterpret_cast<const float2*>(rs + NMAT * 2048 + XM * 1024);
            if (c < m) {
              bh[h][nt] = xps[xp_index(j, c, tq, 0, m)];
              bl[h][nt] = xps[xp_index(j, c, tq, 1, m)];
            }
            if (c0 < m) x0[h][nt] = xss[j * m + c0];
            if (c0 + 1 < m) x1[h][nt] = xss[j * m + c0 + 1];
          } else {
            if (c < m) {
              const uint4* src = xp_st + xp_index(j, c, tq, 0, m);
              bh[h][nt] = __ldg(src);
              bl[h][nt] = __ldg(src + 1);
            }
            if (c0 < m) x0[h][nt] = __ldg(xs_st + j * m + c0);
            if (c0 + 1 < m) x1[h][nt] = __ldg(xs_st + j * m + c0 + 1);
          }
        }
      }
    };
    auto load_b = [&](int jp, uint4 (&bh)[2][NT], uint4 (&bl)[2][NT], float2 (&x0)[2][NT],
                      float2 (&x1)[2][NT]) { load_b_at(gbase, jp, bh, bl, x0, x1); };
    // Pairs of groups.  Each pair issues its tensor-core products, then loads
    // the next pair's activations into the same registers (their latency
    // overlaps the scale/bias epilogue), then applies scales and biases.  The
    // last pair of a stage loads the first pair of the next stage when it
    // continues the same unit (global activations only).  Activations are
    // zero-padded to whole stages of 8 groups.
    bool refilled = false;
    if constexpr (PC && XM > 0 && kTcPcEarly) {
      static_assert(NMAT == 1, "paired columns: one matrix per unit");
      // the whole stage into registers: codes (ldmatrix), the rows'
      // activation fragments and group sums, the lane's scales and biases
      const uint4* xps = reinterpret_cast<const uint4*>(rs + 2048);
      const float2* xss = reinterpret_cast<const float2*>(rs + 2048 + XM * 1024);
      const int cb = gid >> 1, hl = gid & 1;
      uint32_t wr[4][2][4];
      uint4 bpr[4][2];
      float2 xvr[4][2];
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        const uint32_t coff = ((uint32_t)jp << 5) ^ ld_c;
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
          ldmatrix_x4(wr[jp][rt][0], wr[jp][rt][1], wr[jp][rt][2], wr[jp][rt][3],
                      cd + rt * 2048 + coff);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 2 * jp + h;
          bpr[jp][h] = cb < m ? xps[xp_index(j, cb, tq, hl, m)] : make_uint4(0u, 0u, 0u, 0u);
          xvr[jp][h] = tq < m ? xss[j * m + tq] : make_float2(0.f, 0.f);
        }
      }
      // [rt][row gid / gid + 8][groups 0-3 / 4-7] of the [32][8] scale and bias tiles
      float4 scr[2][2][2], bir[2][2][2];
      const float* sbase = reinterpret_cast<const float*>(rs) + sb_lane;
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            scr[rt][r2][q] = *reinterpret_cast<const float4*>(sbase + rt * 128 + r2 * 64 + q * 4);
            bir[rt][r2][q] = *reinterpret_cast<const float4*>(sbase + 256 + rt * 128 + r2 * 64 + q * 4);
          }
      // the slot is free: the warp's reads precede the next copy into it
      __syncwarp();
      if (lane == 0 && pc.u < units) {
        fence_proxy_async_shared_cta();
        issue_w(pc, slot);
        issue_x(pc, slot);
        pc.advance(p, W, units, ksplit, spu, KS, UM);
      }
      refilled = true;
      auto comp = [](const float4& v, int i) {
        return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
      };
#pragma unroll
      for (int jp = 0; jp < 4; ++jp)
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wa = wr[jp][rt][2 * h], wb = wr[jp][rt][2 * h + 1];
            const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
            float dd[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16_16816(dd, codes_lo_f16x2(wa), codes_lo_f16x2(wb), codes_hi_f16x2(wa),
                          codes_hi_f16x2(wb), bpr[jp][h].x, bpr[jp][h].y);
            mma_f16_16816(dd, codes_lo_f16x2(wa8), codes_lo_f16x2(wb8), codes_hi_f16x2(wa8),
                          codes_hi_f16x2(wb8), bpr[jp][h].z, bpr[jp][h].w);
            const int g = 2 * jp + h;
            const float s0 = comp(scr[rt][0][g >> 2], g & 3), s1 = comp(scr[rt][1][g >> 2], g & 3);
            const float b0 = comp(bir[rt][0][g >> 2], g & 3), b1 = comp(bir[rt][1][g >> 2], g & 3);
            accp[0][rt][0] = fmaf(s0 * xvr[jp][h].y, dd[0] + dd[1], fmaf(b0, xvr[jp][h].x, accp[0][rt][0]));
            accp[0][rt][1] = fmaf(s1 * xvr[jp][h].y, dd[2] + dd[3], fmaf(b1, xvr[jp][h].x, accp[0][rt][1]));
          }
    } else if constexpr (PC) {
      // B column gid is part (gid & 1) of activation row gid >> 1; lane tq
      // scales and sums row tq's product
      // the stage's activations: staged with the weights, or read through L1
      const uint4* xps = XM > 0 ? reinterpret_cast<const uint4*>(rs + NMAT * 2048)
                                : p.xp + (size_t)gbase * m * 8;
      const float2* xss = XM > 0 ? reinterpret_cast<const float2*>(rs + NMAT * 2048 + XM * 1024)
                                 : p.xs + (size_t)gbase * m;
      const int cb = gid >> 1, hl = gid & 1;
#pragma unroll 1
      for (int jp = 0; jp < 4; ++jp) {
        const uint32_t coff = ((uint32_t)jp << 5) ^ ld_c;
        uint4 bp[2];
        float2 xv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 2 * jp + h;
          bp[h] = cb < m ? (XM > 0 ? xps[xp_index(j, cb, tq, hl, m)] : __ldg(xps + xp_index(j, cb, tq, hl, m)))
                         : make_uint4(0u, 0u, 0u, 0u);
          xv[h] = tq < m ? (XM > 0 ? xss[j * m + tq] : __ldg(xss + j * m + tq)) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int mi = 0; mi < NMAT; ++mi) {
          const float* ssm = reinterpret_cast<const float*>(rs + mi * 2048) + sb_lane + 2 * jp;
          const float* bsm = ssm + 256;
#pragma unroll
          for (int rt = 0; rt < 2; ++rt) {
            uint32_t w[4];
            ldmatrix_x4(w[0], w[1], w[2], w[3], cd + mi * 4096 + rt * 2048 + coff);
            const float2 sa = *reinterpret_cast<const float2*>(ssm + rt * 128);
            const float2 sb = *reinterpret_cast<const float2*>(ssm + rt * 128 + 64);
            const float2 ba = *reinterpret_cast<const float2*>(bsm + rt * 128);
            const float2 bb = *reinterpret_cast<const float2*>(bsm + rt * 128 + 64);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t wa = w[2 * h], wb = w[2 * h + 1];
              const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
              float dd[4] = {0.f, 0.f, 0.f, 0.f};
              mma_f16_16816(dd, codes_lo_f16x2(wa), codes_lo_f16x2(wb), codes_hi_f16x2(wa),
                            codes_hi_f16x2(wb), bp[h].x, bp[h].y);
              mma_f16_16816(dd, codes_lo_f16x2(wa8), codes_lo_f16x2(wb8), codes_hi_f16x2(wa8),
                            codes_hi_f16x2(wb8), bp[h].z, bp[h].w);
              const float s0 = h ? sa.y : sa.x, s1 = h ? sb.y : sb.x;
              const float b0 = h ? ba.y : ba.x, b1 = h ? bb.y : bb.x;
              accp[mi][rt][0] = fmaf(s0 * xv[h].y, dd[0] + dd[1], fmaf(b0, xv[h].x, accp[mi][rt][0]));
              accp[mi][rt][1] = fmaf(s1 * xv[h].y, dd[2] + dd[3], fmaf(b1, xv[h].x, accp[mi][rt][1]));
            }
          }
        }
      }
    } else {
    if (!b_ready) load_b(0, bh, bl, xs0, xs1);
    const bool next_same_unit = XM == 0 && cc.ks + 1 < cc.ke;
#pragma unroll 1
    for (int jp = 0; jp < 4; ++jp) {
      const uint32_t coff = ((uint32_t)jp << 5) ^ ld_c;
      float d[NMAT][2][2][NT][4];
      float2 sx0[2][NT], sx1[2][NT];  // (sum, scale) of the columns' groups
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          sx0[h][nt] = xs0[h][nt];
          sx1[h][nt] = xs1[h][nt];
        }
#pragma unroll
      for (int mi = 0; mi < NMAT; ++mi) {
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
          // (rows 0-7, group 2jp), (rows 8-15, 2jp), (rows 0-7, 2jp+1), (rows 8-15, 2jp+1)
          uint32_t w[4];
          ldmatrix_x4(w[0], w[1], w[2], w[3], cd + mi * 4096 + rt * 2048 + coff);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wa = w[2 * h], wb = w[2 * h + 1];
            const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
            // exact codes (and 16 * codes) times 2^-24 as f16: the accumulator
            // only ever holds sums of code * x, so its rounding stays at that scale
            const uint32_t a0 = codes_lo_f16x2(wa);
            const uint32_t a1 = codes_lo_f16x2(wb);
            const uint32_t a2 = codes_hi_f16x2(wa);
            const uint32_t a3 = codes_hi_f16x2(wb);
            const uint32_t a4 = codes_lo_f16x2(wa8);
            const uint32_t a5 = codes_lo_f16x2(wb8);
            const uint32_t a6 = codes_hi_f16x2(wa8);
            const uint32_t a7 = codes_hi_f16x2(wb8);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float* dd = d[mi][rt][h][nt];
              dd[0] = dd[1] = dd[2] = dd[3] = 0.f;
              mma_f16_16816(d[mi][rt][h][nt], a0, a1, a2, a3, bh[h][nt].x, bh[h][nt].y);
              mma_f16_16816(d[mi][rt][h][nt], a0, a1, a2, a3, bl[h][nt].x, bl[h][nt].y);
              mma_f16_16816(d[mi][rt][h][nt], a4, a5, a6, a7, bh[h][nt].z, bh[h][nt].w);
              mma_f16_16816(d[mi][rt][h][nt], a4, a5, a6, a7, bl[h][nt].z, bl[h][nt].w);
            }
          }
        }
      }
      if (jp < 3)
        load_b(jp + 1, bh, bl, xs0, xs1);
      else if (next_same_unit)
        load_b_at(gbase + 8, 0, bh, bl, xs0, xs1);
#pragma unroll
      for (int mi = 0; mi < NMAT; ++mi) {
        const float* ssm = reinterpret_cast<const float*>(rs + mi * 2048) + sb_lane + 2 * jp;
        const float* bsm = ssm + 256;
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
          const float2 sa = *reinterpret_cast<const float2*>(ssm + rt * 128);
          const float2 sb = *reinterpret_cast<const float2*>(ssm + rt * 128 + 64);
          const float2 ba = *reinterpret_cast<const float2*>(bsm + rt * 128);
          const float2 bb = *reinterpret_cast<const float2*>(bsm + rt * 128 + 64);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float s0 = h ? sa.y : sa.x, s1 = h ? sb.y : sb.x;
            const float b0 = h ? ba.y : ba.x, b1 = h ? bb.y : bb.x;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float* dd = d[mi][rt][h][nt];
              float* a = acc[mi][rt][nt];
              const float2 x0 = sx0[h][nt], x1 = sx1[h][nt];
              a[0] = fmaf(s0 * x0.y, dd[0], fmaf(b0, x0.x, a[0]));
              a[2] = fmaf(s1 * x0.y, dd[2], fmaf(b1, x0.x, a[2]));
              a[1] = fmaf(s0 * x1.y, dd[1], fmaf(b0, x1.x, a[1]));
              a[3] = fmaf(s1 * x1.y, dd[3], fmaf(b1, x1.x, a[3]));
            }
          }
        }
      }
    }
    b_ready = next_same_unit;
    }  // PC
    __syncwarp();
    if (lane == 0 && !refilled && pc.u < units) {
      issue_w(pc, slot);
      issue_x(pc, slot);
      pc.advance(p, W, units, ksplit, spu, KS, UM);
    }

    const int unit = cc.u;
    const int tile = cc.tile;
    const int seg = cc.seg;
    if (!cc.advance(p, W, units, ksplit, spu, KS, UM)) continue;

    // ------------------------------------------------------------ unit done
    if constexpr (PC) {
      // to the column layout: element e of lane (gid, tq) is row gid + 8 (e >> 1),
      // activation row 2tq + (e & 1), held by lane (gid, 2tq + (e & 1))
#pragma unroll
      for (int mi = 0; mi < NMAT; ++mi)
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 2 * tq + (e & 1);
            const float v = __shfl_sync(0xffffffffu, accp[mi][rt][e >> 1], gid * 4 + (c & 3));
            acc[mi][rt][0][e] = c < 4 ? v : 0.f;
          }
          accp[mi][rt][0] = accp[mi][rt][1] = 0.f;
        }
    }
    // fin[um] is the tile's full sum for matrix um of the unit's tile
    constexpr int NACC = NMAT * 2 * NT * 4;
    float fin[UM][NACC];
    float* af = &acc[0][0][0][0];
    if (ksplit > 1 || PAIRED) {
      if (!splitk_finish<NACC, UM>(p, unit, tile, UM, ksplit, af, fin, lane)) continue;
    } else {
#pragma unroll
      for (int q = 0; q < NACC; ++q) {
        fin[0][q] = af[q];
        af[q] = 0.f;
      }
    }
    // undo the 2^-24 of the subnormal codes (exact) and apply the input-row
    // scales of a folded RMSNorm; q = ((mi * 2 + rt) * NT + nt) * 4 + e
#pragma unroll
    for (int um = 0; um < UM; ++um)
#pragma unroll
      for (int q = 0; q < NACC; ++q) fin[um][q] *= kCodeScale * rsc[(q >> 2) % NT][q & 1];

    const GemvSeg& sg = p.seg[seg];
    const int lt = tile - (seg ? p.seg[seg - 1].tile_end : 0);
    using Frag = float[2][NT][4];
    if constexpr (EPI == kEpiStore) {
      epi_store<NT>(p, sg, lt, m, *reinterpret_cast<const Frag*>(fin[0]), gid, tq);
    } else if constexpr (EPI == kEpiSwiglu) {
      const float* gf = fin[0];
      const float* uf = PAIRED ? fin[UM - 1] : fin[0] + (NMAT - 1) * 2 * NT * 4;
      epi_swiglu<NT>(p, sg, lt, *reinterpret_cast<const Frag*>(gf),
                     *reinterpret_cast<const Frag*>(uf), gid, tq);
    }
  }
}

// ------------------------------------------------------------ one activation row
// m = 1.  One launch streams up to kMaxPhases projections in order (the
// phases of a layer between two dependencies on other kernels): every warp
// walks the phases' work units with one continuous TMA pipeline, so the
// weights of a phase are already streaming while the previous phase
// finishes.  A phase reads its activation row only after all tiles of the
// previous phase are written (per-phase tile counters; bounded waits).
constexpr int kMaxPhases = 4;

// Work a launch does before its first phase: units of one warp each, run
// right after the wait on the previous kernel; the first phase's activation
// copies wait for all of them (pre_done).
enum PreKind : int {
  kPreNone = 0,
  // pack [embed(token) * enorm ; hidden * hnorm] unnormalised (one 32-value
  // group per unit) with each group's sum of squares of the raw values; the
  // first phase scales the units of each half by rsqrt(mean + eps)
  kPreEmbedPack = 1,
  // merge the split-K partials of decode attention (one 32-dim group of the
  // output per unit): sink in the denominator, sigmoid gate, packed output
  kPreAttnMerge = 2,
};

struct PreParams {
  int kind;
  int units;
  uint4* xp;         // packed output row
  float2* xs;
  // kPreEmbedPack
  const float* table;  // [vocab][dim] (or null: rows)
  const int* tokens;
  int vocab;
  const float* rows;   // [dim] embedding row given directly
  const float* hidden; // [dim]
  const float* w0;     // enorm
  const float* w1;     // hnorm
  int dim;
  float eps;
  float* ss;           // [2 * dim / 32] raw sums of squares per group
  // kPreAttnMerge (m = 1)
  const float* part;   // (M, l) pairs [nkv][ns][G] then outputs [nkv][ns][G][dv] at part_o
  const float* part_o;
  int nkv, ns, G, dv, dqk, gated, q_rows;
  const float* sinks;  // [nkv * G] or null
  const float* qp;     // gate source (q projection row)
};

struct StreamParams {
  GemvParams ph[kMaxPhases];  // m = 1; phase epilogues kEpiStore / kEpiSwiglu / kEpiArgmax (last)
  int nphase;
  unsigned* phase_done;       // [kMaxPhases + 1] finished tiles per phase, then pre-units;
                              // zero at launch, cleared at the end
  int* err;
  PreParams pre;
};

// One 32-value group of [embed * enorm ; hidden * hnorm], packed unnormalised,
// with the group's raw sum of squares (one warp).
__device__ __forceinline__ void pre_embed_pack(const PreParams& q, int u, int* err, int lane) {
  const int gpr = q.dim / kGroup;
  const bool first = u < gpr;
  const int k = (first ? u : u - gpr) * kGroup + lane;
  const float* row;
  if (first) {
    if (q.table) {
      int tok = q.tokens[0];
      if (tok < 0 || tok >= q.vocab) {
        if (lane == 0) set_dev_error(err, kErrBadToken);
        tok = 0;
      }
      row = q.table + (size_t)tok * q.dim;
    } else {
      row = q.rows;
    }
  } else {
    row = q.hidden;
  }
  const float wv = first ? q.w0[k] : q.w1[k];
  const float x = __ldcg(row + k);
  const float v = x * wv;
  const float2 hs = xp_store_group(q.xp, 1, u, 0, lane, v);
  const float ss = warp_sum(x * x);
  if (lane == 0) {
    q.xs[u] = hs;
    q.ss[u] = ss;
  }
}

// One 32-dim group of the attention output (m = 1): merges the splits'
// partials with weights exp2(M_s - M) / den, den including the head's sink
// logit, applies the sigmoid gate and packs the group (one warp).  Every
// load of a chunk of 32 splits is issued before any arithmetic.
__device__ __forceinline__ void pre_attn_merge(const PreParams& q, int u, int lane) {
  const int gph = q.dv / kGroup;           // groups per head
  const int h = u / gph, d0 = (u - h * gph) * kGroup;
  const int kvh = h / q.G, qi = h - kvh * q.G;
  const float* ml = q.part + ((size_t)kvh * q.ns * q.G + qi) * 2;  // stride G * 2 per split
  const float* po = q.part_o + ((size_t)kvh * q.ns * q.G + qi) * q.dv + d0 + lane;
  const size_t sstride = (size_t)q.G * q.dv;
  const float g = q.gated ? q.qp[(size_t)h * q.dqk * 2 + q.dqk + d0 + lane] : 0.f;
  const float sinkl2 = q.sinks ? q.sinks[h] * 1.4426950408889634f : -1e30f;
  // running merge over chunks of 32 splits (one chunk for up to 32 splits)
  float Mrun = sinkl2, den = q.sinks ? 1.f : 0.f, acc = 0.f;
  for (int s0 = 0; s0 < q.ns; s0 += 32) {
    const int n = min(32, q.ns - s0);
    const int sl = s0 + lane;
    const float2 mlv = sl < q.ns ? __ldcg(reinterpret_cast<const float2*>(ml + (size_t)sl * q.G * 2))
                                 : make_float2(-1e30f, 0.f);
    float v[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = t < n ? __ldcg(po + (size_t)(s0 + t) * sstride) : 0.f;
    const float M = fmaxf(Mrun, warp_max(mlv.x));
    const float wl = sl < q.ns ? exp2f(mlv.x - M) : 0.f;
    const float scale = exp2f(Mrun - M);
    den = den * scale + warp_sum(wl * mlv.y);
    acc *= scale;
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (t < n) acc = fmaf(__shfl_sync(0xffffffffu, wl, t), v[t], acc);  // split order
    Mrun = M;
  }
  acc = den > 0.f ? acc / den : 0.f;
  if (q.gated) acc = acc / (1.f + __expf(-g));
  const float2 hs = xp_store_group(q.xp, 1, (h * q.dv + d0) / kGroup, 0, lane, acc);
  if (lane == 0) q.xs[(h * q.dv + d0) / kGroup] = hs;
}

constexpr unsigned kPhaseSpinLimit = 4u << 20;  // polls of >= 256 ns each before giving up

// One-row stages: 32 rows x 8 groups, as for several rows (4 KB of codes in a
// 128B-swizzled tile, 1 KB scales, 1 KB biases) plus the staged activations
// of the 8 groups (1 KB) and their sums (64 B).
constexpr int kRowCode = 4096;
constexpr int kRowRest = 2048 + 1152;  // scales, biases, activations (128-byte multiple)
constexpr int kRowStageTx = kStageMatBytes + 8 * (128 + 8);
// with bfloat16 scales and biases: 512-byte tiles in the same places
constexpr int kRowStageTxBf16 = kStageMatBytes - 1024 + 8 * (128 + 8);

// Matrix slot a stage of the cursor reads (its scale type lives per slot).
__device__ __forceinline__ int stage_slot(const GemvParams& p, const Cursor& c) {
  if (p.kseg_len > 0 && p.kseg_last_mat >= 0) {
    const int spk = p.kseg_len / (8 * kGroup);
    if (c.ks / spk >= p.nkseg - 1) return p.kseg_last_mat;
  }
  return c.mat;
}

// Waits until *cnt >= target (acquire); false when the wait gives up.
// Every warp of a launch polls the same counter: sleeps of 512 ns keep the
// polls from slowing the publishers' atomics on it (measured on the draft
// step: 32 or 64 ns cost 6 us, 256 ns 1.4 us, 1024 ns 1.6 us over 512 ns).
__device__ __forceinline__ bool wait_count(const unsigned* cnt, unsigned target, unsigned polls) {
  for (unsigned i = 0; i < polls; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    __nanosleep(512);
  }
  return false;
}

// Position in the phases' work units (lane 0's producer copy and every
// lane's consumer copy are advanced identically).
struct PhaseCursor {
  Cursor c;
  int ph;   // kMaxPhases (or nphase) when done
};

__device__ __forceinline__ int phase_units(const GemvParams& p) {
  return p.seg[p.nseg - 1].tile_end * p.um * p.ksplit;
}
__device__ __forceinline__ int phase_ks(const GemvParams& p) { return (p.K / kGroup + 7) / 8; }

// First unit of this warp in phase `ph` or a later one.
__device__ __forceinline__ void phase_start(const StreamParams& sp, PhaseCursor& x, int ph, int gw) {
  for (; ph < sp.nphase; ++ph) {
    const GemvParams& p = sp.ph[ph];
    if (gw < p.wq) {
      x.ph = ph;
      const int units = phase_units(p);
      x.c.start(p, gw, units, p.ksplit, p.spu, phase_ks(p), p.um);
      return;
    }
  }
  x.ph = sp.nphase;
}

// Advances by one stage; true when a unit just finished.
__device__ __forceinline__ bool phase_advance(const StreamParams& sp, PhaseCursor& x, int gw) {
  const GemvParams& p = sp.ph[x.ph];
  if (++x.c.ks < x.c.ke) return false;
  const int units = phase_units(p);
  const int u = x.c.u + p.wq;
  if (u < units)
    x.c.start(p, u, units, p.ksplit, p.spu, phase_ks(p), p.um);
  else
    phase_start(sp, x, x.ph + 1, gw);
  return true;
}

// Sum of src[32 s] for s < n in order s = 0, 1, ... (loads eight at a time).
__device__ __forceinline__ float sum_rows(const float* src, int n) {
  float t = 0.f;
  int s0 = 0;
  for (; s0 + 8 <= n; s0 += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (size_t)(s0 + j) * 32);
#pragma unroll
    for (int j = 0; j < 8; ++j) t += v[j];
  }
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = s0 + j < n ? __ldcg(src + (size_t)(s0 + j) * 32) : 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (s0 + j < n) t += v[j];
  return t;
}

// SBF: some slot of the launch has bfloat16 scales and biases (the
// MlxAffineMoeStack layout); the all-f32 instantiation has no per-stage test.
template <int S, bool SBF>
__global__ void __launch_bounds__(kGemvWarps * 32, 3)
    gemv_row_kernel(const __grid_constant__ StreamParams sp) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of each codes tile is required by the 128B swizzle
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;
  const int tq = lane & 3;
  uint8_t* code_base = smem + warp * S * kRowCode;
  uint8_t* rest_base = smem + kGemvWarps * S * kRowCode + warp * S * kRowRest;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + kGemvWarps * S * (kRowCode + kRowRest)) + warp * S;
  const int W = gridDim.x * kGemvWarps;
  const int gw = warp * gridDim.x + blockIdx.x;

  __shared__ __align__(16) uint4 zero_b[16];  // B fragments of lanes outside their group's column
  if (threadIdx.x < 16) zero_b[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncwarp();

  const uint64_t pol_w = l2_policy_evict_first();
  const uint64_t pol_x = l2_policy_evict_last();
  auto issue_w = [&](const PhaseCursor& c, int slot) {
    const GemvParams& p = sp.ph[c.ph];
    int mat, row, kx, sx;
    c.c.coords(p, mat, row, kx, sx);
    uint8_t* cd = code_base + slot * kRowCode;
    uint8_t* rs = rest_base + slot * kRowRest;
    const bool bf = SBF && ((p.sbf_mask >> mat) & 1);
    mbar_arrive_expect_tx(&bars[slot], (uint32_t)(bf ? kRowStageTxBf16 : kRowStageTx));
    const QMat& mt = p.mat[mat];
    tma_load_2d(cd, &mt.q, &bars[slot], kx, row, pol_w);
    tma_load_2d(rs, &mt.s, &bars[slot], sx, row, pol_w);
    tma_load_2d(rs + 1024, &mt.b, &bars[slot], sx, row, pol_w);
  };
  auto issue_x = [&](const PhaseCursor& c, int slot) {
    const GemvParams& p = sp.ph[c.ph];
    uint8_t* rs = rest_base + slot * kRowRest + 2048;
    const int g0 = c.c.ks * 8;
    bulk_load(rs, p.xp + (size_t)g0 * 8, 8 * 128, &bars[slot], pol_x);
    bulk_load(rs + 1024, p.xs + g0, 8 * 8, &bars[slot], pol_x);
  };

  // Producer state (lane 0): pc is the next stage to issue; a stage whose
  // phase's input is not yet complete gets its weights now and its
  // activations once the consumer has seen that phase's input complete.
  PhaseCursor pc, cc;
  PhaseCursor pend_c[S];
  bool pend[S];
#pragma unroll
  for (int i = 0; i < S; ++i) pend[i] = false;
  // (slots are indexed with unrolled compares so these stay in registers)
  auto defer_x = [&](const PhaseCursor& c, int slot) {
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2)
      if (s2 == slot) {
        pend_c[s2] = c;
        pend[s2] = true;
      }
  };
  int issued = 0;  // stages issued so far (lane 0)
  // phases <= ready have their input complete (phase 0 after the previous
  // kernel, or after this launch's pre-units)
  int ready = sp.pre.kind != kPreNone ? -1 : 0;
  const bool first_sel = sp.ph[0].rowsel_after_wait != 0;
  if (!first_sel) {
    phase_start(sp, pc, 0, gw);
    cc = pc;
    if (lane == 0)
      for (; issued < S && pc.ph < sp.nphase && !sp.ph[pc.ph].rowsel_after_wait; ++issued) {
        issue_w(pc, issued);
        defer_x(pc, issued);
        phase_advance(sp, pc, gw);
      }
  }
  // the first phase's input comes from the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  if (first_sel) {
    phase_start(sp, pc, 0, gw);
    cc = pc;
  }
  if (lane == 0) {
#pragma unroll
    for (int s2 = 0; s2 < S; ++s2)
      if (pend[s2] && pend_c[s2].ph <= ready) {
        issue_x(pend_c[s2], s2);
        pend[s2] = false;
      }
    for (; issued < S && pc.ph < sp.nphase; ++issued) {
      issue_w(pc, issued);
      if (pc.ph <= ready)
        issue_x(pc, issued);
      else
        defer_x(pc, issued);
      phase_advance(sp, pc, gw);
    }
  }
  // pre-units of this warp (after its first weight copies are in flight)
  if (sp.pre.kind != kPreNone) {
    unsigned n_pre = 0;
    for (int u = gw; u < sp.pre.units; u += W, ++n_pre) {
      if (sp.pre.kind == kPreEmbedPack)
        pre_embed_pack(sp.pre, u, sp.err, lane);
      else
        pre_attn_merge(sp.pre, u, lane);
    }
    __syncwarp();  // the warp's stores, then one release by lane 0
    if (lane == 0 && n_pre > 0) red_add_release_gpu(sp.phase_done + kMaxPhases, n_pre);
  }

  // The eight MMA columns carry (group, hi/lo) pairs instead of activation
  // rows: in set st (0, 1) lane (gid, tq) feeds k-slots {2tq, 2tq+1, 2tq+8,
  // 2tq+9} with codes of group 2tq + st of rows gid and gid + 8, and column
  // 2j + h of B holds part h (hi, lo) of that group's activations in lane j's
  // slots (zeros in the others).  So D[row][2tq + h] is part h of the row's
  // product with group 2tq + st, and each lane applies its own groups' scales.
  const int a_chunk[2] = {((2 * tq) ^ gid) << 4, ((2 * tq + 1) ^ gid) << 4};
  const bool b_active = (gid >> 1) == tq;
  const int b_off = (gid >> 1) * 2 * 8 + (gid & 1);

  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [row tile][row gid, gid + 8]
  unsigned long long best = 0ull;  // argmax key (0 < any real key)
  float rsc = 1.f;
  float seg_r[2] = {1.f, 1.f};  // per-half scales of the first phase (kPreEmbedPack)
  int cur = -1;
  unsigned done_here = 0;  // tiles of phase cur finished by this warp
  bool dead = false;
  int i = 0;
  for (; cc.ph < sp.nphase; ++i) {
    const int slot = i % S;
    if (cc.ph != cur) {
      // entering phase cc.ph: its input is the previous phase's output (or
      // the pre-units' output for phase 0)
      if (cc.ph > 0 || sp.pre.kind != kPreNone) {
        bool ok = true;
        if (lane == 0) {
          const unsigned polls = wait_polls(sp.err, kPhaseSpinLimit);
          if (cc.ph > 0) {
            const GemvParams& pp = sp.ph[cc.ph - 1];
            ok = wait_count(sp.phase_done + cc.ph - 1, (unsigned)pp.seg[pp.nseg - 1].tile_end,
                            polls);
          } else {
            ok = wait_count(sp.phase_done + kMaxPhases, (unsigned)sp.pre.units, polls);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          if (lane == 0) set_dev_error(sp.err, kErrPhaseTimeout);
          dead = true;
          break;
        }
      }
      cur = cc.ph;
      if (lane == 0) {
        fence_proxy_async_global();  // the copies below read what the wait acquired
        ready = cur;
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2)
          if (pend[s2] && pend_c[s2].ph <= ready) {
            issue_x(pend_c[s2], s2);
            pend[s2] = false;
          }
      }
      float r[1][2];
      row_scales<1>(sp.ph[cur], 1, tq, true, r);
      rsc = r[0][0];
      if (cur == 0 && sp.pre.kind == kPreEmbedPack) {
        // the two halves' RMSNorm scales, applied per unit (units never straddle)
        const int gpr = sp.pre.dim / kGroup;
        const float s0 = warp_col_sum(sp.pre.ss, gpr, 1, 0);
        const float s1 = warp_col_sum(sp.pre.ss + gpr, gpr, 1, 0);
        seg_r[0] = rsqrtf(s0 / (float)sp.pre.dim + sp.pre.eps);
        seg_r[1] = rsqrtf(s1 / (float)sp.pre.dim + sp.pre.eps);
      }
    }
    if (!mbar_wait_bounded(&bars[slot], (uint32_t)((i / S) & 1))) {
      if (lane == 0) set_dev_error(sp.err, kErrMbarTimeout);
      dead = true;
      break;
    }
    {
      const bool stage_bf = SBF && ((sp.ph[cc.ph].sbf_mask >> stage_slot(sp.ph[cc.ph], cc.c)) & 1);
      const uint8_t* ct = code_base + slot * kRowCode;
      const uint8_t* rs = rest_base + slot * kRowRest;
      const uint4* xps = reinterpret_cast<const uint4*>(rs + 2048);
      const float4 sxv = *reinterpret_cast<const float4*>(rs + 2048 + 1024 + tq * 16);
      const uint4* bsrc = b_active ? xps + b_off : zero_b;
      uint4 B[2][4];
#pragma unroll
      for (int st = 0; st < 2; ++st)
#pragma unroll
        for (int w = 0; w < 4; ++w) B[st][w] = bsrc[st * 8 + w * 2];
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        // rows rt*16 + gid and + 8: 16-byte chunk 2tq + st, 128B-swizzled
        const uint8_t* rp = ct + rt * 2048 + gid * 128;
        uint4 Wc[2][2];
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          Wc[0][st] = *reinterpret_cast<const uint4*>(rp + a_chunk[st]);
          Wc[1][st] = *reinterpret_cast<const uint4*>(rp + 1024 + a_chunk[st]);
        }
        float2 s0, s1, b0, b1;
        if (SBF && stage_bf) {  // [32 rows][8 groups] bfloat16, biases 1 KB further
          const __nv_bfloat16* sh = reinterpret_cast<const __nv_bfloat16*>(rs) +
                                    (rt * 16 + gid) * 8 + 2 * tq;
          s0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sh));
          s1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sh + 64));
          b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sh + 512));
          b1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sh + 512 + 64));
        } else {
          const float* sr = reinterpret_cast<const float*>(rs) + (rt * 16 + gid) * 8 + 2 * tq;
          s0 = *reinterpret_cast<const float2*>(sr);
          s1 = *reinterpret_cast<const float2*>(sr + 64);
          b0 = *reinterpret_cast<const float2*>(sr + 256);
          b1 = *reinterpret_cast<const float2*>(sr + 256 + 64);
        }
        float d[2][4];
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          d[st][0] = d[st][1] = d[st][2] = d[st][3] = 0.f;
          const uint32_t w0[4] = {Wc[0][st].x, Wc[0][st].y, Wc[0][st].z, Wc[0][st].w};
          const uint32_t w1[4] = {Wc[1][st].x, Wc[1][st].y, Wc[1][st].z, Wc[1][st].w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t x0 = w0[w], x1 = w1[w];
            mma_f16_16816(d[st], codes_lo_f16x2(x0), codes_lo_f16x2(x1), codes_hi_f16x2(x0),
                          codes_hi_f16x2(x1), B[st][w].x, B[st][w].y);
            const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
            mma_f16_16816(d[st], codes_lo_f16x2(y0), codes_lo_f16x2(y1), codes_hi_f16x2(y0),
                          codes_hi_f16x2(y1), B[st][w].z, B[st][w].w);
          }
        }
        // (sxv: the two groups' sums and power-of-two scales)
        acc[rt][0] = fmaf(s0.x * sxv.y, d[0][0] + d[0][1], fmaf(b0.x, sxv.x, acc[rt][0]));
        acc[rt][0] = fmaf(s0.y * sxv.w, d[1][0] + d[1][1], fmaf(b0.y, sxv.z, acc[rt][0]));
        acc[rt][1] = fmaf(s1.x * sxv.y, d[0][2] + d[0][3], fmaf(b1.x, sxv.x, acc[rt][1]));
        acc[rt][1] = fmaf(s1.y * sxv.w, d[1][2] + d[1][3], fmaf(b1.y, sxv.z, acc[rt][1]));
      }
    }
    __syncwarp();
    if (lane == 0 && pc.ph < sp.nphase) {  // refill the slot
      issue_w(pc, slot);
      if (pc.ph <= ready)
        issue_x(pc, slot);
      else
        defer_x(pc, slot);
      ++issued;
      phase_advance(sp, pc, gw);
    }

    const int ph = cc.ph;
    const int unit = cc.c.u, tile = cc.c.tile, seg = cc.c.seg;
    const int unit_ks = cc.c.ks;  // a stage of the unit (for the per-half scale)
    if (!phase_advance(sp, cc, gw)) continue;

    // ------------------------------------------------------------ unit done
    // a row's four lanes each hold two groups per stage: sum them in a fixed
    // order; then lane (gid, tq) keeps tile row rr (one row per lane)
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = acc[rt][e];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        acc[rt][e] = v;
      }
    const int rr = (tq >> 1) * 16 + (tq & 1) * 8 + gid;
    float g = (tq & 2) ? ((tq & 1) ? acc[1][1] : acc[1][0]) : ((tq & 1) ? acc[0][1] : acc[0][0]);
    acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
    const GemvParams& p = sp.ph[ph];
    const GemvSeg& sg = p.seg[seg];
    const int lt = tile - (seg ? p.seg[seg - 1].tile_end : 0);
    const int row = lt * 32 + rr;
    const bool row_ok = row < sg.n;
    // what the epilogue reads, loaded before the split-K round trips
    float resv = 0.f, pw = 0.f;
    if (p.epi == kEpiStore && row_ok) {
      if (sg.res) resv = __ldcg(sg.res + sg.out_col0 + row);
      if (p.pack_w) pw = __ldg(p.pack_w + sg.out_col0 + row);
    }
    if (ph == 0 && sp.pre.kind == kPreEmbedPack)
      g *= seg_r[unit_ks * 8 >= sp.pre.dim / kGroup ? 1 : 0];
    float u = 0.f;
    bool fin = true;
    if (p.ksplit > 1 || p.um > 1) {
      // deterministic split-K (and gate/up pairing): each unit stores its 32
      // rows; the last of the tile's units sums them in k order
      p.part[(size_t)unit * 32 + lane] = g;
      __syncwarp();  // the warp's partial, then one acquire-release count by lane 0
      unsigned prev = 0;
      if (lane == 0) prev = atom_add_acq_rel_gpu(p.tile_cnt + tile, 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      fin = prev == (unsigned)(p.um * p.ksplit) - 1;
      if (fin) {
        const float* src = p.part + (size_t)tile * p.um * p.ksplit * 32 + lane;
        g = sum_rows(src, p.ksplit);
        if (p.um > 1) u = sum_rows(src + (size_t)p.ksplit * 32, p.ksplit);
        if (lane == 0) p.tile_cnt[tile] = 0u;  // leave the counter cleared
      }
    }
    if (fin) {
      // undo the 2^-24 of the subnormal codes (exact), apply a folded RMSNorm
      g *= kCodeScale * rsc;
      u *= kCodeScale * rsc;
      const int g_out = (sg.out_col0 + lt * 32) / kGroup;
      if (p.epi == kEpiStore) {
        const float v = g + resv;
        if (row_ok) sg.out[sg.out_col0 + row] = v;
        if (p.pack_w) {  // full tiles (checked by the host)
          const float2 hs = xp_store_group(p.out_xp, 1, g_out, 0, rr, v * pw);
          const float q2 = warp_sum(v * v);
          if (lane == 0) {
            p.out_xs[g_out] = hs;
            p.ss_out[lt] = q2;
          }
        }
      } else if (p.epi == kEpiSwiglu) {
        const float scale = sg.w_idx >= 0 ? p.segw[sg.w_idx] : 1.f;
        const float hv = g / (1.f + __expf(-g)) * u * scale;
        const float2 hs = xp_store_group(p.out_xp, 1, g_out, 0, rr, hv);
        if (sg.out) sg.out[sg.out_col0 + lt * 32 + rr] = hv;
        if (lane == 0) p.out_xs[g_out] = hs;
      } else {
        if (row_ok) {
          if (p.logits) p.logits[row] = g;
          const unsigned long long key = argmax_key(g, row);
          best = key > best ? key : best;
        }
        // the first K / 32 tiles also write the normed input row, 32 values each
        const int kn = lt * 32 + lane;
        if (p.normed_out && kn < p.K)
          p.normed_out[kn] = __ldcg(p.normed_src + kn) * rsc * p.normed_w[kn];
      }
      ++done_here;
    }
    if (cc.ph != ph) {
      // leaving phase ph: publish this warp's finished tiles (one release
      // per warp and phase); the launch's last tile clears the counters
      __syncwarp();
      if (lane == 0 && done_here > 0) {
        const unsigned tiles = (unsigned)p.seg[p.nseg - 1].tile_end;
        if (ph == sp.nphase - 1) {
          const unsigned prev = atom_add_acq_rel_gpu(sp.phase_done + ph, done_here);
          if (prev + done_here == tiles)
            for (int q = 0; q <= kMaxPhases; ++q) sp.phase_done[q] = 0u;  // every wait has passed
        } else {
          red_add_release_gpu(sp.phase_done + ph, done_here);
        }
      }
      done_here = 0;
    }
  }

  if (dead) {
    // make every issued stage complete before the CTA can exit: issue the
    // activations still pending (their inputs may be incomplete; the results
    // are discarded), then wait for the stages not yet consumed
    const int n_issued = __shfl_sync(0xffffffffu, issued, 0);
    if (lane == 0)
#pragma unroll
      for (int s2 = 0; s2 < S; ++s2)
        if (pend[s2]) issue_x(pend_c[s2], s2);
    __syncwarp();
    for (int j = i; j < n_issued; ++j) mbar_wait_bounded(&bars[j % S], (uint32_t)((j / S) & 1));
  }
  if (sp.ph[sp.nphase - 1].epi == kEpiArgmax) argmax_finish(sp.ph[sp.nphase - 1], best);
}

// Plain CUDA-core fallback for shapes the TMA path cannot describe
// (K % 128 != 0 or unaligned rows): one warp per output row.
__global__ void gemv_simple_kernel(const float* __restrict__ x, int m, int K,
                                   const uint32_t* __restrict__ q, const float* __restrict__ s,
                                   const float* __restrict__ b, int N, float* __restrict__ y);

}  // namespace mtp
