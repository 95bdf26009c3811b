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
// Two nibbles become one bf16x2 register with a single LOP3 (128 + code,
// exact), the dot products run on the tensor pipe against the activations
// split into bf16 hi + lo parts (fp32 accumulation), and the per-group scale
// and bias are applied in fp32 after each group:
//     y += s * D + (b - 128 s) * sum_group(x)          D = sum (128+code) x
// Activations arrive pre-packed ("xpack") in the B-fragment order with the
// per-group sums precomputed by the producer kernel.
#pragma once

#include "common.cuh"

namespace mtp {

// ------------------------------------------------------------------ xpack
// For activations X[m][K]: xp is uint4 [K/32][m][4][2] and xs float [K/32][m].
// Entry (g, c, t, hl): hl = 0 holds the bf16 "hi" parts, 1 the "lo" parts, of
// x[c][32g + 8t + p] for p in (0,4),(1,5),(2,6),(3,7) as bf16x2 words
// (first element in the low half).  xs[g][c] = sum over the group of hi + lo.
__host__ __device__ inline size_t xpack_bytes(int m, int K) {
  return (size_t)(K / kGroup) * m * 128 + (size_t)(K / kGroup) * m * 4;
}
__device__ __forceinline__ int xp_index(int g, int c, int t, int hl, int m) {
  return ((g * m + c) * 4 + t) * 2 + hl;
}

// Packs the eight values of (g, c, t); returns their hi+lo sum.
__device__ __forceinline__ float pack8(const float v[8], uint4& hi, uint4& lo) {
  __nv_bfloat16 h[8], l[8];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    split_bf16(v[i], h[i], l[i]);
    sum += __bfloat162float(h[i]) + __bfloat162float(l[i]);
  }
  auto pk = [](__nv_bfloat16 a, __nv_bfloat16 b) -> uint32_t {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
  };
  hi = make_uint4(pk(h[0], h[4]), pk(h[1], h[5]), pk(h[2], h[6]), pk(h[3], h[7]));
  lo = make_uint4(pk(l[0], l[4]), pk(l[1], l[5]), pk(l[2], l[6]), pk(l[3], l[7]));
  return sum;
}

// Position of element p (0..7) of an (g, c, t) octet inside its uint4:
// word p % 4, half p / 4.
__device__ __forceinline__ void xp_store_elem(uint4* xp, int m, int g, int c, int t, int p,
                                              float v, float* hilo_sum) {
  __nv_bfloat16 h, l;
  split_bf16(v, h, l);
  unsigned short* base = reinterpret_cast<unsigned short*>(xp);
  size_t w_hi = (size_t)xp_index(g, c, t, 0, m) * 8 + (p & 3) * 2 + (p >> 2);
  size_t w_lo = (size_t)xp_index(g, c, t, 1, m) * 8 + (p & 3) * 2 + (p >> 2);
  base[w_hi] = __bfloat16_as_ushort(h);
  base[w_lo] = __bfloat16_as_ushort(l);
  *hilo_sum = __bfloat162float(h) + __bfloat162float(l);
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
  const float* xs;
  int m;
  int K;                 // reduction length (concatenated length in K-segment mode)
  int nseg;
  GemvSeg seg[kMaxSeg];
  const int* rowsel;     // routed expert ids (device), or null
  const float* segw;     // routed weights (device), or null
  int rowsel_after_wait; // 1: rowsel is produced by the previous kernel
  // K-segment mode (MoE down projection): K = nkseg * kseg_len
  int kseg_len;          // 0: off
  int nkseg;
  int kseg_row_mult;
  int kseg_last_mat;     // < 0: every K segment is routed; else the last one reads this slot
  // SwiGLU pack target
  uint4* out_xp;
  float* out_xs;
  int out_m;
  // argmax
  unsigned long long* am_partial;  // [gridDim.x]
  unsigned* am_counter;
  int* am_token;
  float* am_value;
  float* logits;                    // optional fp32 logits
  int* err;
};

constexpr int kStageMatBytes = 6144;  // 4 KB codes + 1 KB scales + 1 KB biases
constexpr int kGemvWarps = 4;

template <int NMAT, int S>
constexpr int gemv_smem_bytes() {
  return kGemvWarps * S * NMAT * kStageMatBytes + 2048;  // + barriers + alignment slack
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

struct StageInfo {
  int seg, mat, row, kx, sx;
};

__device__ __forceinline__ int find_seg(const GemvParams& p, int tile) {
  int s = 0;
#pragma unroll 1
  while (s < p.nseg - 1 && tile >= p.seg[s].tile_end) ++s;
  return s;
}

__device__ __forceinline__ StageInfo stage_info(const GemvParams& p, int tile, int ks) {
  StageInfo si;
  si.seg = find_seg(p, tile);
  const GemvSeg& sg = p.seg[si.seg];
  const int lt = tile - (si.seg ? p.seg[si.seg - 1].tile_end : 0);
  if (p.kseg_len > 0) {
    const int spk = p.kseg_len / 256;
    const int kj = ks / spk;
    const int kin = ks - kj * spk;
    if (p.kseg_last_mat < 0 || kj < p.nkseg - 1) {
      si.mat = sg.mat;
      si.row = p.rowsel[kj] * p.kseg_row_mult + lt * 32;
    } else {
      si.mat = p.kseg_last_mat;
      si.row = lt * 32;
    }
    si.kx = kin * 32;
    si.sx = kin * 8;
  } else {
    si.mat = sg.mat;
    si.row = (sg.sel_idx >= 0 ? p.rowsel[sg.sel_idx] * sg.row_mult : 0) + lt * 32;
    si.kx = ks * 32;
    si.sx = ks * 8;
  }
  return si;
}

template <int NMAT, int NT, int EPI, int S>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_tc_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of each codes tile is required by the 128B swizzle.
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;
  const int tq = lane & 3;

  constexpr int kWarpBytes = S * NMAT * kStageMatBytes;
  uint8_t* wbase = smem + warp * kWarpBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kGemvWarps * kWarpBytes) + warp * S;

  const int G = p.K / kGroup;
  const int KS = (G + 7) / 8;
  const int W = gridDim.x * kGemvWarps;
  const int gw = warp * gridDim.x + blockIdx.x;
  const int total_tiles = p.seg[p.nseg - 1].tile_end;
  const int my_tiles = gw < total_tiles ? (total_tiles - gw + W - 1) / W : 0;
  const int total = my_tiles * KS;

  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncwarp();

  const uint64_t pol = l2_policy_evict_first();
  auto issue = [&](int i) {
    const int ti = i / KS;
    const int ks = i - ti * KS;
    const StageInfo si = stage_info(p, gw + ti * W, ks);
    const int slot = i % S;
    uint8_t* st = wbase + slot * NMAT * kStageMatBytes;
    mbar_arrive_expect_tx(&bars[slot], NMAT * kStageMatBytes);
#pragma unroll
    for (int mi = 0; mi < NMAT; ++mi) {
      const QMat& mt = p.mat[si.mat + mi];
      uint8_t* d = st + mi * kStageMatBytes;
      tma_load_2d(d, &mt.q, &bars[slot], si.kx, si.row, pol);
      tma_load_2d(d + 4096, &mt.s, &bars[slot], si.sx, si.row, pol);
      tma_load_2d(d + 5120, &mt.b, &bars[slot], si.sx, si.row, pol);
    }
  };

  // Weights never depend on the previous kernel: start streaming them before
  // waiting on it, unless the rows to stream are chosen by it.
  if (!p.rowsel_after_wait && lane == 0) {
    for (int i = 0; i < S && i < total; ++i) issue(i);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (p.rowsel_after_wait && lane == 0) {
    for (int i = 0; i < S && i < total; ++i) issue(i);
  }

  float acc[NMAT][2][NT][4];
  unsigned long long best = 0ull;  // argmax key (0 < any real key)

  int ti = 0, ks = 0;
  int tile = gw;
  int seg = total > 0 ? find_seg(p, tile) : 0;
#pragma unroll
  for (int mi = 0; mi < NMAT; ++mi)
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][rt][nt][e] = 0.f;

  for (int i = 0; i < total; ++i) {
    const int slot = i % S;
    if (!mbar_wait_bounded(&bars[slot], (uint32_t)((i / S) & 1))) {
      if (lane == 0) set_dev_error(p.err, kErrMbarTimeout);
      return;
    }
    const uint8_t* st = wbase + slot * NMAT * kStageMatBytes;
    const int gcount = min(8, G - ks * 8);
    const int gbase = ks * 8;

#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {  // pairs of groups
      if (2 * jp >= gcount) break;
      // B fragments (activations) for the two groups of this pair
      uint4 bh[2][NT], bl[2][NT];
      float xs0[2][NT], xs1[2][NT];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int g = gbase + 2 * jp + h;
        const bool gv = (2 * jp + h) < gcount;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int c = nt * 8 + gid;
          if (gv && c < p.m) {
            const uint4* src = p.xp + xp_index(g, c, tq, 0, p.m);
            bh[h][nt] = __ldg(src);
            bl[h][nt] = __ldg(src + 1);
          } else {
            bh[h][nt] = make_uint4(0, 0, 0, 0);
            bl[h][nt] = make_uint4(0, 0, 0, 0);
          }
          const int c0 = nt * 8 + 2 * tq;
          xs0[h][nt] = (gv && c0 < p.m) ? __ldg(p.xs + g * p.m + c0) : 0.f;
          xs1[h][nt] = (gv && c0 + 1 < p.m) ? __ldg(p.xs + g * p.m + c0 + 1) : 0.f;
        }
      }
#pragma unroll
      for (int mi = 0; mi < NMAT; ++mi) {
        const uint8_t* codes = st + mi * kStageMatBytes;
        const float* ssm = reinterpret_cast<const float*>(codes + 4096);
        const float* bsm = reinterpret_cast<const float*>(codes + 5120);
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
          // ldmatrix.x4: (rows 0-7, group 2jp), (rows 8-15, 2jp), (rows 0-7, 2jp+1), (rows 8-15, 2jp+1)
          const int mtx = lane >> 3, ri = lane & 7;
          const int row = rt * 16 + ri + 8 * (mtx & 1);
          const int jj = 2 * jp + (mtx >> 1);
          const uint32_t addr = smem_u32(codes + row * 128 + ((jj ^ ri) << 4));
          uint32_t w[4];
          ldmatrix_x4(w[0], w[1], w[2], w[3], addr);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (2 * jp + h >= gcount) break;
            const uint32_t wa = w[2 * h], wb = w[2 * h + 1];
            const uint32_t a0 = codes_to_bf16x2_biased(wa);
            const uint32_t a1 = codes_to_bf16x2_biased(wb);
            const uint32_t a2 = codes_to_bf16x2_biased(wa >> 4);
            const uint32_t a3 = codes_to_bf16x2_biased(wb >> 4);
            const uint32_t a4 = codes_to_bf16x2_biased(wa >> 8);
            const uint32_t a5 = codes_to_bf16x2_biased(wb >> 8);
            const uint32_t a6 = codes_to_bf16x2_biased(wa >> 12);
            const uint32_t a7 = codes_to_bf16x2_biased(wb >> 12);
            const int j = 2 * jp + h;
            const int r0 = rt * 16 + gid;
            const float s0 = ssm[r0 * 8 + j], s1 = ssm[(r0 + 8) * 8 + j];
            const float b0 = fmaf(-128.f, s0, bsm[r0 * 8 + j]);
            const float b1 = fmaf(-128.f, s1, bsm[(r0 + 8) * 8 + j]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float d[4] = {0.f, 0.f, 0.f, 0.f};
              mma_bf16_16816(d, a0, a1, a2, a3, bh[h][nt].x, bh[h][nt].y);
              mma_bf16_16816(d, a0, a1, a2, a3, bl[h][nt].x, bl[h][nt].y);
              mma_bf16_16816(d, a4, a5, a6, a7, bh[h][nt].z, bh[h][nt].w);
              mma_bf16_16816(d, a4, a5, a6, a7, bl[h][nt].z, bl[h][nt].w);
              float* a = acc[mi][rt][nt];
              a[0] = fmaf(s0, d[0], fmaf(b0, xs0[h][nt], a[0]));
              a[1] = fmaf(s0, d[1], fmaf(b0, xs1[h][nt], a[1]));
              a[2] = fmaf(s1, d[2], fmaf(b1, xs0[h][nt], a[2]));
              a[3] = fmaf(s1, d[3], fmaf(b1, xs1[h][nt], a[3]));
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + S < total) issue(i + S);

    if (++ks == KS) {
      // ---------------------------------------------------------- epilogue
      const GemvSeg& sg = p.seg[seg];
      const int lt = tile - (seg ? p.seg[seg - 1].tile_end : 0);
      const int rbase = lt * 32;
      if constexpr (EPI == kEpiStore) {
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int row = rbase + rt * 16 + gid + ((e & 2) ? 8 : 0);
              const int c = nt * 8 + 2 * tq + (e & 1);
              if (row < sg.n && c < p.m) {
                const size_t o = (size_t)c * sg.ld + sg.out_col0 + row;
                float v = acc[0][rt][nt][e];
                if (sg.res) v += sg.res[o];
                sg.out[o] = v;
              }
            }
      } else if constexpr (EPI == kEpiSwiglu) {
        const float scale = sg.w_idx >= 0 ? p.segw[sg.w_idx] : 1.f;
        const int g_out = (sg.out_col0 + rbase) / kGroup;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float part[2] = {0.f, 0.f};
#pragma unroll
          for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int rloc = rt * 16 + gid + ((e & 2) ? 8 : 0);
              const int c = nt * 8 + 2 * tq + (e & 1);
              const float gv = acc[0][rt][nt][e];
              const float uv = acc[1][rt][nt][e];
              const float hv = gv / (1.f + __expf(-gv)) * uv * scale;
              if (c < p.out_m) {
                float hs;
                xp_store_elem(p.out_xp, p.out_m, g_out, c, rloc >> 3, rloc & 7, hv, &hs);
                part[e & 1] += hs;
                if (sg.out) sg.out[(size_t)c * sg.ld + sg.out_col0 + rbase + rloc] = hv;
              }
            }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = part[e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            const int c = nt * 8 + 2 * tq + e;
            if (gid == 0 && c < p.out_m) p.out_xs[g_out * p.out_m + c] = v;
          }
        }
      } else {  // argmax over column 0 (one activation row)
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int row = rbase + rt * 16 + gid + ((e & 2) ? 8 : 0);
            if (tq == 0 && row < sg.n) {
              const float v = acc[0][rt][0][e];
              if (p.logits) p.logits[row] = v;
              const unsigned long long key = argmax_key(v, row);
              best = key > best ? key : best;
            }
          }
      }
#pragma unroll
      for (int mi = 0; mi < NMAT; ++mi)
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mi][rt][nt][e] = 0.f;
      ks = 0;
      ++ti;
      tile += W;
      if (ti < my_tiles) seg = find_seg(p, tile);
    }
  }

  if constexpr (EPI == kEpiArgmax) {
    __shared__ unsigned long long red[kGemvWarps];
    __shared__ bool last;
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
      __threadfence();
      const unsigned prev = atomicAdd(p.am_counter, 1u);
      last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (last) {
      __threadfence();
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
}

// Plain CUDA-core fallback for shapes the TMA path cannot describe
// (K % 128 != 0 or unaligned rows): one warp per output row.
__global__ void gemv_simple_kernel(const float* __restrict__ x, int m, int K,
                                   const uint32_t* __restrict__ q, const float* __restrict__ s,
                                   const float* __restrict__ b, int N, float* __restrict__ y);

}  // namespace mtp
