// Affine 4-bit GEMV/skinny-GEMM kernels and their host launchers.
#include <cudaTypedefs.h>

#include <mutex>

#include "host.h"

namespace mtp {

// --------------------------------------------------------------- fallback
__global__ void gemv_simple_kernel(const float* __restrict__ x, int m, int K,
                                   const uint32_t* __restrict__ q, const float* __restrict__ s,
                                   const float* __restrict__ b, int N, float* __restrict__ y) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  if (warp >= N) return;
  const int n = warp;
  const int KW = K / 8;
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;
  for (int kw = lane; kw < KW; kw += 32) {
    const uint32_t word = q[(size_t)n * KW + kw];
    const int g = kw / 4;
    const float sc = s[(size_t)n * (K / kGroup) + g];
    const float bi = b[(size_t)n * (K / kGroup) + g];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = fmaf(sc, (float)((word >> (4 * i)) & 0xFu), bi);
      const int k = kw * 8 + i;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c < m) acc[c] = fmaf(x[(size_t)c * K + k], w, acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    if (c < m) {
      const float v = warp_sum(acc[c]);
      if (lane == 0) y[(size_t)c * N + n] = v;
    }
  }
}

// --------------------------------------------------------------- packing
// One thread per (group, column, octet); the four octets of a group are
// adjacent lanes and combine their sums with two shuffles.
__global__ void pack_x_kernel(const float* __restrict__ x, int m, int K, uint4* __restrict__ xp,
                              float2* __restrict__ xs) {
  pdl_launch_dependents();  // the projection that follows only reads weights before its wait
  pdl_wait();
  const int G = K / kGroup;
  const int total = G * m * 4;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = i < total;
  const int t = i & 3;
  const int gc = i >> 2;
  const int c = gc % m;
  const int g = gc / m;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (valid) {
    const float4* src = reinterpret_cast<const float4*>(x + (size_t)c * K + g * kGroup + t * 8);
    const float4 v0 = src[0], v1 = src[1];
    v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
    v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
  }
  uint4 hi, lo;
  const float2 gx = pack8_group(v, valid, hi, lo);
  if (valid) {
    xp[xp_index(g, c, t, 0, m)] = hi;
    xp[xp_index(g, c, t, 1, m)] = lo;
    if (t == 0) xs[g * m + c] = gx;
  }
}

// --------------------------------------------------------------- launchers
static cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Split-K plan: units of `spu` stages; a split is only used when all its
// units fit in one round of the resident warps, and the plan minimises the
// stages on a warp's critical path (plus a small cost per partial).
struct Plan {
  int ksplit, spu, units;
};
// kalign > 0: units must not straddle a multiple of kalign stages.
// split_rounds > 1: a split may take up to that many rounds of the warps (a
// tile's k chunks then run on different warps in different rounds); such a
// plan must beat the others by a margin (its partials and combines cost
// more than the model counts).
static Plan plan_split(int tiles, int KS, int warps_cap, int nacc, int um,
                       const GemvScratch& sc, int kalign = 0, int split_rounds = 1) {
  Plan best = {0, 0, 0};
  double best_cost = 1e30;
  for (int spu = KS; spu >= 1; --spu) {
    if (kalign > 0 && kalign % spu) continue;
    const int ksplit = (KS + spu - 1) / spu;
    if (ksplit > 1 && spu * (ksplit - 1) >= KS) continue;  // same split as a larger spu
    const long long units = (long long)tiles * um * ksplit;
    if (ksplit > 1 || um > 1) {
      if (ksplit > 1 && units > (long long)warps_cap * split_rounds) continue;
      if (tiles > sc.cnt_len) continue;
      if ((size_t)units * 32 * nacc * sizeof(float) > sc.part_bytes) continue;
    }
    const long long rounds = (units + warps_cap - 1) / warps_cap;
    double cost = (double)rounds * spu + (ksplit > 1 ? 1.0 + 0.15 * ksplit : 0.0);
    if (ksplit > 1 && rounds > 1) cost += 0.1 * rounds * spu;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = {ksplit, spu, (int)units};
    }
  }
  return best;
}

// Rounds of warps a split-K plan of the one-row kernel may take (tuning
// knob; 2 lets the Qwen-style gate/up phase, 1088 tiles x 20 stages, run as
// 3 k chunks over two rounds of every warp instead of one chunk on 1088).
#ifndef MTP_ROW_SPLIT_ROUNDS
#define MTP_ROW_SPLIT_ROUNDS 2
#endif
constexpr int kRowSplitRounds = MTP_ROW_SPLIT_ROUNDS;

size_t gemv_scratch_part_bytes() {
  // one round of resident warps (at most 16 per SM) x 32 lanes x 32 floats
  return (size_t)sm_count() * 16 * 32 * 32 * sizeof(float);
}

// Stage depth of each warp's pipeline (compile-time tuning knob).
#ifndef MTP_GEMV_STAGES
#define MTP_GEMV_STAGES 2
#endif

#ifndef MTP_TC_PC_XM
#define MTP_TC_PC_XM 4
#endif
constexpr int kTcPcXm = MTP_TC_PC_XM;
#ifndef MTP_TC_STAGES
#define MTP_TC_STAGES MTP_GEMV_STAGES
#endif
// Shared-memory carveout (percent of the maximum) of the tensor-core kernels
// that read activations through L1, and a cap on their CTAs per SM (tuning
// knobs; -1 / 0: the driver's choice).
#ifndef MTP_TC_CARVEOUT
#define MTP_TC_CARVEOUT -1
#endif
#ifndef MTP_TC_MAX_CTAS
#define MTP_TC_MAX_CTAS 0
#endif
template <int NMAT, int NT, int EPI, int XM, bool PAIRED = false, bool PC = false>
static cudaError_t launch_gemv_t(GemvParams p, int tiles, const GemvScratch& sc,
                                 cudaStream_t st) {
  constexpr int S = MTP_TC_STAGES;
  auto kern = gemv_tc_kernel<NMAT, NT, EPI, S, XM, PAIRED, PC>;
  const int smem = gemv_smem_bytes<NMAT, S, XM>();
  static thread_local int configured_dev = -1;
  static thread_local int ctas_per_sm = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (XM == 0 && MTP_TC_CARVEOUT >= 0) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               MTP_TC_CARVEOUT);
      if (e != cudaSuccess) return e;
    }
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kGemvWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (XM == 0 && MTP_TC_MAX_CTAS > 0 && nb > MTP_TC_MAX_CTAS) nb = MTP_TC_MAX_CTAS;
    ctas_per_sm = nb > 0 ? nb : 1;
    configured_dev = dev;
  }
  const int warps_cap = sm_count() * ctas_per_sm * kGemvWarps;
  const int KS = (p.K / kGroup + 7) / 8;
  const Plan pl = plan_split(tiles, KS, warps_cap, NMAT * 2 * NT * 4, PAIRED ? 2 : 1, sc);
  if (pl.ksplit == 0) return cudaErrorInvalidValue;  // scratch too small for the split
  p.ksplit = pl.ksplit;
  p.spu = pl.spu;
  p.part = sc.part;
  p.tile_cnt = sc.cnt;
  int warps = pl.units < warps_cap ? pl.units : warps_cap;
  int grid = (warps + kGemvWarps - 1) / kGemvWarps;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr = pdl_attr();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool SBF>
static cudaError_t launch_gemv_rows_t(GemvParams* ph, const int* tiles, int nphase,
                                      const GemvScratch& sc, int* err, cudaStream_t st,
                                      const PreParams* pre) {
  constexpr int S = MTP_GEMV_STAGES;
  auto kern = gemv_row_kernel<S, SBF>;
  const int smem = kGemvWarps * S * (kRowCode + kRowRest) + 2048;  // + barriers, alignment
  static_assert(sizeof(StreamParams) <= 32764, "kernel parameters fit the 32 KB limit");
  if (nphase < 1 || nphase > kMaxPhases) return cudaErrorInvalidValue;
  static thread_local int configured_dev = -1;
  static thread_local int ctas_per_sm = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kGemvWarps * 32, smem);
    if (e != cudaSuccess) return e;
    ctas_per_sm = nb > 0 ? nb : 1;
    configured_dev = dev;
  }
  // every CTA must be resident at once (phases wait on each other's tiles)
  const int warps_cap = sm_count() * ctas_per_sm * kGemvWarps;
  StreamParams sp = {};
  int max_units = 1;
  int units_q[kMaxPhases];
  for (int q = 0; q < nphase; ++q) {
    GemvParams& p = ph[q];
    if (p.m != 1 || (q + 1 < nphase && p.epi == kEpiArgmax)) return cudaErrorInvalidValue;
    const int um = p.epi == kEpiSwiglu ? 2 : 1;
    const int KS = (p.K / kGroup + 7) / 8;
    // with packed halves (kPreEmbedPack) the first phase's units stay in one half
    const int kalign = (q == 0 && pre && pre->kind == kPreEmbedPack) ? pre->dim / 256 : 0;
    const Plan pl = plan_split(tiles[q], KS, warps_cap, 1, um, sc, kalign,
                               kRowSplitRounds);  // 32 floats per unit
    if (pl.ksplit == 0) return cudaErrorInvalidValue;  // scratch too small for the split
    p.um = um;
    p.ksplit = pl.ksplit;
    p.spu = pl.spu;
    p.part = sc.part;
    p.tile_cnt = sc.cnt;
    p.err = err;
    units_q[q] = pl.units;
    if (pl.units > max_units) max_units = pl.units;
    sp.ph[q] = p;
  }
  sp.nphase = nphase;
  sp.phase_done = sc.phase_done;
  sp.err = err;
  if (pre) sp.pre = *pre;
  const int warps = max_units < warps_cap ? max_units : warps_cap;
  // each phase spreads its units evenly: ceil(units / warps) rounds on as
  // few warps as that number of rounds needs (a part-filled last round runs
  // the stream on fewer warps than it needs for full bandwidth)
  for (int q = 0; q < nphase; ++q) {
    const int rounds = (units_q[q] + warps - 1) / warps;
    sp.ph[q].wq = (units_q[q] + rounds - 1) / rounds;
  }
  const int grid = (warps + kGemvWarps - 1) / kGemvWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr = pdl_attr();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, kern, sp);
}

cudaError_t launch_gemv_rows(GemvParams* ph, const int* tiles, int nphase,
                             const GemvScratch& sc, int* err, cudaStream_t st,
                             const PreParams* pre) {
  bool sbf = false;
  for (int q = 0; q < nphase && q < kMaxPhases; ++q) sbf = sbf || ph[q].sbf_mask != 0;
  return sbf ? launch_gemv_rows_t<true>(ph, tiles, nphase, sc, err, st, pre)
             : launch_gemv_rows_t<false>(ph, tiles, nphase, sc, err, st, pre);
}

cudaError_t launch_gemv(int nmat, int nt, int epi, GemvParams p, int tiles,
                        const GemvScratch& sc, cudaStream_t st) {
  const int m = p.m;
  if (m == 1) {  // one activation row: the one-row kernel, a single phase
    if ((epi == kEpiSwiglu) != (nmat == 2) || nt != 1) return cudaErrorInvalidValue;
    p.epi = epi;
    return launch_gemv_rows(&p, &tiles, 1, sc, p.err, st);
  }
  if (epi == kEpiArgmax) return cudaErrorInvalidValue;
  // 2-4 rows: paired columns, activations staged per stage by bulk copy
  // (kTcPcXm = 4) or read through L1 (0); 5-16 rows: one column per row
  if (nmat == 1) {
    if (epi != kEpiStore) return cudaErrorInvalidValue;
    if (nt == 2) return launch_gemv_t<1, 2, kEpiStore, 0>(p, tiles, sc, st);
    if (m <= 4) return launch_gemv_t<1, 1, kEpiStore, kTcPcXm, false, true>(p, tiles, sc, st);
    return launch_gemv_t<1, 1, kEpiStore, 0>(p, tiles, sc, st);
  }
  // SwiGLU: gate (slot mat) and up (slot mat + 1) tiles are separate units
  if (epi != kEpiSwiglu) return cudaErrorInvalidValue;
  if (nt == 2) return launch_gemv_t<1, 2, kEpiSwiglu, 0, true>(p, tiles, sc, st);
  if (m <= 4) return launch_gemv_t<1, 1, kEpiSwiglu, kTcPcXm, true, true>(p, tiles, sc, st);
  return launch_gemv_t<1, 1, kEpiSwiglu, 0, true>(p, tiles, sc, st);
}

cudaError_t launch_pack(const float* x, int m, int K, uint4* xp, float2* xs, cudaStream_t st) {
  const int total = (K / kGroup) * m * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((total + 255) / 256);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr = pdl_attr();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, pack_x_kernel, x, m, K, xp, xs);
}

cudaError_t launch_gemv_simple(const float* x, int m, int K, const mtp_affine4& w, float* y,
                               cudaStream_t st) {
  const int threads = 256;
  const int blocks = (w.n * 32 + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = st;
  cudaLaunchAttribute attr = pdl_attr();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, gemv_simple_kernel, x, m, K, w.q, w.s, w.b, (int)w.n, y);
}

// --------------------------------------------------------------- row argmax
// Logits of `rows` rows [rows][V], in place: l *= mult, then
// l = cap * tanh(l / cap) when cap > 0; then each row's argmax (lowest index
// among equal maxima).  Block (x, r) takes a slice of row r; the last block
// of a row to finish writes its token and value and clears keys[r], cnt[r].
constexpr int kRowArgmaxThreads = 256;

__global__ void __launch_bounds__(kRowArgmaxThreads)
    rows_argmax_kernel(float* __restrict__ logits, int V, float mult, float cap,
                       int32_t* __restrict__ tok, float* __restrict__ val,
                       unsigned long long* keys, unsigned* cnt) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ unsigned long long red[kRowArgmaxThreads / 32];
  const int r = blockIdx.y;
  float* row = logits + (size_t)r * V;
  // slices of whole octets; a thread's octet is read with two 16-byte loads
  // when the row allows it (one round trip instead of one per logit)
  const int per = ((V + gridDim.x - 1) / gridDim.x + 7) / 8 * 8;
  const int v0 = blockIdx.x * per, v1 = min(V, v0 + per);
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  unsigned long long best = 0ull;  // below any real key
  for (int v8 = v0 + threadIdx.x * 8; v8 < v1; v8 += blockDim.x * 8) {
    float l[8];
    const bool full = vec && v8 + 8 <= v1;
    if (full) {
      const float4 a = *reinterpret_cast<const float4*>(row + v8);
      const float4 b = *reinterpret_cast<const float4*>(row + v8 + 4);
      l[0] = a.x; l[1] = a.y; l[2] = a.z; l[3] = a.w;
      l[4] = b.x; l[5] = b.y; l[6] = b.z; l[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) l[i] = v8 + i < v1 ? row[v8 + i] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      l[i] *= mult;
      if (cap > 0.f) l[i] = cap * tanhf(l[i] / cap);
    }
    if (full) {
      *reinterpret_cast<float4*>(row + v8) = make_float4(l[0], l[1], l[2], l[3]);
      *reinterpret_cast<float4*>(row + v8 + 4) = make_float4(l[4], l[5], l[6], l[7]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (v8 + i < v1) {
        if (!full) row[v8 + i] = l[i];
        const unsigned long long k = argmax_key(l[i], v8 + i);
        best = k > best ? k : best;
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
    best = other > best ? other : best;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kRowArgmaxThreads / 32; ++w) best = red[w] > best ? red[w] : best;
    if (best) atomicMax(keys + r, best);
    __threadfence();
    const unsigned prev = atomicAdd(cnt + r, 1u);
    if (prev == gridDim.x - 1) {  // every block of the row has merged its key
      __threadfence();
      const unsigned long long k = atomicMax(keys + r, 0ull);
      tok[r] = argmax_key_index(k);
      val[r] = argmax_key_value(k);
      keys[r] = 0ull;  // leave the workspace cleared for the next call
      cnt[r] = 0u;
    }
  }
}

cudaError_t launch_rows_argmax(float* logits, int rows, int V, float mult, float cap, int32_t* tok,
                               float* val, unsigned long long* keys, unsigned* cnt,
                               cudaStream_t st) {
  if (rows < 1 || rows > 65535 || V < 1) return cudaErrorInvalidValue;
  int blocks = (V + kRowArgmaxThreads * 8 - 1) / (kRowArgmaxThreads * 8);  // >= 8 logits a thread
  if (blocks > 1024) blocks = 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, rows);
  cfg.blockDim = dim3(kRowArgmaxThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr = pdl_attr();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_mark(cfg.stream);
  return cudaLaunchKernelEx(&cfg, rows_argmax_kernel, logits, V, mult, cap, tok, val, keys, cnt);
}

// --------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &ptr, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

static CUresult encode2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                         uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                         CUtensorMapSwizzle sw) {
  auto fn = get_encode();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

cudaError_t encode_f32_tile_map(CUtensorMap* out, const float* base, uint64_t rows, uint64_t cols,
                                int box_rows) {
  // rows of `cols` floats, box box_rows x 32 floats, 128-byte swizzle
  CUresult r = encode2d(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, cols, rows, cols * 4, 32,
                        (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_bf16_rows_map(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols,
                                 int box_rows) {
  // rows of `cols` bf16, box box_rows x 64 (128 bytes), 128-byte swizzle;
  // rows past `rows` read as zeros
  CUresult r = encode2d(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, cols, rows, cols * 2, 64,
                        (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

mtp_status encode_qmat(QMat* out, const mtp_affine4& w, const char* name, bool sb_bf16) {
  const uint64_t kw = (uint64_t)w.k / 8, kg = (uint64_t)w.k / kGroup;
  CUresult r = encode2d(&out->q, CU_TENSOR_MAP_DATA_TYPE_UINT32, w.q, kw, (uint64_t)w.n, kw * 4,
                        32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  const CUtensorMapDataType sdt = sb_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const uint64_t esz = sb_bf16 ? 2 : 4;
  if (r == CUDA_SUCCESS)
    r = encode2d(&out->s, sdt, w.s, kg, (uint64_t)w.n, kg * esz, 8, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (r == CUDA_SUCCESS)
    r = encode2d(&out->b, sdt, w.b, kg, (uint64_t)w.n, kg * esz, 8, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MTP_ERR_CUDA, std::string("tensor map encoding failed for ") + name +
                                  " (CUresult " + std::to_string((int)r) + ")");
  return MTP_OK;
}

}  // namespace mtp
