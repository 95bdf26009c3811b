// Host-side internals shared by the entry points (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "../../include/mtpdraft.h"
#include "gemv.cuh"

namespace mtp {

// Records a thread-local error message and returns `st`.
mtp_status fail(mtp_status st, const std::string& msg);
mtp_status cuda_fail(cudaError_t e, const char* what);

bool aligned16(const void* p);

// Records the next event of this thread's launch-timing session (if one is
// open) on `st`; every launcher calls it right before its kernel launch.
void launch_mark(cudaStream_t st);

// Number of SMs of the current device (cached per device).
int sm_count();

// Encodes the three tensor maps of an affine weight viewed as [rows][k].
// With sb_bf16 the scales and biases are bfloat16 [rows][k/32] (rows of 2k/32
// bytes, a multiple of 16 when k % 256 == 0).
mtp_status encode_qmat(QMat* out, const mtp_affine4& w, const char* name, bool sb_bf16 = false);

// Checks an affine weight descriptor: non-null, aligned, positive sizes,
// k % 32 == 0, and (when `need_tma`) k % 128 == 0 so the scale rows are
// 16-byte aligned for the tensor maps.
mtp_status check_affine(const mtp_affine4* w, int n, int k, const char* name, bool need_tma);

// Workspace regions a GEMV launch may use for split-K partial sums.
struct GemvScratch {
  float* part;          // partial fragments
  size_t part_bytes;
  unsigned* cnt;        // per-tile completion counters (cleared)
  int cnt_len;
  unsigned* phase_done; // [kMaxPhases + 1] per-phase tile and pre-unit counters of the one-row kernel (cleared)
};
size_t gemv_scratch_part_bytes();
constexpr int kGemvCounters = 4096;

// Launch helpers (programmatic dependent launch on `stream`).  Fills in the
// split-K plan of `p` (ksplit, spu, part, tile_cnt) from the scratch given.
// One-row (m = 1) projections in order in one launch: phase q reads its
// activation row only after every tile of phase q - 1 is written.
cudaError_t launch_gemv_rows(GemvParams* ph, const int* tiles, int nphase,
                             const GemvScratch& sc, int* err, cudaStream_t st,
                             const PreParams* pre = nullptr);
cudaError_t launch_gemv(int nmat, int nt, int epi, GemvParams p, int tiles,
                        const GemvScratch& scratch, cudaStream_t stream);
cudaError_t launch_pack(const float* x, int m, int K, uint4* xp, float2* xs, cudaStream_t st);
cudaError_t launch_gemv_simple(const float* x, int m, int K, const mtp_affine4& w, float* y,
                               cudaStream_t st);
// In-place multiplier/softcap of rows x V logits and each row's argmax;
// keys[rows] and cnt[rows] are zero at rest and left zero.
cudaError_t launch_rows_argmax(float* logits, int rows, int V, float mult, float cap, int32_t* tok,
                               float* val, unsigned long long* keys, unsigned* cnt,
                               cudaStream_t st);

struct NormSeg {
  const float* src;       // row 0 source (row stride = src_ld); null when gathered from `table`
  const float* delta;     // residual added to src (same layout), or null
  const float* table;     // embedding table [V][dim] gathered with tokens[c]
  const int* tokens;
  int vocab;
  const float* w;         // norm weight, or null (no normalisation)
  float eps;
  int dim;
  int src_ld;
  float* out_sum;         // fp32 sum (ld = dim), or null
  float* out_norm;        // fp32 normalised row (ld = dim), or null
};

// Normalises m rows (up to two segments concatenated along K) and writes
// the packed activations of the concatenation (xp may be null).
cudaError_t launch_norm_pack(const NormSeg* segs, int nseg, int m, uint4* xp, float2* xs,
                             int* err, cudaStream_t st);

// Tensor map over bf16 rows [rows][cols] with boxes of box_rows x 64 values
// (128 bytes), 128-byte swizzle (the tcgen05 K-major operand layout).
cudaError_t encode_bf16_rows_map(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols,
                                 int box_rows);

// Tensor map over float rows [rows][cols] with boxes of box_rows x 32 floats,
// 128-byte swizzle.
cudaError_t encode_f32_tile_map(CUtensorMap* out, const float* base, uint64_t rows, uint64_t cols,
                                int box_rows);

struct alignas(64) AttnParams {
  CUtensorMap kmap;     // K cache viewed as [n_kv * cap][dqk]
  CUtensorMap vmap;     // V cache viewed as [n_kv * cap][dv] (tensor-core tile path)
  int nh, nkv, dqk, dv, rot, window, gated;
  float eps, scale;
  const float *qp, *kp, *vp, *qn, *kn, *rope, *sinks;
  float *kc, *vc;
  int L, cap, m;
  int pos_base;        // rotary position of cache row 0
  float* out;          // [m][nh*dv] fp32 (may be null)
  uint4* out_xp;       // packed output for the next projection (may be null)
  float2* out_xs;
  float* part;         // partials
  unsigned* counters;  // [2 * nkv] arrivals, departures
  int nsplit;
  int nbuf;            // tile buffers per CTA (set by launch_attn)
  int qgroups;         // warps per buffer, each with a slice of the query rows (set by launch_attn)
  // 1: stream cached rows before waiting on the previous kernel.  Only valid
  // when that kernel signals its dependents after its own wait (so every
  // earlier kernel, including the step that wrote those rows, has finished).
  int prefetch_before_wait;
  // 1: the splits merge the output in this kernel; 0: they only write their
  // partials (the next launch merges them, m = 1)
  int merge_in_kernel;
  int* err;
};
// Start of the split outputs inside the partials buffer.
const float* attn_part_outputs(const float* part, int nkv, int nsplit, int q_per_kv);
// Split count for `cached` keys inside the window, and an upper bound of it
// that grows with `cached` (sizes the partials).
int attn_splits(int nkv, int cached, int q_rows_per_kv, int dqk, int dv, int m);
int attn_splits_bound(int nkv, int cached);
// Whether one CTA can serve QG query rows of the given head dims and m.
bool attn_supported(int QG, int dqk, int dv, int m);
size_t attn_part_bytes(int nkv, int nsplit, int q_per_kv, int dv);
cudaError_t launch_attn(const AttnParams& a, cudaStream_t st);

struct RouterParams {
  const float* u1;       // [H] residual stream row
  const float* post_norm;
  float eps;
  int H;
  const float* router;   // [E][H]
  int E, top_k;
  const float* sh_gate_inp;  // [H] or null
  float* logits;         // [E] scratch
  unsigned* counter;
  int* sel;              // [top_k]
  float* weight;         // [top_k + 1]
  uint4* xp;             // packed normalised row for the expert projections
  float2* xs;
  int* err;
  int rows_per_cta;      // set by launch_router
};
cudaError_t launch_router(const RouterParams& r, cudaStream_t st);

cudaError_t launch_rope_table(float* d, int max_pos, int rot, double theta, cudaStream_t st);

}  // namespace mtp
