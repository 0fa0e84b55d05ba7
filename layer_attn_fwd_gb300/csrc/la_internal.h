// la_internal.h -- contract between the C-ABI layer (la_api.cu) and the kernel
// translation units.  Host code only passes plain structs and CUtensorMaps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layerattn.h"

// The checked build (-DLA_CHECKED=1) adds buffer extents to the kernel
// arguments and bounds checks to every global store (la_device.cuh).
#ifndef LA_CHECKED
#define LA_CHECKED 0
#endif

namespace la {

// Per-launch timing (la_profile_start / la_profile_stop): when on, every
// launch is bracketed by two CUDA events on its stream.  Both are no-ops
// otherwise.  prof_on(): recording is on (launches then run without
// programmatic serialization, so that no kernel overlaps the events of the
// one before it).
void prof_before(cudaStream_t st, const char* name);
void prof_after(cudaStream_t st);
bool prof_on();

// Every kernel of the library is launched here.  pdl: with programmatic
// stream serialization, so the grid may be scheduled while the previous grid
// in the stream is still running; it must call pdl_wait() before touching
// memory that grid produces or consumes.
template <typename... KArgs, typename... Args>
cudaError_t launch(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (pdl && !prof_on()) ? 1 : 0;
  prof_before(st, name);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  prof_after(st);
  return e;
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  return launch(name, kern, grid, block, smem, st, true, static_cast<Args&&>(args)...);
}

// Rows of one query tile (the M of every tcgen05 MMA here).
constexpr int kTileM = 128;

// Arguments of the attention kernel (everything but the tensor maps).
struct AttnArgs {
  void* o;                    // output base (unsplit launch)
  long long o_sb, o_sh, o_ss; // output strides in elements: batch, head, row
  float* part_o;              // split partials [splits][B*H][S_q][D] (split launch) or null
  float* part_lse;            // split log2-sum-exp [splits][B*H][S_q] or null
  const int32_t* kv_len;      // [B] or null
  int B, H, S_q, S_kv;
  int causal;
  float sl2;                  // softmax scale times log2(e)
  int num_qblk;               // query blocks (of rows_per_cta rows) per (b, h)
  int tiles_per_split;        // key tiles handled by one split
  int splits;                 // key-range splits (set by the launcher)
  int head_group;             // causal order: (b, h) pairs per group (>= 1; B*H = one group)
  unsigned long long* sched;  // persistent form: ticket word and done word, in the caller's workspace
  unsigned sched_gen;         // this launch's tag in the high half of both words (never 0)
  uint32_t* err;              // device error word
  int skip_loads;             // test hook: issue no TMA load, so every wait runs out
  int v_raw;                  // fp32, one key tile, one CTA per item: tm_v maps V itself and the kernel transposes it
#if LA_CHECKED
  long long o_elems;          // elements of the output buffer
  long long part_elems;       // elements of part_o (part_lse holds part_elems / D)
#endif
};

// Static launch shape of the attention kernel for a dtype and head dim.
struct AttnShape {
  int rows_per_cta;   // query rows per CTA
  int block_n;        // keys per tile
  int box_q_rows;     // TMA box rows for q
  int box_kv_rows;    // TMA box rows for k / v
  int box_cols;       // TMA box columns (one 128-byte swizzle row)
};
bool attn_shape(la_dtype dt, int D, AttnShape* s);

// Launch the attention kernel over its num_qblk * B*H * splits work items:
// one CTA per item when they fit on the SMs at once, or when a.sched is null
// (no workspace for the ticket words); otherwise the persistent form, one
// CTA per SM drawing items by ticket from a.sched.
cudaError_t launch_attn(la_dtype dt, int D, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const AttnArgs& a, int splits, cudaStream_t st);

// Merge split partials into o.
struct CombineArgs {
  const float* part_o;
  const float* part_lse;
  void* o;
  long long o_sb, o_sh, o_ss;
  int B, H, S_q, D, splits;
#if LA_CHECKED
  long long o_elems;  // elements of o
  uint32_t* err;      // device error word
#endif
};
cudaError_t launch_combine(la_dtype dt, const CombineArgs& a, cudaStream_t st);

// Batched transpose of 4-byte elements: dst[b][c][r] = src[b][r][c]; source
// rows of C elements, batches src_batch apart; destination rows of ld_dst
// elements, batches C*ld_dst apart.  pdl: launch with programmatic stream
// serialization, so that it may overlap the previous grid (it must touch
// nothing that grid writes; it waits for that grid before it exits, so the
// grids after it still see everything before it finished).
cudaError_t launch_transpose32(const void* src, long long src_batch, void* dst, long long ld_dst, long long batches,
                               int R, int C, cudaStream_t st, bool pdl = false);

// LayerNorm of M rows of d elements (d a multiple of 64, 16-byte aligned
// pointers), statistics in fp32.  pdl: as for launch_transpose32.  With
// stats non-null only the row statistics (mean, 1 / sqrt(var + eps)) are
// written there (y is not touched).
cudaError_t launch_layernorm(la_dtype dt, const void* x, const void* gamma, const void* beta, void* y, long long M,
                             int d, float eps, cudaStream_t st, bool pdl = false, float2* stats = nullptr);

// Copy k_src, v_src [B,H,rows,D] into k_dst, v_dst [B,H,S_max,D] at row `at`
// (keys only when v_src is null).
cudaError_t launch_kv_append(const void* k_src, const void* v_src, void* k_dst, void* v_dst, int B, int H,
                             int rows, int D, int S_max, int at, int elem_bytes, cudaStream_t st);

// Fused Q/K/V projection.
struct ProjArgs {
  const void* bias;
  void* q;
  void* k;
  void* v;
  int M, N, K;        // rows (B*S), output columns (3*d_model), d_model
  int S, H, D;
  float q_scale;
  uint32_t* err;
  int v_transposed;   // write V as V^T [B, H, D, S_pad] (fp32 sublayer) instead of [B, H, S, D]
  long long S_pad;    // row length of V^T
  // LayerNorm in front (the pre-norm block), or all null: per-row (mean,
  // 1 / sqrt(var + eps)) [M] and gamma, beta [K]; x is then the raw input
  const float2* ln_stats;
  const void* ln_gamma;
  const void* ln_beta;
#if LA_CHECKED
  long long qk_elems; // elements of each of q and k
  long long v_elems;  // elements of v, or of V^T
#endif
};
struct ProjShape {
  int block_n;        // output columns per tile (the wide tile or 128)
  int box_cols;       // TMA box columns (one 128-byte swizzle row)
  int box_k_rows;     // TMA box rows of the weight tile (= K per stage)
  bool w_transposed;  // the weight is read as Wqkv^T [3d, d] (TF32: K-major only)
};
// Shape of a projection launch over an M x N output on `sms` SMs.
bool proj_shape(la_dtype dt, long long M, long long N, int sms, ProjShape* s);
// The persistent projection GEMM.  A row-major [M, N] output is the
// head-major case with one batch entry (S = M), one head (H = 1, D = N) and
// N <= K, so that every column belongs to the q block.
cudaError_t launch_proj(la_dtype dt, int block_n, const CUtensorMap& tx, const CUtensorMap& tw, const ProjArgs& a,
                        cudaStream_t st);

}  // namespace la
