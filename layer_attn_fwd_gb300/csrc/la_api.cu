// la_api.cu -- the C ABI of liblayerattn.so (declared in include/layerattn.h).
//
// Host side only: argument validation (before anything touches a device),
// TMA tensor-map encoding, the split-KV plan, workspace carving and the
// launches.  The library allocates no device memory.  The one piece of device
// state is the error word below, which kernels latch when a bounded wait runs
// out.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "la_device.cuh"
#include "la_internal.h"

__device__ uint32_t la_device_error_word;

// Scratch of la_attn_fwd_noalloc(): split-KV partials (and, for fp32, V
// transposed) for callers that cannot supply a workspace.  Every GPU that
// loads the library holds it until the process exits.
static constexpr size_t kNoAllocScratchBytes = 16u << 20;
static __device__ __align__(256) uint8_t la_noalloc_scratch[kNoAllocScratchBytes];

namespace la {
namespace {

// ---------------------------------------------------------------------------
// small utilities
// ---------------------------------------------------------------------------
int elem_bytes(la_dtype dt) { return dt == LA_F32 ? 4 : 2; }
bool dtype_ok(int dt) { return dt == LA_F32 || dt == LA_BF16 || dt == LA_F16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

la_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;

// One-shot request from la_debug_inject_timeout().
std::atomic<int> g_skip_loads_once{0};
// One-shot request from la_debug_shrink_output_extent().
std::atomic<int> g_shrink_once{0};
// Raw device error word seen by the latest la_get_last_error().
std::atomic<uint32_t> g_last_word{0};

uint32_t* error_word() {
  static std::mutex mu;
  static uint32_t* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, la_device_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  return addr[dev];
}

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

// fp32 operands feed TF32 products: the TFLOAT32 map type has the copy round
// them to TF32 (measured: half the error of letting the tensor core drop the
// low mantissa bits).
CUtensorMapDataType tma_type(la_dtype dt) {
  return dt == LA_F32 ? CU_TENSOR_MAP_DATA_TYPE_TFLOAT32
                      : (dt == LA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

// 4-D tiled map, 128-byte swizzle: extents d0 (innermost, contiguous) .. d3,
// strides s1..s3 in elements, box box0 x box1 x 1 x 1.
la_status map_4d(CUtensorMap* m, const void* base, la_dtype dt, long long d0, long long d1, long long d2,
                 long long d3, long long s1, long long s2, long long s3, int box0, int box1) {
  auto fn = encode_fn();
  if (fn == nullptr) return LA_ERR_CUDA;
  const long long e = elem_bytes(dt);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d0 > 0 ? d0 : 1), static_cast<cuuint64_t>(d1 > 0 ? d1 : 1),
                        static_cast<cuuint64_t>(d2), static_cast<cuuint64_t>(d3)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s1 * e), static_cast<cuuint64_t>(s2 * e),
                           static_cast<cuuint64_t>(s3 * e)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, tma_type(dt), 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LA_OK : LA_ERR_CUDA;
}

// [B, H, rows, D] view with the given element strides.
la_status map_bhsd(CUtensorMap* m, const void* base, la_dtype dt, int B, int H, long long rows, int D,
                   long long s_row, long long s_head, long long s_batch, int box_rows, int box_cols) {
  return map_4d(m, base, dt, D, rows, H, B, s_row, s_head, s_batch, box_cols, box_rows);
}

// 2-D map over a row-major [rows, cols] matrix.
la_status map_2d(CUtensorMap* m, const void* base, la_dtype dt, long long rows, long long cols, int box_rows,
                 int box_cols, bool raw = false) {
  auto fn = encode_fn();
  if (fn == nullptr) return LA_ERR_CUDA;
  const long long e = elem_bytes(dt);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * e)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, raw && dt == LA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tma_type(dt), 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LA_OK : LA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// split-KV plan
// ---------------------------------------------------------------------------
struct Plan {
  int num_qblk = 0;
  int n_tiles = 0;  // key tiles of the longest query tile
  int splits = 1;
  int tiles_per_split = 1;
  size_t ws_bytes = 0;  // partials the plan needs
};

// Bytes of keys and values the concurrently running causal items share
// (a quarter of the 126 MB of L2, which the two dies split between them).
constexpr long long kGroupBytes = 32LL << 20;

// The persistent attention's ticket word and done word (two 64-bit words,
// padded so that what follows stays 256-byte aligned).
constexpr size_t kSchedBytes = 256;

// Tag of the next persistent launch (never 0, the value of a word at rest).
unsigned next_sched_tag() {
  static std::atomic<unsigned> tag{0};
  unsigned t = tag.fetch_add(1u) + 1u;
  while (t == 0u) t = tag.fetch_add(1u) + 1u;
  return t;
}

size_t split_bytes(int splits, int B, int H, int S_q, int D) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(splits) * B * H * S_q;
  return round_up(rows * D * sizeof(float), 256) + round_up(rows * sizeof(float), 256);
}

// fp32 only: V^T [B, H, D, S_pad] for the TF32 PV product (K-major operands).
long long vt_pad(long long S_kv) { return (S_kv + 3) / 4 * 4; }
size_t vt_bytes(la_dtype dt, int B, int H, long long S_kv, int D) {
  if (dt != LA_F32) return 0;
  return round_up(static_cast<size_t>(B) * H * D * vt_pad(S_kv) * 4, 256);
}
// fp32 only: Wqkv^T [3d, d] for the TF32 projection.
size_t wt_bytes(la_dtype dt, int d_model) {
  if (dt != LA_F32) return 0;
  return round_up(static_cast<size_t>(3) * d_model * d_model * 4, 256);
}
// fp32 only: Wo^T [d, d] for the TF32 output projection.
size_t wot_bytes(la_dtype dt, int d_model) {
  if (dt != LA_F32) return 0;
  return round_up(static_cast<size_t>(d_model) * d_model * 4, 256);
}

// Split the key range only when the unsplit grid leaves the GPU short of
// full waves; estimate makespan as waves x tiles per CTA (+2 tiles of fixed
// cost per CTA) and take the smallest, within what the workspace holds.
Plan make_plan(la_dtype dt, int B, int H, int S_q, int S_kv, int D, size_t ws_avail, int sms) {
  Plan p;
  AttnShape sh;
  attn_shape(dt, D, &sh);
  p.num_qblk = (S_q + sh.rows_per_cta - 1) / sh.rows_per_cta;
  p.n_tiles = (S_kv + sh.block_n - 1) / sh.block_n;
  if (p.n_tiles < 1) p.n_tiles = 1;
  p.tiles_per_split = p.n_tiles;
  const long long ctas = static_cast<long long>(p.num_qblk) * B * H;
  double best = 0.0;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && p.n_tiles / s < 4) break;
    if (static_cast<long long>(s) * B * H > 65535LL * 65535LL) break;
    const size_t need = split_bytes(s, B, H, S_q, D);
    if (need > ws_avail) break;
    const int per = (p.n_tiles + s - 1) / s;
    const long long waves = (ctas * s + sms - 1) / sms;
    const double cost = static_cast<double>(waves) * (per + 2) + (s > 1 ? 1.0 : 0.0);
    if (s == 1 || cost < best * 0.95) {
      best = cost;
      p.splits = s;
      p.tiles_per_split = per;
      p.ws_bytes = need;
    }
  }
  return p;
}

// ---------------------------------------------------------------------------
// validation shared by the attention entry points
// ---------------------------------------------------------------------------
la_status check_attn_args(int B, int H, int S_q, int S_kv, int D, float scale, int dt) {
  if (B < 1 || H < 1 || S_q < 0 || S_kv < 0) return LA_ERR_INVALID;
  if (!dtype_ok(dt)) return LA_ERR_INVALID;
  if (!(scale > 0.f) || !isfinite(scale)) return LA_ERR_INVALID;
  if (D != 64 && D != 128) return LA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return LA_ERR_UNSUPPORTED;  // grid.y
  return LA_OK;
}

// Key/value operands of one attention call: rows [0, S_kv) of k/v buffers
// [B, H, rows_alloc, D]; for fp32 V may instead be given already transposed
// as V^T [B, H, D, vt_ld] (vt != nullptr).
struct KVView {
  const void* k;
  const void* v;
  long long rows_alloc;
  const void* vt;
  long long vt_ld;
};

// Attention: q [B,H,S_q,D] contiguous; o with the given element strides.
// Scratch from ws, in this order: the fp32 V^T (unless given; required),
// the ticket words of the persistent form (without room for them every item
// gets a CTA of its own), then the split partials (the plan splits only as
// far as what is left allows).
la_status run_attention(const void* q, const KVView& kv, void* o, long long o_sb, long long o_sh, long long o_ss,
                        int B, int H, int S_q, int S_kv, int D, int causal, float scale, const int32_t* kv_len,
                        la_dtype dt, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (S_q == 0) return LA_OK;
  AttnShape sh;
  if (!attn_shape(dt, D, &sh)) return LA_ERR_UNSUPPORTED;
  // No key at all: every row is a zero row.  Both output layouts used here
  // (head-major, and heads merged) cover exactly B*H*S_q*D contiguous
  // elements; no tensor map is built (a V^T map over zero keys has no valid
  // stride).
  if (S_kv == 0)
    return cuda_status(cudaMemsetAsync(o, 0, static_cast<size_t>(B) * H * S_q * D * elem_bytes(dt), st));
  uint8_t* w = static_cast<uint8_t*>(ws);
  size_t w_left = ws == nullptr ? 0 : ws_bytes;
  const void* vt = kv.vt;
  long long vt_ld = kv.vt_ld;
  // fp32 with a single key tile and one CTA per item (the small shapes): the
  // attention kernel transposes its one V tile in shared memory itself, so
  // there is no V^T pre-pass launch and no V^T workspace
  const long long items1 = static_cast<long long>((S_q + sh.rows_per_cta - 1) / sh.rows_per_cta) * B * H;
  const bool v_raw = dt == LA_F32 && vt == nullptr && S_kv <= sh.block_n && items1 <= device_sms();
  if (dt == LA_F32 && vt == nullptr && !v_raw) {
    const size_t need = vt_bytes(dt, B, H, S_kv, D);
    if (w_left < need) return LA_ERR_WORKSPACE;
    vt_ld = vt_pad(S_kv);
    if (S_kv > 0 && launch_transpose32(kv.v, kv.rows_alloc * D, w, vt_ld, static_cast<long long>(B) * H, S_kv, D,
                                       st) != cudaSuccess)
      return LA_ERR_CUDA;
    vt = w;
    w += need;
    w_left -= need;
  }
  unsigned long long* sched = nullptr;
  if (w_left >= kSchedBytes) {
    sched = reinterpret_cast<unsigned long long*>(w);
    w += kSchedBytes;
    w_left -= kSchedBytes;
  }
  const Plan p = make_plan(dt, B, H, S_q, S_kv, D, w_left, device_sms());
  uint32_t* err = error_word();
  if (err == nullptr) return LA_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  la_status s;
  s = map_bhsd(&tq, q, dt, B, H, S_q, D, D, static_cast<long long>(S_q) * D, static_cast<long long>(H) * S_q * D,
               sh.box_q_rows, sh.box_cols);
  if (s != LA_OK) return s;
  s = map_bhsd(&tk, kv.k, dt, B, H, S_kv, D, D, kv.rows_alloc * D, static_cast<long long>(H) * kv.rows_alloc * D,
               sh.box_kv_rows, sh.box_cols);
  if (s != LA_OK) return s;
  if (dt == LA_F32 && !v_raw) {
    // V^T: keys innermost (the K dimension of the PV product), head dims as rows
    s = map_4d(&tv, vt, dt, S_kv, D, H, B, vt_ld, static_cast<long long>(D) * vt_ld,
               static_cast<long long>(H) * D * vt_ld, sh.box_cols, D);
  } else {
    s = map_bhsd(&tv, kv.v, dt, B, H, S_kv, D, D, kv.rows_alloc * D, static_cast<long long>(H) * kv.rows_alloc * D,
                 sh.box_kv_rows, sh.box_cols);
  }
  if (s != LA_OK) return s;

  AttnArgs a;
  memset(&a, 0, sizeof a);
  a.o = o;
  a.o_sb = o_sb;
  a.o_sh = o_sh;
  a.o_ss = o_ss;
  a.kv_len = kv_len;
  a.B = B;
  a.H = H;
  a.S_q = S_q;
  a.S_kv = S_kv;
  a.causal = causal ? 1 : 0;
  a.sl2 = scale * 1.4426950408889634f;
  a.num_qblk = p.num_qblk;
  a.tiles_per_split = p.tiles_per_split;
  {
    // Causal items go out heaviest first within groups of (b, h) pairs whose
    // keys and values together fill about a quarter of L2, so that the items
    // that read the same keys run at about the same time and find them there.
    const long long pair_bytes =
        std::max(1LL, static_cast<long long>(S_kv) * D * static_cast<long long>(elem_bytes(dt)) * 2);
    const long long g = std::min(static_cast<long long>(B) * H, kGroupBytes / pair_bytes);
    a.head_group = static_cast<int>(std::max(1LL, g));
  }
  a.err = err;
  a.sched = sched;
  a.sched_gen = next_sched_tag();
  a.skip_loads = g_skip_loads_once.exchange(0);
  a.v_raw = v_raw ? 1 : 0;
#if LA_CHECKED
  // extents for the bounds checks: [B, H, S_q, D] elements either layout
  a.o_elems = static_cast<long long>(B) * H * S_q * D;
  if (g_shrink_once.exchange(0)) a.o_elems -= D;  // test hook: declare the last row outside
#else
  g_shrink_once.store(0);  // nothing is checked here: the hook has no effect
#endif
  if (p.splits > 1) {
    const size_t rows = static_cast<size_t>(p.splits) * B * H * S_q;
    a.part_o = reinterpret_cast<float*>(w);
    a.part_lse = reinterpret_cast<float*>(w + round_up(rows * D * sizeof(float), 256));
#if LA_CHECKED
    a.part_elems = static_cast<long long>(rows) * D;
#endif
  }
  cudaError_t e = launch_attn(dt, D, tq, tk, tv, a, p.splits, st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  if (p.splits > 1) {
    CombineArgs c;
    c.part_o = a.part_o;
    c.part_lse = a.part_lse;
    c.o = o;
    c.o_sb = o_sb;
    c.o_sh = o_sh;
    c.o_ss = o_ss;
    c.B = B;
    c.H = H;
    c.S_q = S_q;
    c.D = D;
    c.splits = p.splits;
#if LA_CHECKED
    c.o_elems = a.o_elems;
    c.err = err;
#endif
    e = launch_combine(dt, c, st);
    if (e != cudaSuccess) return LA_ERR_CUDA;
  }
  return LA_OK;
}

size_t attn_ws_bytes(la_dtype dt, int B, int H, int S_q, int S_kv, int D, bool need_vt) {
  if (S_q == 0) return 0;
  const size_t vt = need_vt ? vt_bytes(dt, B, H, S_kv, D) : 0;
  return vt + kSchedBytes + make_plan(dt, B, H, S_q, S_kv, D, static_cast<size_t>(-1), device_sms()).ws_bytes;
}

la_status check_proj_args(const void* x, const void* W, const void* bias, const void* q, const void* k,
                          const void* v, int B, int S, int d_model, int H, float q_scale, int dt) {
  if (!x || !W || !q || !k || !v) return LA_ERR_INVALID;
  if (B < 1 || S < 0 || d_model < 1 || H < 1) return LA_ERR_INVALID;
  if (!dtype_ok(dt) || !isfinite(q_scale)) return LA_ERR_INVALID;
  if (d_model % H != 0) return LA_ERR_INVALID;
  const int D = d_model / H;
  if (D != 64 && D != 128) return LA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(W) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return LA_ERR_INVALID;
  if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 3u)) return LA_ERR_INVALID;
  if (static_cast<long long>(B) * S > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
  return LA_OK;
}

// LayerNorm in front of the projection: per-row statistics (from the stats
// pre-pass) and gamma, beta; the projection normalises x as it loads it.
struct LnIn {
  const float2* stats = nullptr;
  const void* gamma = nullptr;
  const void* beta = nullptr;
};

// Projection.  w_kernel: the weight already in the layout the kernel reads
// (fp32: Wqkv^T [3d, d]; half precision: Wqkv itself), or null: then fp32
// transposes W into ws first.  With vt != nullptr (fp32 sublayer) V is
// written as V^T [B, H, D, vt_ld] there instead of into v.
la_status run_proj(const void* x, const void* W, const void* bias, void* q, void* k, void* v, int B, int S,
                   int d_model, int H, float q_scale, la_dtype dt, void* ws, size_t ws_bytes, const void* w_kernel,
                   void* vt, long long vt_ld, cudaStream_t st, const LnIn& ln = LnIn()) {
  const long long M = static_cast<long long>(B) * S;
  if (M == 0) return LA_OK;
  ProjShape ps;
  if (!proj_shape(dt, M, 3LL * d_model, device_sms(), &ps)) return LA_ERR_UNSUPPORTED;
  uint32_t* err = error_word();
  if (err == nullptr) return LA_ERR_CUDA;
  CUtensorMap tx, tw;
  // with LayerNorm in front, fp32 x is copied unrounded (it is normalised,
  // then rounded to TF32, in shared memory)
  la_status s = map_2d(&tx, x, dt, M, d_model, kTileM, ps.box_cols, ln.stats != nullptr);
  if (s != LA_OK) return s;
  if (ps.w_transposed) {
    if (w_kernel == nullptr) {
      const size_t need = wt_bytes(dt, d_model);
      if (ws == nullptr || ws_bytes < need) return LA_ERR_WORKSPACE;
      if (launch_transpose32(W, 0, ws, d_model, 1, d_model, 3 * d_model, st) != cudaSuccess) return LA_ERR_CUDA;
      w_kernel = ws;
    }
    s = map_2d(&tw, w_kernel, dt, 3LL * d_model, d_model, ps.block_n, ps.box_cols);
  } else {
    s = map_2d(&tw, w_kernel != nullptr ? w_kernel : W, dt, d_model, 3LL * d_model, ps.box_k_rows, ps.box_cols);
  }
  if (s != LA_OK) return s;
  ProjArgs a;
  memset(&a, 0, sizeof a);
  a.bias = bias;
  a.q = q;
  a.k = k;
  a.v = vt != nullptr ? vt : v;
  a.M = static_cast<int>(M);
  a.N = 3 * d_model;
  a.K = d_model;
  a.S = S;
  a.H = H;
  a.D = d_model / H;
  a.q_scale = q_scale;
  a.err = err;
  a.v_transposed = vt != nullptr;
  a.S_pad = vt_ld;
  a.ln_stats = ln.stats;
  a.ln_gamma = ln.gamma;
  a.ln_beta = ln.beta;
#if LA_CHECKED
  a.qk_elems = M * d_model;
  a.v_elems = vt != nullptr ? static_cast<long long>(B) * d_model * vt_ld : M * d_model;
#endif
  return cuda_status(launch_proj(dt, ps.block_n, tx, tw, a, st));
}

// Output projection y [M, d] = a [M, d] . Wo [d, d] + bo on the projection
// GEMM: a row-major output is its head-major case with one batch entry and
// one head as wide as the row.  fp32 reads Wo^T [d, d] from wot, transposed
// there beforehand (TF32 products take K-major operands only).
la_status run_out_proj(const void* a_in, const void* Wo, const void* wot, const void* bo, void* y, long long M,
                       int d, la_dtype dt, cudaStream_t st) {
  if (M == 0) return LA_OK;
  ProjShape ps;
  if (!proj_shape(dt, M, d, device_sms(), &ps)) return LA_ERR_UNSUPPORTED;
  uint32_t* err = error_word();
  if (err == nullptr) return LA_ERR_CUDA;
  CUtensorMap tx, tw;
  la_status s = map_2d(&tx, a_in, dt, M, d, kTileM, ps.box_cols);
  if (s != LA_OK) return s;
  if (ps.w_transposed)
    s = map_2d(&tw, wot, dt, d, d, ps.block_n, ps.box_cols);
  else
    s = map_2d(&tw, Wo, dt, d, d, ps.box_k_rows, ps.box_cols);
  if (s != LA_OK) return s;
  ProjArgs a;
  memset(&a, 0, sizeof a);
  a.bias = bo;
  a.q = a.k = a.v = y;  // N == K: every column is in the first block
  a.M = static_cast<int>(M);
  a.N = d;
  a.K = d;
  a.S = static_cast<int>(M);
  a.H = 1;
  a.D = d;
  a.q_scale = 1.f;
  a.err = err;
#if LA_CHECKED
  a.qk_elems = a.v_elems = M * d;
#endif
  return cuda_status(launch_proj(dt, ps.block_n, tx, tw, a, st));
}

la_status check_out_proj_args(const void* a_in, const void* Wo, const void* bo, const void* y, long long M,
                              int d_model, int dt) {
  if (!a_in || !Wo || !y) return LA_ERR_INVALID;
  if (M < 0 || d_model < 1 || !dtype_ok(dt)) return LA_ERR_INVALID;
  if (d_model % 64 != 0) return LA_ERR_UNSUPPORTED;
  if (M > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
  if (!aligned16(a_in) || !aligned16(Wo) || !aligned16(y)) return LA_ERR_INVALID;
  if (bo != nullptr && (reinterpret_cast<uintptr_t>(bo) & 3u)) return LA_ERR_INVALID;
  return LA_OK;
}

size_t layer_qkv_bytes(int B, int S, int d_model, la_dtype dt) {
  return round_up(static_cast<size_t>(B) * S * d_model * elem_bytes(dt), 256);
}

size_t layer_fixed_bytes(int B, int S, int d_model, int H, la_dtype dt) {
  const size_t one = layer_qkv_bytes(B, S, d_model, dt);
  const size_t vbytes = dt == LA_F32 ? vt_bytes(dt, B, H, S, d_model / H) : one;
  return 2 * one + vbytes + wt_bytes(dt, d_model);
}

// The sublayer without its output projection: ws holds q | k | v (fp32: V^T
// [B,H,D,S_pad]) | fp32 Wqkv^T | split partials.  w_kernel: the weight in
// the projection kernel's layout (see run_proj), or null.
la_status run_layer(const void* x, const void* Wqkv, const void* bqkv, void* o, int B, int S, int d_model, int H,
                    int causal, const int32_t* kv_len, la_dtype dt, void* ws, size_t ws_bytes, const void* w_kernel,
                    cudaStream_t cs, const LnIn& ln = LnIn()) {
  const int D = d_model / H;
  const size_t one = layer_qkv_bytes(B, S, d_model, dt);
  const size_t vbytes = dt == LA_F32 ? vt_bytes(dt, B, H, S, D) : one;
  const size_t fixed = layer_fixed_bytes(B, S, d_model, H, dt);
  if (ws_bytes < fixed) return LA_ERR_WORKSPACE;
  if (S == 0) return LA_OK;
  uint8_t* w = static_cast<uint8_t*>(ws);
  void *q = w, *k = w + one, *v = w + 2 * one;
  uint8_t* wt = w + 2 * one + vbytes;
  const bool vt = dt == LA_F32;
  la_status s = run_proj(x, Wqkv, bqkv, q, k, v, B, S, d_model, H, 1.f, dt, wt, wt_bytes(dt, d_model), w_kernel,
                         vt ? v : nullptr, vt_pad(S), cs, ln);
  if (s != LA_OK) return s;
  const float scale = 1.0f / sqrtf(static_cast<float>(D));
  const KVView kv{k, v, S, vt ? v : nullptr, vt_pad(S)};
  return run_attention(q, kv, o, static_cast<long long>(S) * d_model, D, d_model, B, H, S, S, D, causal, scale,
                       kv_len, dt, w + fixed, ws_bytes - fixed, cs);
}

la_status check_layer_args(const void* x, const void* Wqkv, const void* bqkv, const void* o, const void* ws, int B,
                           int S, int d_model, int H, const int32_t* kv_len, int dt) {
  if (!o || !ws) return LA_ERR_INVALID;
  if (!aligned16(o) || !aligned16(ws)) return LA_ERR_INVALID;
  // validate with placeholders for the q/k/v pointers, which live in ws
  la_status s = check_proj_args(x, Wqkv, bqkv, ws, ws, ws, B, S, d_model, H, 1.f, dt);
  if (s != LA_OK) return s;
  s = check_attn_args(B, H, S, S, d_model / H, 1.f, dt);
  if (s != LA_OK) return s;
  if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return LA_ERR_INVALID;
  return LA_OK;
}

la_status check_ln_args(const void* gamma, const void* beta, float eps) {
  if (!gamma || !beta) return LA_ERR_INVALID;
  if (!aligned16(gamma) || !aligned16(beta)) return LA_ERR_INVALID;
  if (!(eps >= 0.f) || !isfinite(eps)) return LA_ERR_INVALID;
  return LA_OK;
}

// Row statistics of the LayerNorm in front: (mean, 1 / sqrt(var + eps)) per row.
size_t ln_stats_bytes(int B, int S) { return round_up(static_cast<size_t>(B) * S * sizeof(float2), 256); }

// Workspace of the block: the row statistics (with LayerNorm) | the merged
// attention output and the fp32 Wo^T (with the output projection) | the
// sublayer's own workspace.
size_t block_fixed_bytes(int B, int S, int d_model, int H, la_dtype dt, bool ln, bool out) {
  const size_t act = layer_qkv_bytes(B, S, d_model, dt);
  return (ln ? ln_stats_bytes(B, S) : 0) + (out ? act + wot_bytes(dt, d_model) : 0) +
         layer_fixed_bytes(B, S, d_model, H, dt);
}

// The attention block: [LayerNorm] -> projection -> attention (heads merged)
// -> [output projection].  Arguments already validated.  For fp32 the
// weight transposes come first: Wqkv^T as an ordinary launch (everything
// before this call has finished), then Wo^T and the LayerNorm statistics,
// which may overlap it (each waits for the grid before it before exiting).
// prepared: Wqkv and Wo are already in the kernels' layout
// (la_prepare_weight), so nothing is transposed.
la_status run_block(const void* x, const void* gamma, const void* beta, float eps, const void* Wqkv,
                    const void* bqkv, const void* Wo, const void* bo, void* y, int B, int S, int d_model, int H,
                    int causal, const int32_t* kv_len, la_dtype dt, void* ws, size_t ws_bytes, cudaStream_t cs,
                    bool prepared = false) {
  const bool ln = gamma != nullptr, out = Wo != nullptr;
  if (ws_bytes < block_fixed_bytes(B, S, d_model, H, dt, ln, out)) return LA_ERR_WORKSPACE;
  if (S == 0) return LA_OK;
  const size_t act = layer_qkv_bytes(B, S, d_model, dt);
  const long long M = static_cast<long long>(B) * S;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float2* stats = ln ? reinterpret_cast<float2*>(w) : nullptr;
  w += ln ? ln_stats_bytes(B, S) : 0;
  void* o = out ? w : y;
  void* wot = out ? w + act : nullptr;
  w += out ? act + wot_bytes(dt, d_model) : 0;
  const size_t lw_bytes = ws_bytes - static_cast<size_t>(w - static_cast<uint8_t*>(ws));
  bool first = true;  // the first launch of the call is an ordinary one
  const void* w_kernel = prepared ? Wqkv : nullptr;
  if (prepared) {
    wot = const_cast<void*>(Wo);
  } else if (dt == LA_F32) {
    uint8_t* wt = w + 2 * act + vt_bytes(dt, B, H, S, d_model / H);  // where run_layer keeps Wqkv^T
    if (launch_transpose32(Wqkv, 0, wt, d_model, 1, d_model, 3 * d_model, cs) != cudaSuccess) return LA_ERR_CUDA;
    first = false;
    w_kernel = wt;
    if (out && launch_transpose32(Wo, 0, wot, d_model, 1, d_model, d_model, cs, true) != cudaSuccess)
      return LA_ERR_CUDA;
  }
  LnIn lni;
  if (ln) {  // the statistics only; the projection normalises x as it loads it
    if (launch_layernorm(dt, x, gamma, beta, nullptr, M, d_model, eps, cs, !first, stats) != cudaSuccess)
      return LA_ERR_CUDA;
    first = false;
    lni.stats = stats;
    lni.gamma = gamma;
    lni.beta = beta;
  }
  la_status s = run_layer(x, Wqkv, bqkv, o, B, S, d_model, H, causal, kv_len, dt, w, lw_bytes, w_kernel, cs, lni);
  if (s != LA_OK || !out) return s;
  return run_out_proj(o, Wo, wot, bo, y, M, d_model, dt, cs);
}

}  // namespace

// ---------------------------------------------------------------------------
// per-launch timing (la_profile_start / la_profile_stop)
// ---------------------------------------------------------------------------
namespace {
struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::vector<ProfRecord> g_prof;
size_t g_prof_max = 0;
std::atomic<bool> g_prof_on{false};
// index of the record the launch being made on this thread opened, or -1
// (past the record limit, nothing is recorded for it)
thread_local long t_prof_open = -1;
}  // namespace

bool prof_on() { return g_prof_on.load(std::memory_order_relaxed); }

void prof_before(cudaStream_t st, const char* name) {
  t_prof_open = -1;
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof.size() >= g_prof_max) return;
  ProfRecord r{name, nullptr, nullptr};
  if (cudaEventCreate(&r.start) != cudaSuccess) return;
  if (cudaEventCreate(&r.stop) != cudaSuccess) {
    cudaEventDestroy(r.start);
    return;
  }
  cudaEventRecord(r.start, st);
  t_prof_open = static_cast<long>(g_prof.size());
  g_prof.push_back(r);
}

void prof_after(cudaStream_t st) {
  if (t_prof_open < 0) return;  // this launch was not recorded
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (static_cast<size_t>(t_prof_open) < g_prof.size()) cudaEventRecord(g_prof[t_prof_open].stop, st);
  t_prof_open = -1;
}

}  // namespace la

using namespace la;

extern "C" {

la_status la_qkv_proj(const void* x, const void* Wqkv, const void* bqkv, void* q, void* k, void* v, int B, int S,
                      int d_model, int H, float q_scale, la_dtype dt, void* ws, size_t ws_bytes, la_stream_t st) {
  la_status s = check_proj_args(x, Wqkv, bqkv, q, k, v, B, S, d_model, H, q_scale, dt);
  if (s != LA_OK) return s;
  if (ws != nullptr && !aligned16(ws)) return LA_ERR_INVALID;
  if (S > 0 && (ws == nullptr ? 0 : ws_bytes) < wt_bytes(dt, d_model)) return LA_ERR_WORKSPACE;
  return run_proj(x, Wqkv, bqkv, q, k, v, B, S, d_model, H, q_scale, dt, ws, ws_bytes, nullptr, nullptr, 0,
                  reinterpret_cast<cudaStream_t>(st));
}

la_status la_attn_fwd(const void* q, const void* k, const void* v, void* o, int B, int H, int S_q, int S_kv,
                      int D, int causal, float scale, const int32_t* kv_len, la_dtype dt, void* ws,
                      size_t ws_bytes, la_stream_t st) {
  // a pointer may be NULL only when its tensor is empty
  if ((!q || !o) && S_q != 0) return LA_ERR_INVALID;
  if ((!k || !v) && S_kv != 0) return LA_ERR_INVALID;
  la_status s = check_attn_args(B, H, S_q, S_kv, D, scale, dt);
  if (s != LA_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LA_ERR_INVALID;
  if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return LA_ERR_INVALID;
  if (ws != nullptr && !aligned16(ws)) return LA_ERR_INVALID;
  if (S_q == 0) return LA_OK;
  if (S_kv == 0) k = v = q;  // no key is ever loaded; the maps only need a valid base
  if ((ws == nullptr ? 0 : ws_bytes) < vt_bytes(dt, B, H, S_kv, D)) return LA_ERR_WORKSPACE;
  const KVView kv{k, v, S_kv, nullptr, 0};
  return run_attention(q, kv, o, static_cast<long long>(H) * S_q * D, static_cast<long long>(S_q) * D, D, B, H,
                       S_q, S_kv, D, causal, scale, kv_len, dt, ws, ws_bytes, reinterpret_cast<cudaStream_t>(st));
}

la_status la_attn_chunked(const void* q_chunk, const void* k_chunk, const void* v_chunk, la_kv_cache* cache,
                          void* o_chunk, int chunk, int causal, float scale, void* ws, size_t ws_bytes,
                          la_stream_t st) {
  if (!cache || !q_chunk || !k_chunk || !v_chunk || !o_chunk || !cache->k || !cache->v) return LA_ERR_INVALID;
  const int B = cache->B, H = cache->H, D = cache->D;
  if (chunk < 0 || cache->len < 0 || cache->S_max < 1) return LA_ERR_INVALID;
  if (static_cast<long long>(cache->len) + chunk > cache->S_max) return LA_ERR_INVALID;
  la_status s = check_attn_args(B, H, chunk, cache->len + chunk, D, scale, cache->dtype);
  if (s != LA_OK) return s;
  if (!aligned16(q_chunk) || !aligned16(k_chunk) || !aligned16(v_chunk) || !aligned16(o_chunk) ||
      !aligned16(cache->k) || !aligned16(cache->v))
    return LA_ERR_INVALID;
  if (ws != nullptr && !aligned16(ws)) return LA_ERR_INVALID;
  const la_dtype dt = cache->dtype;
  // fp32: the cache holds V^T [B, H, D, S_max]; its rows must start 16-byte
  // aligned for the tensor map
  if (dt == LA_F32 && cache->S_max % 4 != 0) return LA_ERR_INVALID;
  if (chunk == 0) return LA_OK;
  const int S_kv = cache->len + chunk;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(st);
  if (dt == LA_F32) {
    // keys appended as rows; values appended transposed, at columns
    // [len, len + chunk) of every (b, h) block of V^T
    if (launch_kv_append(k_chunk, nullptr, cache->k, nullptr, B, H, chunk, D, cache->S_max, cache->len,
                         elem_bytes(dt), cs) != cudaSuccess ||
        launch_transpose32(v_chunk, static_cast<long long>(chunk) * D,
                           static_cast<float*>(cache->v) + cache->len, cache->S_max,
                           static_cast<long long>(B) * H, chunk, D, cs) != cudaSuccess)
      return LA_ERR_CUDA;
  } else if (launch_kv_append(k_chunk, v_chunk, cache->k, cache->v, B, H, chunk, D, cache->S_max, cache->len,
                              elem_bytes(dt), cs) != cudaSuccess) {
    return LA_ERR_CUDA;
  }
  const KVView kv{cache->k, cache->v, cache->S_max, dt == LA_F32 ? cache->v : nullptr, cache->S_max};
  s = run_attention(q_chunk, kv, o_chunk, static_cast<long long>(H) * chunk * D, static_cast<long long>(chunk) * D,
                    D, B, H, chunk, S_kv, D, causal, scale, nullptr, dt, ws, ws_bytes, cs);
  if (s == LA_OK) cache->len = S_kv;
  return s;
}

la_status la_layer_attn(const void* x, const void* Wqkv, const void* bqkv, void* o, int B, int S, int d_model,
                        int H, int causal, const int32_t* kv_len, la_dtype dt, void* ws, size_t ws_bytes,
                        la_stream_t st) {
  la_status s = check_layer_args(x, Wqkv, bqkv, o, ws, B, S, d_model, H, kv_len, dt);
  if (s != LA_OK) return s;
  return run_layer(x, Wqkv, bqkv, o, B, S, d_model, H, causal, kv_len, dt, ws, ws_bytes, nullptr,
                   reinterpret_cast<cudaStream_t>(st));
}

la_status la_out_proj(const void* a, const void* Wo, const void* bo, void* y, int M, int d_model, la_dtype dt,
                      void* ws, size_t ws_bytes, la_stream_t st) {
  la_status s = check_out_proj_args(a, Wo, bo, y, M, d_model, dt);
  if (s != LA_OK) return s;
  if (ws != nullptr && !aligned16(ws)) return LA_ERR_INVALID;
  if (M == 0) return LA_OK;
  if ((ws == nullptr ? 0 : ws_bytes) < wot_bytes(dt, d_model)) return LA_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(st);
  if (dt == LA_F32 && launch_transpose32(Wo, 0, ws, d_model, 1, d_model, d_model, cs) != cudaSuccess)
    return LA_ERR_CUDA;
  return run_out_proj(a, Wo, ws, bo, y, M, d_model, dt, cs);
}

la_status la_layer_attn_out(const void* x, const void* Wqkv, const void* bqkv, const void* Wo, const void* bo,
                            void* y, int B, int S, int d_model, int H, int causal, const int32_t* kv_len,
                            la_dtype dt, void* ws, size_t ws_bytes, la_stream_t st) {
  la_status s = check_layer_args(x, Wqkv, bqkv, y, ws, B, S, d_model, H, kv_len, dt);
  if (s != LA_OK) return s;
  s = check_out_proj_args(ws, Wo, bo, y, static_cast<long long>(B) * S, d_model, dt);
  if (s != LA_OK) return s;
  return run_block(x, nullptr, nullptr, 0.f, Wqkv, bqkv, Wo, bo, y, B, S, d_model, H, causal, kv_len, dt, ws,
                   ws_bytes, reinterpret_cast<cudaStream_t>(st));
}

la_status la_layernorm(const void* x, const void* gamma, const void* beta, void* y, int M, int d, float eps,
                       la_dtype dt, la_stream_t st) {
  if (!x || !y) return LA_ERR_INVALID;
  if (M < 0 || d < 1 || !dtype_ok(dt)) return LA_ERR_INVALID;
  la_status s = check_ln_args(gamma, beta, eps);
  if (s != LA_OK) return s;
  if (d % 64 != 0) return LA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y)) return LA_ERR_INVALID;
  if (M == 0) return LA_OK;
  return cuda_status(launch_layernorm(dt, x, gamma, beta, y, M, d, eps, reinterpret_cast<cudaStream_t>(st)));
}

la_status la_layer_attn_ln(const void* x, const void* gamma, const void* beta, float eps, const void* Wqkv,
                           const void* bqkv, const void* Wo, const void* bo, void* y, int B, int S, int d_model,
                           int H, int causal, const int32_t* kv_len, la_dtype dt, void* ws, size_t ws_bytes,
                           la_stream_t st) {
  la_status s = check_layer_args(x, Wqkv, bqkv, y, ws, B, S, d_model, H, kv_len, dt);
  if (s != LA_OK) return s;
  s = check_ln_args(gamma, beta, eps);
  if (s != LA_OK) return s;
  if (Wo != nullptr) {
    s = check_out_proj_args(ws, Wo, bo, y, static_cast<long long>(B) * S, d_model, dt);
    if (s != LA_OK) return s;
  } else if (bo != nullptr) {
    return LA_ERR_INVALID;
  }
  return run_block(x, gamma, beta, eps, Wqkv, bqkv, Wo, bo, y, B, S, d_model, H, causal, kv_len, dt, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(st));
}

la_status la_prepare_weight(const void* W, void* Wp, int rows, int cols, la_dtype dt, la_stream_t st) {
  if (!W || !Wp || rows < 1 || cols < 1 || !dtype_ok(dt)) return LA_ERR_INVALID;
  if (!aligned16(W) || !aligned16(Wp)) return LA_ERR_INVALID;
  if (rows % 64 != 0 || cols % 64 != 0) return LA_ERR_UNSUPPORTED;
  const size_t bytes = static_cast<size_t>(rows) * cols * elem_bytes(dt);
  const char* a = static_cast<const char*>(W);
  const char* b = static_cast<const char*>(Wp);
  if (a < b + bytes && b < a + bytes) return LA_ERR_INVALID;  // overlapping buffers
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(st);
  if (dt == LA_F32) return cuda_status(launch_transpose32(W, 0, Wp, rows, 1, rows, cols, cs));
  return cuda_status(cudaMemcpyAsync(Wp, W, bytes, cudaMemcpyDeviceToDevice, cs));
}

la_status la_layer_attn_prepared(const void* x, const void* gamma, const void* beta, float eps, const void* Wqkv_p,
                                 const void* bqkv, const void* Wo_p, const void* bo, void* y, int B, int S,
                                 int d_model, int H, int causal, const int32_t* kv_len, la_dtype dt, void* ws,
                                 size_t ws_bytes, la_stream_t st) {
  la_status s = check_layer_args(x, Wqkv_p, bqkv, y, ws, B, S, d_model, H, kv_len, dt);
  if (s != LA_OK) return s;
  if (gamma != nullptr || beta != nullptr) {
    s = check_ln_args(gamma, beta, eps);
    if (s != LA_OK) return s;
  }
  if (Wo_p != nullptr) {
    s = check_out_proj_args(ws, Wo_p, bo, y, static_cast<long long>(B) * S, d_model, dt);
    if (s != LA_OK) return s;
  } else if (bo != nullptr) {
    return LA_ERR_INVALID;
  }
  return run_block(x, gamma, beta, eps, Wqkv_p, bqkv, Wo_p, bo, y, B, S, d_model, H, causal, kv_len, dt, ws,
                   ws_bytes, reinterpret_cast<cudaStream_t>(st), true);
}

size_t la_workspace_size(int op, int B, int H, int S_q, int S_kv, int D, la_dtype dt) {
  const size_t bad = static_cast<size_t>(-1);
  if (check_attn_args(B, H, S_q, S_kv, D, 1.f, dt) != LA_OK) return bad;
  switch (op) {
    case LA_OP_ATTN_FWD:
      return attn_ws_bytes(dt, B, H, S_q, S_kv, D, true);
    case LA_OP_ATTN_CHUNKED:  // (an fp32 cache holds V^T already)
      return attn_ws_bytes(dt, B, H, S_q, S_kv, D, false);
    case LA_OP_LAYER_ATTN: {
      if (S_q != S_kv) return bad;
      return layer_fixed_bytes(B, S_q, H * D, H, dt) + attn_ws_bytes(dt, B, H, S_q, S_kv, D, false);
    }
    case LA_OP_QKV_PROJ:
      return wt_bytes(dt, H * D);
    case LA_OP_OUT_PROJ:
      return wot_bytes(dt, H * D);
    case LA_OP_LAYER_ATTN_OUT:
    case LA_OP_LAYER_ATTN_LN: {
      if (S_q != S_kv) return bad;
      return block_fixed_bytes(B, S_q, H * D, H, dt, op == LA_OP_LAYER_ATTN_LN, true) +
             attn_ws_bytes(dt, B, H, S_q, S_kv, D, false);
    }
    default:
      return bad;
  }
}

// Device address of la_noalloc_scratch on the current device.  Host code only
// has a stand-in symbol for it, so the address is looked up once per device
// (with that device current) and cached.
static la_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[la::kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= la::kMaxDevices) return LA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, la_noalloc_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return LA_OK;
}

la_status la_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, int B, int H, int S_q, int S_kv,
                              int D, int causal, float scale, const int32_t* kv_len, la_dtype dt, la_stream_t st) {
  if ((!q || !o) && S_q != 0) return LA_ERR_INVALID;
  if ((!k || !v) && S_kv != 0) return LA_ERR_INVALID;
  la_status s = check_attn_args(B, H, S_q, S_kv, D, scale, dt);
  if (s != LA_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LA_ERR_INVALID;
  if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return LA_ERR_INVALID;
  if (S_q == 0) return LA_OK;
  // fp32 needs V transposed in the scratch; beyond the array's size: refuse
  if (vt_bytes(dt, B, H, S_kv, D) > kNoAllocScratchBytes) return LA_ERR_WORKSPACE;
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != LA_OK) return s;
  if (S_kv == 0) k = v = q;  // no key is ever loaded; the maps only need a valid base
  // Split partials go after the fp32 V^T; the split plan takes only what fits.
  // Nothing in the scratch needs to start at zero: every byte a call reads is
  // written earlier in the same call.
  const KVView kv{k, v, S_kv, nullptr, 0};
  return run_attention(q, kv, o, static_cast<long long>(H) * S_q * D, static_cast<long long>(S_q) * D, D, B, H,
                       S_q, S_kv, D, causal, scale, kv_len, dt, scratch, kNoAllocScratchBytes,
                       reinterpret_cast<cudaStream_t>(st));
}

la_status la_profile_start(int max_launches) {
  if (max_launches < 1) return LA_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (auto& r : g_prof) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof.clear();
  g_prof.reserve(static_cast<size_t>(max_launches));
  g_prof_max = static_cast<size_t>(max_launches);
  g_prof_on.store(true);
  return LA_OK;
}

int la_profile_stop(const char** names, float* ms, int max) {
  g_prof_on.store(false);
  std::lock_guard<std::mutex> lock(g_prof_mu);
  int n = 0;
  bool ok = true;
  for (auto& r : g_prof) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      ok = false;
    if (n < max && names != nullptr && ms != nullptr) {
      names[n] = r.name;
      ms[n] = t;
    }
    ++n;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof.clear();
  return ok ? (n < max ? n : max) : -1;
}

la_status la_get_last_error(la_stream_t st) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(st));
  if (e != cudaSuccess) return LA_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, la_device_error_word, sizeof w) != cudaSuccess) return LA_ERR_CUDA;
  g_last_word.store(w);
  if (w != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(la_device_error_word, &zero, sizeof zero) != cudaSuccess) return LA_ERR_CUDA;
  }
  if (w & DEVERR_TIMEOUT) return LA_ERR_TIMEOUT;
  if (w & DEVERR_INTERNAL) return LA_ERR_INTERNAL;
  return LA_OK;
}

uint32_t la_last_error_detail(void) { return g_last_word.load(); }

la_status la_debug_shrink_output_extent(int mode) {
  if (mode != 0 && mode != 1) return LA_ERR_INVALID;
  g_shrink_once.store(mode);
  return LA_OK;
}

int la_is_checked_build(void) { return LA_CHECKED; }

la_status la_debug_inject_timeout(int mode) {
  if (mode != 0 && mode != 1) return LA_ERR_INVALID;
  g_skip_loads_once.store(mode);
  return LA_OK;
}

const char* la_status_string(la_status s) {
  switch (s) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID: return "LA_ERR_INVALID: invalid argument";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: unsupported head dim, dtype or size";
    case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE: workspace too small";
    case LA_ERR_CUDA: return "LA_ERR_CUDA: CUDA runtime call or launch failed";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a device-side wait ran out";
    case LA_ERR_INTERNAL: return "LA_ERR_INTERNAL: device consistency check failed";
  }
  return "unknown la_status";
}

}  // extern "C"
