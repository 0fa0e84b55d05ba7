/*
 * layerattn.h -- C ABI of the GB300 (sm_103a) attention-sublayer library
 * liblayerattn.so.
 *
 * The operation is the attention step of a transformer inference layer,
 * O = softmax(Q K^T * scale) V ("Shape-Aware Attention", section Inspiration,
 * the attention equation), computed by online softmax over key/value tiles so
 * that the [B, H, S_q, S_kv] score matrix never exists ("GPU Kernel for a
 * Transformer Layer", section What we learned), with causal masking ("GPU
 * Kernel for a Transformer Layer", section How we built it), an optional key
 * padding mask, a fused Q/K/V projection feeding it and a chunked
 * long-context mode that streams query windows against a growing key/value
 * cache ("Roofline", sections What it does and How we built it).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned, to contiguous row-major tensors.  The library allocates no
 *    device memory on any call; scratch comes from the caller's workspace
 *    `ws` of `ws_bytes` bytes (size it with la_workspace_size()).
 *  - q, k, v, o are head-major [B, H, S, D] unless stated otherwise.
 *  - Element types: LA_F32 (fp32 storage; the products run on the tensor
 *    cores in TF32 with fp32 accumulation), LA_BF16 and LA_F16 (half-precision
 *    storage; fp32 softmax statistics and fp32 accumulation).  Outputs have
 *    the input element type, rounded to nearest-even.
 *  - Supported head dimension: D in {64, 128}.  Any other D returns
 *    LA_ERR_UNSUPPORTED; there is no fallback path.
 *  - Causal masking aligns query rows to the END of the key range: query row
 *    i (0 <= i < S_q) is absolute position S_kv - S_q + i and sees keys
 *    j <= S_kv - S_q + i.  With S_q == S_kv this is ordinary causal attention.
 *  - kv_len (nullable) is a device array of B int32: keys j >= kv_len[b] of
 *    batch entry b are masked out (key padding).  Values above S_kv are
 *    clamped to S_kv.
 *  - A query row with no visible key yields a zero output row.
 *  - scale must be positive and finite (usually 1/sqrt(D)).
 *  - Every call is asynchronous on the caller's stream `st` (a cudaStream_t;
 *    NULL is the legacy default stream).  Arguments are validated on the
 *    host before any launch; an invalid call launches nothing and returns a
 *    status.  Device-side failures (a bounded wait that ran out) are latched
 *    in a device error word and reported by la_get_last_error().
 *  - Nothing throws, aborts, prints or traps across this boundary.
 *  - Inputs must be finite.  Masked keys are excluded by their weight, so
 *    padding keys must hold finite values.
 */
#ifndef LAYERATTN_H
#define LAYERATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID = 1,      /* bad pointer, size, alignment or parameter  */
    LA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (D, dtype)       */
    LA_ERR_WORKSPACE = 3,    /* ws smaller than the call needs             */
    LA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed       */
    LA_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out         */
    LA_ERR_INTERNAL = 6      /* a device-side consistency check failed     */
} la_status;

typedef enum { LA_F32 = 0, LA_BF16 = 1, LA_F16 = 2 } la_dtype;

/* Operation codes for la_workspace_size(). */
typedef enum {
    LA_OP_ATTN_FWD = 0,
    LA_OP_ATTN_CHUNKED = 1,
    LA_OP_LAYER_ATTN = 2,
    LA_OP_QKV_PROJ = 3,
    LA_OP_OUT_PROJ = 4,
    LA_OP_LAYER_ATTN_OUT = 5,
    LA_OP_LAYER_ATTN_LN = 6
} la_op;

/*
 * Growing key/value cache for the chunked mode.  k and v are caller-owned
 * device buffers of element type `dtype`: k [B, H, S_max, D]; v the same
 * for bf16/fp16, and for fp32 V transposed, [B, H, D, S_max] (the TF32
 * tensor cores take the PV product's V only with keys contiguous, so each
 * window's values are appended transposed once instead of the whole cache
 * being transposed on every window; fp32 S_max must then be a multiple of
 * 4).  Positions [0, len) hold valid keys/values.  la_attn_chunked()
 * appends to it and advances `len` on the host struct.
 */
typedef struct {
    void *k;
    void *v;
    int B, H, D, S_max, len;
    la_dtype dtype;
} la_kv_cache;

/*
 * Fused Q/K/V projection ("Roofline", sections What it does and How we built
 * it: one product x.Wqkv instead of three).
 *   x     [B, S, d_model]            input activations
 *   Wqkv  [d_model, 3*d_model]       columns: the Q block, the K block, the V
 *                                    block; inside each block head h owns
 *                                    columns h*D .. h*D+D-1 (D = d_model / H)
 *   bqkv  [3*d_model] or NULL        bias, same column order
 *   q,k,v [B, H, S, D] outputs       y = x.Wqkv + bqkv split per head; q is
 *                                    further multiplied by q_scale
 * d_model must be H*D with D in {64, 128}.  S >= 0 (S == 0 is a no-op).
 * ws, ws_bytes: workspace of la_workspace_size(LA_OP_QKV_PROJ, B, H, S, S,
 *   D, dt) bytes; fp32 needs 3*d_model*d_model*4 bytes there (the TF32
 *   tensor cores take K-major operands only, so the weight is transposed
 *   into it first), bf16/fp16 need none (ws may be NULL).  The workspace
 *   argument is an addition to the projection's statement as a product
 *   x.Wqkv + b: every scratch buffer of this library comes from the caller,
 *   and the fp32 transpose needs one.
 * Returns LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE or
 * LA_ERR_CUDA.
 */
la_status la_qkv_proj(const void *x, const void *Wqkv, const void *bqkv,
                      void *q, void *k, void *v,
                      int B, int S, int d_model, int H, float q_scale,
                      la_dtype dt, void *ws, size_t ws_bytes, la_stream_t st);

/*
 * Attention forward ("Shape-Aware Attention", section Inspiration, the
 * attention equation; online softmax per "GPU Kernel for a Transformer
 * Layer", section What we learned).
 *   q [B, H, S_q, D]; k, v [B, H, S_kv, D]; o [B, H, S_q, D] output.
 *   causal, scale, kv_len: see the conventions above.
 *   ws, ws_bytes: workspace.  With at least
 *     la_workspace_size(LA_OP_ATTN_FWD, ...) bytes the call schedules its
 *     work items dynamically (one thread block per SM drawing items by
 *     ticket; the ticket words live in ws) and may split long key ranges
 *     across thread blocks and merge the partial results (split-KV).  With
 *     less it gives every work item a thread block of its own and splits
 *     only as far as ws allows.  Results agree to rounding either way.
 *     bf16/fp16 need no workspace (ws may be NULL, slower on large shapes).
 *     fp32 needs at least B*H*D*round_up(S_kv, 4)*4 bytes (rounded up to
 *     256): V is transposed there first, because the TF32 tensor cores take
 *     K-major operands only; with less the call returns LA_ERR_WORKSPACE.
 *     ws needs no clearing.  Calls whose kernels may run at the same time
 *     (on different streams, or a graph replay beside a direct call) must
 *     use disjoint workspaces; a call may reuse its workspace as soon as the
 *     previous call on it is ordered before it (same stream).
 * S_q == 0 is a no-op; S_kv == 0 writes zero rows.  q and o may be NULL
 * only when S_q == 0, k and v only when S_kv == 0.
 * Returns LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE or
 * LA_ERR_CUDA.
 */
la_status la_attn_fwd(const void *q, const void *k, const void *v, void *o,
                      int B, int H, int S_q, int S_kv, int D, int causal, float scale,
                      const int32_t *kv_len, la_dtype dt,
                      void *ws, size_t ws_bytes, la_stream_t st);

/*
 * One window of the chunked long-context mode ("Roofline", sections What it
 * does and How we built it: bounded-memory query windows against a growing
 * key/value cache).  The window's keys and values
 *   k_chunk, v_chunk [B, H, chunk, D]
 * are appended to the cache at positions [len, len+chunk), then the window's
 * queries q_chunk [B, H, chunk, D] attend to cache positions [0, len+chunk)
 * (causal rows aligned to the end), writing o_chunk [B, H, chunk, D], and
 * cache->len grows by chunk.  Calling it window after window over a sequence
 * gives the same result as attending the whole sequence at once.
 * cache->len + chunk must not exceed cache->S_max; cache->dtype, B, H and D
 * describe all five tensors; an fp32 cache whose S_max is not a multiple of
 * 4 is refused (LA_ERR_INVALID).  ws: as for la_attn_fwd, sized with
 * la_workspace_size(LA_OP_ATTN_CHUNKED, B, H, chunk, S_max, D, dtype) (no
 * V^T scratch: an fp32 cache already holds V transposed).
 * On any non-OK status cache->len is unchanged.
 */
la_status la_attn_chunked(const void *q_chunk, const void *k_chunk, const void *v_chunk,
                          la_kv_cache *cache, void *o_chunk, int chunk, int causal,
                          float scale, void *ws, size_t ws_bytes, la_stream_t st);

/*
 * The attention sublayer as a layer runs it: la_qkv_proj (q_scale 1), then
 * attention per head with scale 1/sqrt(D), heads merged in the store:
 *   x [B, S, d_model], Wqkv [d_model, 3*d_model], bqkv [3*d_model] or NULL,
 *   o [B, S, d_model] with head h in columns h*D .. h*D+D-1.
 * The output projection is not applied (la_layer_attn_out applies it).  ws
 * must hold at least
 * la_workspace_size(LA_OP_LAYER_ATTN, B, H, S, S, d_model / H, dt) bytes
 * (the head-major q, k, v; for fp32 V is kept transposed and the weight's
 * transpose is kept too); otherwise LA_ERR_WORKSPACE.
 */
la_status la_layer_attn(const void *x, const void *Wqkv, const void *bqkv, void *o,
                        int B, int S, int d_model, int H, int causal,
                        const int32_t *kv_len, la_dtype dt,
                        void *ws, size_t ws_bytes, la_stream_t st);

/*
 * Output projection of the sublayer, the fourth of the layer's d x d
 * projections ("Shape-Aware Attention", section How we built it: the 8BSd^2
 * term of the per-layer FLOP count covers the Q, K, V and output
 * projections):
 *   y [M, d_model] = a [M, d_model] . Wo [d_model, d_model] + bo
 *   a   row-major activations (for the sublayer: the heads-merged attention
 *       output, M = B*S)
 *   Wo  [d_model, d_model] row-major (input features are rows)
 *   bo  [d_model] or NULL
 * d_model must be a positive multiple of 64 (else LA_ERR_UNSUPPORTED); M >= 0
 * (M == 0 is a no-op).  fp32 runs the products in TF32 like the other
 * projections.  ws, ws_bytes: la_workspace_size(LA_OP_OUT_PROJ, 1, H, M, M,
 * D, dt) bytes for any H, D with H*D = d_model; fp32 needs
 * d_model*d_model*4 bytes there (Wo is transposed into it first; TF32
 * products take K-major operands only), bf16/fp16 none (ws may be NULL).
 * a and y must not overlap.
 * Returns LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE or
 * LA_ERR_CUDA.
 */
la_status la_out_proj(const void *a, const void *Wo, const void *bo, void *y,
                      int M, int d_model, la_dtype dt,
                      void *ws, size_t ws_bytes, la_stream_t st);

/*
 * The sublayer with its output projection: la_layer_attn, then la_out_proj
 * on its heads-merged output, which is stored in the element type dt in
 * between (as a separate la_out_proj call would see it):
 *   x [B, S, d_model], Wqkv [d_model, 3*d_model], bqkv [3*d_model] or NULL,
 *   Wo [d_model, d_model], bo [d_model] or NULL,
 *   y [B, S, d_model] = merge_heads(attention) . Wo + bo.
 * Arguments otherwise as for la_layer_attn.  ws must hold at least
 * la_workspace_size(LA_OP_LAYER_ATTN_OUT, B, H, S, S, d_model / H, dt)
 * bytes (the intermediate output, the fp32 weight transposes and the
 * sublayer's own workspace); otherwise LA_ERR_WORKSPACE.
 */
la_status la_layer_attn_out(const void *x, const void *Wqkv, const void *bqkv,
                            const void *Wo, const void *bo, void *y,
                            int B, int S, int d_model, int H, int causal,
                            const int32_t *kv_len, la_dtype dt,
                            void *ws, size_t ws_bytes, la_stream_t st);

/*
 * LayerNorm over the last dimension, the normalisation in front of the
 * attention sublayer of a pre-norm layer ("Shape-Aware Attention", section
 * What's next: fusing LayerNorm; statistics in fp32 as "GPU Kernel for a
 * Transformer Layer", section What we learned, asks of reductions):
 *   y[r, c] = (x[r, c] - mean_r) / sqrt(var_r + eps) * gamma[c] + beta[c]
 * with mean_r and the biased variance var_r (mean squared deviation) of row
 * r, computed in fp32 in two passes over the row.
 *   x, y  [M, d] row-major (may be the same buffer); gamma, beta [d]
 * d must be a positive multiple of 64 (else LA_ERR_UNSUPPORTED); eps >= 0
 * and finite; all four pointers 16-byte aligned.  M == 0 is a no-op.
 * Returns LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED or LA_ERR_CUDA.
 */
la_status la_layernorm(const void *x, const void *gamma, const void *beta, void *y,
                       int M, int d, float eps, la_dtype dt, la_stream_t st);

/*
 * The pre-norm attention block: LayerNorm of x as la_layernorm computes it,
 * fused into the Q/K/V projection ("Shape-Aware Attention", section What's
 * next: fusing LayerNorm), then the attention of la_layer_attn and, when Wo
 * is not NULL, the output projection of la_out_proj.  A pre-pass computes
 * each row's statistics (mean and 1/sqrt(var + eps), fp32, 8 bytes a row);
 * the projection normalises every x tile in shared memory as it loads it and
 * rounds it to the operand type of its products (dt; TF32 for fp32), so the
 * normalised activations are never written to memory:
 *   y [B, S, d_model] = [merge_heads(attention(LN(x) . Wqkv + bqkv)) . Wo + bo]
 * gamma, beta [d_model] and eps as for la_layernorm; Wo [d_model, d_model]
 * and bo [d_model] may be NULL (bo must be NULL when Wo is).  Arguments
 * otherwise as for la_layer_attn.  The layer's residual add is not part of
 * it.  ws must hold at least
 * la_workspace_size(LA_OP_LAYER_ATTN_LN, B, H, S, S, d_model / H, dt) bytes
 * (sized for the output projection; without it less is needed); otherwise
 * LA_ERR_WORKSPACE.
 */
la_status la_layer_attn_ln(const void *x, const void *gamma, const void *beta, float eps,
                           const void *Wqkv, const void *bqkv,
                           const void *Wo, const void *bo, void *y,
                           int B, int S, int d_model, int H, int causal,
                           const int32_t *kv_len, la_dtype dt,
                           void *ws, size_t ws_bytes, la_stream_t st);

/*
 * Weights prepared once, as a server does when it loads a model: the layout
 * the projection kernels read, so that la_layer_attn_prepared does no
 * per-call conversion of its constant weights.  W [rows, cols] row-major
 * (Wqkv: rows = d_model, cols = 3*d_model; Wo: rows = cols = d_model);
 * Wp: a caller-owned buffer of rows*cols elements of the same type, not
 * overlapping W.  fp32 writes the transpose W^T [cols, rows] (the TF32
 * tensor cores take K-major operands only); bf16/fp16 copy W unchanged.
 * rows and cols must be multiples of 64.  Asynchronous on st.  Returns LA_OK,
 * LA_ERR_INVALID, LA_ERR_UNSUPPORTED or LA_ERR_CUDA.  The pages have no
 * counterpart (their weights live in a framework's modules).
 */
la_status la_prepare_weight(const void *W, void *Wp, int rows, int cols, la_dtype dt, la_stream_t st);

/*
 * The block of la_layer_attn_ln on prepared weights: Wqkv_p and Wo_p are
 * la_prepare_weight's outputs for Wqkv and Wo.  gamma and beta may both be
 * NULL (no LayerNorm: the sublayer of la_layer_attn, or with Wo_p that of
 * la_layer_attn_out); Wo_p and bo may be NULL (no output projection; bo
 * must be NULL when Wo_p is).  ws: as for la_layer_attn_ln (its size covers
 * every form).  Results equal those of the unprepared calls bit for bit.
 */
la_status la_layer_attn_prepared(const void *x, const void *gamma, const void *beta, float eps,
                                 const void *Wqkv_p, const void *bqkv, const void *Wo_p, const void *bo, void *y,
                                 int B, int S, int d_model, int H, int causal,
                                 const int32_t *kv_len, la_dtype dt,
                                 void *ws, size_t ws_bytes, la_stream_t st);

/*
 * la_attn_fwd without a workspace, for callers that cannot allocate device
 * memory: a host framework whose plugin interface hands over only the input
 * and output tensors, a service that sizes all of its device memory once at
 * start-up and allows no allocation afterwards, or a latency-critical loop
 * that must not call cudaMalloc (which can synchronise the device).  The
 * pages have no counterpart; it is an addition of this library.
 *
 * Same arguments, meaning and result as la_attn_fwd, minus ws/ws_bytes.  Its
 * scratch (the work-item ticket words, split-KV partials; for fp32 also V
 * transposed) is one static device array of 16 MiB inside the library,
 * which every GPU that loads the library keeps until the process exits; the
 * call itself allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).
 *   - Limit: fp32 needs B*H*D*round_up(S_kv, 4)*4 bytes of it (rounded up to
 *     256); a call beyond 16 MiB returns LA_ERR_WORKSPACE and launches
 *     nothing.  Split partials take what is left; a call that would want more
 *     simply splits less (bf16/fp16 never fail for lack of scratch).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose kernels can overlap
 *     on the GPU (different streams without ordering) race on it: serialise
 *     them.
 * Returns LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE or
 * LA_ERR_CUDA.
 */
la_status la_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o,
                              int B, int H, int S_q, int S_kv, int D, int causal, float scale,
                              const int32_t *kv_len, la_dtype dt, la_stream_t st);

/*
 * Workspace bytes an operation wants (0 if none).  op is an la_op; the
 * remaining arguments are those of the call (for LA_OP_ATTN_CHUNKED pass
 * S_q = chunk and S_kv = the cache's S_max; for LA_OP_LAYER_ATTN,
 * LA_OP_LAYER_ATTN_OUT, LA_OP_LAYER_ATTN_LN and LA_OP_QKV_PROJ pass S_q =
 * S_kv = S and
 * D = d_model / H; for LA_OP_OUT_PROJ see la_out_proj).  Returns (size_t)-1
 * for invalid arguments.  Host only; touches no device.
 */
size_t la_workspace_size(int op, int B, int H, int S_q, int S_kv, int D, la_dtype dt);

/*
 * Synchronises `st`, then reports and clears the device error word of the
 * current device: LA_ERR_TIMEOUT if a kernel's bounded wait ran out since
 * the last query, LA_ERR_INTERNAL if a device consistency check failed,
 * LA_ERR_CUDA if the stream itself reports an error, else LA_OK.
 */
la_status la_get_last_error(la_stream_t st);

/*
 * The raw device error word read by the latest la_get_last_error() of this
 * process: bit 0 a bounded wait ran out, bit 1 a consistency check failed,
 * bit 8+i wait site i gave up (0 Q loaded, 1 K loaded (or the K and V tiles of
 * a stage, where they share a barrier), 2 V loaded, 3 K slot free, 4 V slot
 * free, 5 scores ready, 6 probabilities ready, 7 output ready,
 * 8 projection stage loaded, 9 projection stage free, 10 projection
 * accumulator ready, 11 projection accumulator free).  For diagnostics; 0
 * when all was well.
 */
uint32_t la_last_error_detail(void);

/*
 * Test hook for the failure path (the pages have no counterpart).  mode 1:
 * the next attention launch of this process issues none of its tile loads,
 * so every consumer's bounded wait runs out (about a second); that kernel
 * writes no output, the call itself returns LA_OK and the next
 * la_get_last_error() returns LA_ERR_TIMEOUT, with the CUDA context intact.
 * mode 0 withdraws a pending request.  Nothing faults, traps or hangs.
 * Returns LA_OK, or LA_ERR_INVALID for another mode.
 */
la_status la_debug_inject_timeout(int mode);

/*
 * The checked build: liblayerattn_checked.so is the same library compiled
 * with bounds checks on every global store of the attention, merge and
 * projection kernels (each flat element index against its buffer's extent).
 * A store that would leave its buffer is skipped and the next
 * la_get_last_error() returns LA_ERR_INTERNAL; nothing faults.  For
 * debugging and tests; slower.  la_is_checked_build() returns 1 there, 0 in
 * liblayerattn.so.
 */
int la_is_checked_build(void);

/*
 * Test hook for the checked build (the pages have no counterpart).  mode 1:
 * the next attention launch declares its output buffer one row (D elements)
 * shorter than it is, so the checked build skips the stores of the last row
 * and reports LA_ERR_INTERNAL; the normal build ignores extents and writes
 * every row.  mode 0 withdraws a pending request.  Returns LA_OK, or
 * LA_ERR_INVALID for another mode.
 */
la_status la_debug_shrink_output_extent(int mode);

/*
 * Per-launch device timing, for measurement (the pages time their kernels
 * with CUDA events on the stream; "Shape-Aware Attention", How we built it).
 * la_profile_start(n): the next launches of this process (at most n, from
 * any entry point) are each bracketed by two CUDA events recorded on the
 * stream the kernel is launched on.  While recording is on, kernels are
 * launched without programmatic dependent launch and an event sits between
 * consecutive kernels of a call, so each kernel's time is its own (the
 * overlap of a kernel's set-up with the previous kernel is lost).  The events are
 * created on the host as launches are recorded (no device memory); do not
 * record during stream capture.
 * la_profile_stop(names, ms, max): turns recording off, waits for the
 * recorded events, writes up to max (kernel name, milliseconds) pairs in
 * launch order (names point to static strings) and returns how many were
 * written, or -1 if a CUDA call failed.  Returns LA_ERR_INVALID for n < 1.
 */
la_status la_profile_start(int max_launches);
int la_profile_stop(const char **names, float *ms, int max);

/* Static, human-readable name of a status. */
const char *la_status_string(la_status s);

#ifdef __cplusplus
}
#endif

#endif /* LAYERATTN_H */
