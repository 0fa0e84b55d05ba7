/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU oracle for the attention sublayer, in
 * fp64.  Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg may load it.  The product (the CUDA library) never calls it,
 * and the two share no code, header, table or helper.
 *
 * What it computes (sources, by page and section):
 *   - Scaled dot-product attention, softmax(Q K^T / sqrt(d_k)) V:
 *     "Shape-Aware Attention", section Inspiration (the attention equation).
 *     Here the scale is a parameter; callers pass 1/sqrt(D).
 *   - Causal masking: "GPU Kernel for a Transformer Layer", section How we
 *     built it ("online-softmax causal attention"); with S_q != S_kv the query
 *     rows are aligned to the END of the key range (query i sits at absolute
 *     position S_kv - S_q + i), the only alignment under which attending a
 *     chunk against a growing key/value cache equals unchunked attention
 *     ("Roofline", section How we built it).
 *   - Key padding: "GPU Kernel for a Transformer Layer", section How we built
 *     it (padding masks).  Keys j >= kv_len[b] are excluded.
 *   - Online softmax (running max, running sum, rescaled accumulator over
 *     key/value blocks): "GPU Kernel for a Transformer Layer", section What we
 *     learned.  oracle_attn_online() takes those steps in fp64.
 *   - Fused Q/K/V projection (one x.Wqkv product instead of three):
 *     "Roofline", sections What it does / How we built it.
 *   - Chunked long-context mode (query windows against a growing K/V cache):
 *     "Roofline", sections What it does / How we built it.
 *   - Split-KV partials merged by log-sum-exp: the same algebra as the online
 *     softmax above, applied to disjoint key ranges.
 *   - Output projection y = o Wo + bo after the heads are merged: the
 *     fourth d x d projection of the layer ("Shape-Aware Attention", section
 *     How we built it: the 8BSd^2 term counts Q, K, V and output).
 *   - LayerNorm before the projection (the pre-norm block): "Shape-Aware
 *     Attention", section What's next (fusing LayerNorm).
 *
 * Readings taken where the pages are silent:
 *   - a query row with no valid key returns a zero row;
 *   - inputs are the exact stored values (fp32, bf16 or fp16) widened to fp64;
 *     nothing is rounded inside the oracle.
 *   - the sublayer's attention output enters the output projection
 *     unrounded (the GPU stores it in the model's element type first);
 *     likewise the normalised activations enter the projection unrounded;
 *   - LayerNorm divides by sqrt(var + eps) with the biased variance (the
 *     mean of squared deviations), eps a parameter.
 *
 * Every function here is pinned by tests that do not re-type its formula:
 * closed forms (Q = 0 gives the mean of V, S_kv = 1 returns v_0, two keys give
 * a logistic weight), invariants (rows of P sum to 1, key permutation and key
 * shift invariance, linearity in V), brute force on tiny shapes and a library
 * routine for the special case (torch CPU float64 scaled_dot_product_attention).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type codes of the input buffers */
enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2, ORC_F16 = 3 };

/* IEEE 754 binary16 -> double, from the format's definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 word. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load(const void *p, int dt, long long idx)
{
    switch (dt) {
    case ORC_F64: return ((const double *)p)[idx];
    case ORC_F32: return (double)((const float *)p)[idx];
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t *)p)[idx]);
    case ORC_F16: return half_bits_to_double(((const uint16_t *)p)[idx]);
    default: return NAN;
    }
}

/* element (b, h, s, d) of a contiguous [B, H, S, D] tensor */
static long long bhsd(int b, int h, long long s, int d, int H, long long S, int D)
{
    return (((long long)b * H + h) * S + s) * D + d;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the later calls (for timing the oracle on one core as well as on
   all of them); n < 1 restores the default.  Touches no arithmetic. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n >= 1 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

/* Is key j visible to query row i of batch b?  Definition of the mask. */
static int key_valid(long long i, long long j, long long S_q, long long S_kv,
                     int causal, long long kv_len_b)
{
    long long off = S_kv - S_q;           /* query i is absolute position i + off */
    if (j >= kv_len_b) return 0;          /* key padding */
    if (causal && j > i + off) return 0;  /* no attending to the future */
    return 1;
}

/*
 * One output row: o = sum_j softmax_j(s) v_j over the valid keys, with
 * s_j = scale * <q_i, k_j>.  The max is subtracted before exp only to keep exp
 * finite; it cancels in the quotient.
 * s: caller scratch of S_kv doubles.  qrow: caller scratch of D doubles.
 */
static void attn_row(const void *q, const void *k, const void *v, int dt,
                     int b, int h, long long i, int H, long long S_q, long long S_kv,
                     int D, int causal, double scale, long long kv_len_b,
                     double *s, double *qrow, double *out)
{
    for (int d = 0; d < D; ++d) qrow[d] = load(q, dt, bhsd(b, h, i, d, H, S_q, D));
    double m = -INFINITY;
    for (long long j = 0; j < S_kv; ++j) {
        if (!key_valid(i, j, S_q, S_kv, causal, kv_len_b)) { s[j] = -INFINITY; continue; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qrow[d] * load(k, dt, bhsd(b, h, j, d, H, S_kv, D));
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (m == -INFINITY) return;           /* no valid key: zero row */
    double l = 0.0;
    for (long long j = 0; j < S_kv; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < D; ++d) out[d] += p * load(v, dt, bhsd(b, h, j, d, H, S_kv, D));
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
}

static long long kvlen_of(const int32_t *kv_len, int b, long long S_kv)
{
    return kv_len ? (long long)kv_len[b] : S_kv;
}

/*
 * Full attention.  q: [B,H,S_q,D]; k, v: [B,H,S_kv,D], all of element type dt.
 * kv_len: [B] or NULL.  o: [B,H,S_q,D] fp64.  Returns 0, or -1 on bad input.
 */
int oracle_attn(const void *q, const void *k, const void *v, int dt, double *o,
                int B, int H, long long S_q, long long S_kv, int D, int causal,
                double scale, const int32_t *kv_len)
{
    if (B < 0 || H < 0 || S_q < 0 || S_kv < 0 || D <= 0) return -1;
    long long rows = (long long)B * H * S_q;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(S_kv > 0 ? S_kv : 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qrow) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (long long r = 0; r < rows; ++r) {
                int b = (int)(r / ((long long)H * S_q));
                int h = (int)((r / S_q) % H);
                long long i = r % S_q;
                attn_row(q, k, v, dt, b, h, i, H, S_q, S_kv, D, causal, scale,
                         kvlen_of(kv_len, b, S_kv), s, qrow, o + r * D);
            }
        }
        free(s);
        free(qrow);
    }
    return err ? -1 : 0;
}

/*
 * Selected rows only (for shapes whose full output is too costly on a CPU).
 * rows: n triples (b, h, i).  out: [n, D] fp64.
 */
int oracle_attn_rows(const void *q, const void *k, const void *v, int dt,
                     int B, int H, long long S_q, long long S_kv, int D, int causal,
                     double scale, const int32_t *kv_len,
                     const int64_t *rows, long long n, double *out)
{
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(S_kv > 0 ? S_kv : 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qrow) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long long r = 0; r < n; ++r) {
                int b = (int)rows[3 * r], h = (int)rows[3 * r + 1];
                long long i = rows[3 * r + 2];
                if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= S_q) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                attn_row(q, k, v, dt, b, h, i, H, S_q, S_kv, D, causal, scale,
                         kvlen_of(kv_len, b, S_kv), s, qrow, out + r * D);
            }
        }
        free(s);
        free(qrow);
    }
    return err ? -1 : 0;
}

/*
 * The probability matrix P = softmax(scale Q K^T) with masked entries 0, for
 * tiny shapes: p: [B,H,S_q,S_kv] fp64.
 */
int oracle_attn_probs(const void *q, const void *k, int dt, double *p,
                      int B, int H, long long S_q, long long S_kv, int D, int causal,
                      double scale, const int32_t *kv_len)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (long long i = 0; i < S_q; ++i) {
                double *row = p + (((long long)b * H + h) * S_q + i) * S_kv;
                long long kl = kvlen_of(kv_len, b, S_kv);
                double m = -INFINITY;
                for (long long j = 0; j < S_kv; ++j) {
                    if (!key_valid(i, j, S_q, S_kv, causal, kl)) { row[j] = -INFINITY; continue; }
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += load(q, dt, bhsd(b, h, i, d, H, S_q, D)) *
                               load(k, dt, bhsd(b, h, j, d, H, S_kv, D));
                    row[j] = scale * dot;
                    if (row[j] > m) m = row[j];
                }
                double l = 0.0;
                for (long long j = 0; j < S_kv; ++j) {
                    row[j] = (m == -INFINITY || row[j] == -INFINITY) ? 0.0 : exp(row[j] - m);
                    l += row[j];
                }
                if (l > 0.0)
                    for (long long j = 0; j < S_kv; ++j) row[j] /= l;
            }
    return 0;
}

/*
 * Online softmax over key/value blocks of `block` keys, in the order the
 * method states it: per block, the running max m moves to max(m, block max),
 * the running sum l and the accumulator acc are rescaled by exp(m_old - m_new),
 * and the block's exp(s - m_new) terms are added; at the end o = acc / l.
 * Exact in real arithmetic, so it must agree with oracle_attn().
 */
int oracle_attn_online(const void *q, const void *k, const void *v, int dt, double *o,
                       int B, int H, long long S_q, long long S_kv, int D, int causal,
                       double scale, const int32_t *kv_len, long long block)
{
    if (block <= 0) return -1;
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    double *sblk = (double *)malloc(sizeof(double) * (size_t)block);
    if (!acc || !sblk) { free(acc); free(sblk); return -1; }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (long long i = 0; i < S_q; ++i) {
                long long kl = kvlen_of(kv_len, b, S_kv);
                double m = -INFINITY, l = 0.0;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (long long j0 = 0; j0 < S_kv; j0 += block) {
                    long long n = (S_kv - j0 < block) ? S_kv - j0 : block;
                    double bm = -INFINITY;
                    for (long long t = 0; t < n; ++t) {
                        long long j = j0 + t;
                        if (!key_valid(i, j, S_q, S_kv, causal, kl)) { sblk[t] = -INFINITY; continue; }
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d)
                            dot += load(q, dt, bhsd(b, h, i, d, H, S_q, D)) *
                                   load(k, dt, bhsd(b, h, j, d, H, S_kv, D));
                        sblk[t] = scale * dot;
                        if (sblk[t] > bm) bm = sblk[t];
                    }
                    double m_new = bm > m ? bm : m;
                    if (m_new == -INFINITY) continue;        /* nothing valid yet */
                    double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
                    l *= alpha;
                    for (int d = 0; d < D; ++d) acc[d] *= alpha;
                    for (long long t = 0; t < n; ++t) {
                        if (sblk[t] == -INFINITY) continue;
                        double p = exp(sblk[t] - m_new);
                        l += p;
                        for (int d = 0; d < D; ++d)
                            acc[d] += p * load(v, dt, bhsd(b, h, j0 + t, d, H, S_kv, D));
                    }
                    m = m_new;
                }
                double *out = o + (((long long)b * H + h) * S_q + i) * D;
                for (int d = 0; d < D; ++d) out[d] = (l > 0.0) ? acc[d] / l : 0.0;
            }
    free(acc);
    free(sblk);
    return 0;
}

/*
 * Split-KV: the key range [0, S_kv) is cut into n_split contiguous pieces of
 * ceil(S_kv / n_split) keys.  Each piece yields its own normalised partial
 * output O_s and log-sum-exp lse_s = m_s + log(l_s) (-inf when the piece has
 * no valid key).  The pieces merge as o = sum_s w_s O_s / sum_s w_s with
 * w_s = exp(lse_s - max_s lse_s).  Must agree with oracle_attn().
 */
int oracle_attn_split(const void *q, const void *k, const void *v, int dt, double *o,
                      int B, int H, long long S_q, long long S_kv, int D, int causal,
                      double scale, const int32_t *kv_len, int n_split)
{
    if (n_split <= 0) return -1;
    long long per = (S_kv + n_split - 1) / n_split;
    if (per == 0) per = 1;
    double *Os = (double *)malloc(sizeof(double) * (size_t)n_split * D);
    double *lse = (double *)malloc(sizeof(double) * (size_t)n_split);
    if (!Os || !lse) { free(Os); free(lse); return -1; }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (long long i = 0; i < S_q; ++i) {
                long long kl = kvlen_of(kv_len, b, S_kv);
                for (int sp = 0; sp < n_split; ++sp) {
                    long long j0 = (long long)sp * per, j1 = j0 + per;
                    if (j1 > S_kv) j1 = S_kv;
                    double m = -INFINITY;
                    for (long long j = j0; j < j1; ++j) {
                        if (!key_valid(i, j, S_q, S_kv, causal, kl)) continue;
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d)
                            dot += load(q, dt, bhsd(b, h, i, d, H, S_q, D)) *
                                   load(k, dt, bhsd(b, h, j, d, H, S_kv, D));
                        if (scale * dot > m) m = scale * dot;
                    }
                    double *Op = Os + (size_t)sp * D;
                    for (int d = 0; d < D; ++d) Op[d] = 0.0;
                    if (m == -INFINITY) { lse[sp] = -INFINITY; continue; }
                    double l = 0.0;
                    for (long long j = j0; j < j1; ++j) {
                        if (!key_valid(i, j, S_q, S_kv, causal, kl)) continue;
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d)
                            dot += load(q, dt, bhsd(b, h, i, d, H, S_q, D)) *
                                   load(k, dt, bhsd(b, h, j, d, H, S_kv, D));
                        double p = exp(scale * dot - m);
                        l += p;
                        for (int d = 0; d < D; ++d)
                            Op[d] += p * load(v, dt, bhsd(b, h, j, d, H, S_kv, D));
                    }
                    for (int d = 0; d < D; ++d) Op[d] /= l;
                    lse[sp] = m + log(l);
                }
                double M = -INFINITY;
                for (int sp = 0; sp < n_split; ++sp) if (lse[sp] > M) M = lse[sp];
                double *out = o + (((long long)b * H + h) * S_q + i) * D;
                for (int d = 0; d < D; ++d) out[d] = 0.0;
                if (M == -INFINITY) continue;
                double wsum = 0.0;
                for (int sp = 0; sp < n_split; ++sp) {
                    if (lse[sp] == -INFINITY) continue;
                    double w = exp(lse[sp] - M);
                    wsum += w;
                    for (int d = 0; d < D; ++d) out[d] += w * Os[(size_t)sp * D + d];
                }
                for (int d = 0; d < D; ++d) out[d] /= wsum;
            }
    free(Os);
    free(lse);
    return 0;
}

/*
 * Chunked long-context mode, step by step: a key/value cache starts empty;
 * for each window of `chunk` consecutive positions, that window's keys and
 * values are appended to the cache, then the window's queries attend to the
 * whole cache so far (causal rows aligned to the end of the cache).
 * q, k, v: full sequences [B,H,S,D]; o: [B,H,S,D] fp64.
 * The cache is a private fp64 copy [B,H,S,D] filled window by window.
 */
int oracle_attn_chunked(const void *q, const void *k, const void *v, int dt, double *o,
                        int B, int H, long long S, int D, int causal, double scale,
                        long long chunk)
{
    if (chunk <= 0) return -1;
    size_t n = (size_t)B * H * S * D;
    double *kc = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *vc = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *qw = (double *)malloc(sizeof(double) * (size_t)B * H * chunk * D);
    double *ow = (double *)malloc(sizeof(double) * (size_t)B * H * chunk * D);
    if (!kc || !vc || !qw || !ow) { free(kc); free(vc); free(qw); free(ow); return -1; }
    long long len = 0;
    int rc = 0;
    while (len < S && rc == 0) {
        long long c = (S - len < chunk) ? S - len : chunk;
        /* append this window's keys and values; the cache keeps [B,H,len+c,D] packed */
        double *kn = (double *)malloc(sizeof(double) * (size_t)B * H * (len + c) * D);
        double *vn = (double *)malloc(sizeof(double) * (size_t)B * H * (len + c) * D);
        if (!kn || !vn) { free(kn); free(vn); rc = -1; break; }
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h)
                for (long long j = 0; j < len + c; ++j)
                    for (int d = 0; d < D; ++d) {
                        long long dst = bhsd(b, h, j, d, H, len + c, D);
                        if (j < len) {
                            long long src = bhsd(b, h, j, d, H, len, D);
                            kn[dst] = kc[src];
                            vn[dst] = vc[src];
                        } else {
                            kn[dst] = load(k, dt, bhsd(b, h, j, d, H, S, D));
                            vn[dst] = load(v, dt, bhsd(b, h, j, d, H, S, D));
                        }
                    }
        memcpy(kc, kn, sizeof(double) * (size_t)B * H * (len + c) * D);
        memcpy(vc, vn, sizeof(double) * (size_t)B * H * (len + c) * D);
        free(kn);
        free(vn);
        /* this window's queries */
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h)
                for (long long i = 0; i < c; ++i)
                    for (int d = 0; d < D; ++d)
                        qw[bhsd(b, h, i, d, H, c, D)] = load(q, dt, bhsd(b, h, len + i, d, H, S, D));
        rc = oracle_attn(qw, kc, vc, ORC_F64, ow, B, H, c, len + c, D, causal, scale, NULL);
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h)
                for (long long i = 0; i < c; ++i)
                    for (int d = 0; d < D; ++d)
                        o[bhsd(b, h, len + i, d, H, S, D)] = ow[bhsd(b, h, i, d, H, c, D)];
        len += c;
    }
    free(kc);
    free(vc);
    free(qw);
    free(ow);
    return rc;
}

/*
 * Fused Q/K/V projection: y = x Wqkv + bqkv with x [B,S,d_model],
 * Wqkv [d_model, 3 d_model] (columns: the Q block, then K, then V; head h owns
 * columns h*D .. h*D+D-1 of each block), bqkv [3 d_model] or NULL.
 * Outputs q, k, v are head-major [B,H,S,D] fp64; q is multiplied by q_scale.
 * x has element type dt_x, Wqkv and bqkv dt_w (the pre-norm block passes its
 * fp64 normalised activations).
 */
static int qkv_proj_mixed(const void *x, int dt_x, const void *W, const void *bias, int dt_w,
                          double *q, double *k, double *v,
                          int B, long long S, int d_model, int H, double q_scale)
{
    if (H <= 0 || d_model % H) return -1;
    int D = d_model / H;
    long long N = 3LL * d_model;
    long long rows = (long long)B * S;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long r = 0; r < rows; ++r) {
        int b = (int)(r / S);
        long long s = r % S;
        for (long long n = 0; n < N; ++n) {
            double y = 0.0;
            for (int c = 0; c < d_model; ++c)
                y += load(x, dt_x, r * d_model + c) * load(W, dt_w, (long long)c * N + n);
            if (bias) y += load(bias, dt_w, n);
            int which = (int)(n / d_model);
            int h = (int)((n % d_model) / D);
            int d = (int)(n % D);
            long long dst = bhsd(b, h, s, d, H, S, D);
            if (which == 0) q[dst] = q_scale * y;
            else if (which == 1) k[dst] = y;
            else v[dst] = y;
        }
    }
    return 0;
}

int oracle_qkv_proj(const void *x, const void *W, const void *bias, int dt,
                    double *q, double *k, double *v,
                    int B, long long S, int d_model, int H, double q_scale)
{
    return qkv_proj_mixed(x, dt, W, bias, dt, q, k, v, B, S, d_model, H, q_scale);
}

/*
 * The attention sublayer as the layer runs it: the fused projection, then
 * attention per head with scale 1/sqrt(D), heads merged back into
 * o [B, S, d_model] (head h in columns h*D .. h*D+D-1).  The output
 * projection is not part of it.  x has element type dt_x, the weights dt_w.
 */
static int layer_attn_mixed(const void *x, int dt_x, const void *W, const void *bias, int dt_w, double *o,
                            int B, long long S, int d_model, int H, int causal,
                            const int32_t *kv_len)
{
    if (H <= 0 || d_model % H) return -1;
    int D = d_model / H;
    size_t n = (size_t)B * S * d_model;
    double *q = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *k = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *v = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *oh = (double *)malloc(sizeof(double) * (n ? n : 1));
    int rc = -1;
    if (q && k && v && oh) {
        rc = qkv_proj_mixed(x, dt_x, W, bias, dt_w, q, k, v, B, S, d_model, H, 1.0);
        if (rc == 0)
            rc = oracle_attn(q, k, v, ORC_F64, oh, B, H, S, S, D, causal, 1.0 / sqrt((double)D), kv_len);
        if (rc == 0)
            for (int b = 0; b < B; ++b)
                for (int h = 0; h < H; ++h)
                    for (long long s = 0; s < S; ++s)
                        for (int d = 0; d < D; ++d)
                            o[((long long)b * S + s) * d_model + (long long)h * D + d] =
                                oh[bhsd(b, h, s, d, H, S, D)];
    }
    free(q);
    free(k);
    free(v);
    free(oh);
    return rc;
}

int oracle_layer_attn(const void *x, const void *W, const void *bias, int dt, double *o,
                      int B, long long S, int d_model, int H, int causal,
                      const int32_t *kv_len)
{
    return layer_attn_mixed(x, dt, W, bias, dt, o, B, S, d_model, H, causal, kv_len);
}

/*
 * Output projection of the sublayer: the fourth of the layer's d x d
 * projections ("Shape-Aware Attention", section How we built it: the 8BSd^2
 * term of the per-layer FLOP count covers Q, K, V and output).
 *   y [M, d_out] = a [M, d_in] . Wo [d_in, d_out] + bo [d_out] (bo may be NULL)
 * a has its own element type code (the sublayer below passes its fp64
 * attention output); Wo and bo share dt_w.  y is fp64.
 */
int oracle_out_proj(const void *a, int dt_a, const void *W, const void *bias, int dt_w,
                    double *y, long long M, int d_in, int d_out)
{
    if (M < 0 || d_in < 1 || d_out < 1) return -1;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long r = 0; r < M; ++r) {
        for (int n = 0; n < d_out; ++n) {
            double acc = 0.0;
            for (int c = 0; c < d_in; ++c)
                acc += load(a, dt_a, r * d_in + c) * load(W, dt_w, (long long)c * d_out + n);
            if (bias) acc += load(bias, dt_w, n);
            y[r * d_out + n] = acc;
        }
    }
    return 0;
}

/*
 * The sublayer with its output projection: oracle_layer_attn, then
 * oracle_out_proj (d_model -> d_model) applied to its fp64 result, which is
 * not rounded in between.  y [B, S, d_model].  x has element type dt_x, the
 * weights dt_w.
 */
static int layer_attn_out_mixed(const void *x, int dt_x, const void *Wqkv, const void *bqkv,
                                const void *Wo, const void *bo, int dt_w, double *y,
                                int B, long long S, int d_model, int H, int causal,
                                const int32_t *kv_len)
{
    size_t n = (size_t)B * S * d_model;
    double *o = (double *)malloc(sizeof(double) * (n ? n : 1));
    if (!o) return -1;
    int rc = layer_attn_mixed(x, dt_x, Wqkv, bqkv, dt_w, o, B, S, d_model, H, causal, kv_len);
    if (rc == 0) rc = oracle_out_proj(o, ORC_F64, Wo, bo, dt_w, y, (long long)B * S, d_model, d_model);
    free(o);
    return rc;
}

int oracle_layer_attn_out(const void *x, const void *Wqkv, const void *bqkv,
                          const void *Wo, const void *bo, int dt, double *y,
                          int B, long long S, int d_model, int H, int causal,
                          const int32_t *kv_len)
{
    return layer_attn_out_mixed(x, dt, Wqkv, bqkv, Wo, bo, dt, y, B, S, d_model, H, causal, kv_len);
}

/*
 * LayerNorm over the last dimension ("Shape-Aware Attention", section
 * What's next: fusing LayerNorm; "GPU Kernel for a Transformer Layer",
 * section What we learned: its statistics are reductions kept in full
 * precision):
 *   mu_r = mean_c x[r,c],  var_r = mean_c (x[r,c] - mu_r)^2   (biased)
 *   y[r,c] = (x[r,c] - mu_r) / sqrt(var_r + eps) * gamma[c] + beta[c]
 * x [M, d] in element type dt_x (fp64 allowed), gamma and beta [d] in dt_g.
 */
int oracle_layernorm(const void *x, int dt_x, const void *gamma, const void *beta, int dt_g,
                     double *y, long long M, int d, double eps)
{
    if (M < 0 || d < 1 || !(eps >= 0.0)) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (long long r = 0; r < M; ++r) {
        double mu = 0.0, var = 0.0;
        for (int c = 0; c < d; ++c) mu += load(x, dt_x, r * d + c);
        mu /= d;
        for (int c = 0; c < d; ++c) {
            double t = load(x, dt_x, r * d + c) - mu;
            var += t * t;
        }
        var /= d;
        double rstd = 1.0 / sqrt(var + eps);
        for (int c = 0; c < d; ++c)
            y[r * d + c] = (load(x, dt_x, r * d + c) - mu) * rstd * load(gamma, dt_g, c) + load(beta, dt_g, c);
    }
    return 0;
}

/*
 * The pre-norm attention block: LayerNorm, then the sublayer (projection,
 * attention, heads merged), then the output projection when Wo is given.
 * Intermediate results stay in fp64.  y [B, S, d_model].
 */
int oracle_layer_attn_ln(const void *x, const void *gamma, const void *beta, double eps,
                         const void *Wqkv, const void *bqkv, const void *Wo, const void *bo, int dt,
                         double *y, int B, long long S, int d_model, int H, int causal,
                         const int32_t *kv_len)
{
    size_t n = (size_t)B * S * d_model;
    double *xn = (double *)malloc(sizeof(double) * (n ? n : 1));
    if (!xn) return -1;
    int rc = oracle_layernorm(x, dt, gamma, beta, dt, xn, (long long)B * S, d_model, eps);
    if (rc == 0) {
        if (Wo)
            rc = layer_attn_out_mixed(xn, ORC_F64, Wqkv, bqkv, Wo, bo, dt, y, B, S, d_model, H, causal, kv_len);
        else
            rc = layer_attn_mixed(xn, ORC_F64, Wqkv, bqkv, dt, y, B, S, d_model, H, causal, kv_len);
    }
    free(xn);
    return rc;
}

/* exposed so the tests can pin the widening of stored values */
double oracle_widen(const void *p, int dt, long long idx) { return load(p, dt, idx); }
