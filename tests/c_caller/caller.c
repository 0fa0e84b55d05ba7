/*
 * A plain C11 caller of liblayerattn.so: no Python, no torch.  It allocates
 * device memory with the CUDA runtime, calls the C ABI declared in
 * include/layerattn.h (attention with and without a workspace, the sublayer
 * on per-call and prepared weights, the chunked mode on a caller-owned
 * cache, per-launch timing), and checks the results element by element
 * against the fp64 oracle's C entry points (test infrastructure, linked from
 * oracle/_build/liboracle.so).  Exit status 0 when every check passes.
 *
 *   caller        run the GPU checks (needs a GPU)
 *   caller --abi  argument-validation checks only (no device is touched)
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "layerattn.h"

/* the oracle's C entry point and element codes (oracle/attn_oracle.c) */
int oracle_attn(const void *q, const void *k, const void *v, int dt, double *o, int B, int H, long long S_q,
                long long S_kv, int D, int causal, double scale, const int32_t *kv_len);
enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

static int failures = 0;
#define CHECK(cond, ...)                  \
    do {                                  \
        if (!(cond)) {                    \
            fprintf(stderr, __VA_ARGS__); \
            fputc('\n', stderr);          \
            ++failures;                   \
        }                                 \
    } while (0)

/* xorshift64*: a seeded stream of uniform doubles in [-1, 1) */
static uint64_t rng_state;
static double uniform(void) {
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (double)((rng_state * 0x2545F4914F6CDD1DULL) >> 11) / 4503599627370496.0 - 1.0;
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static void compare(const double *got, const double *want, size_t n, double atol, double rtol, const char *what) {
    size_t bad = 0;
    double worst = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double err = fabs(got[i] - want[i]);
        if (err > atol + rtol * fabs(want[i])) ++bad;
        if (err > worst) worst = err;
    }
    CHECK(bad == 0, "%s: %zu of %zu elements outside atol=%g rtol=%g (max abs err %g)", what, bad, n, atol, rtol, worst);
}

static int abi_checks(void) {
    /* invalid calls are rejected on the host before any device is touched */
    void *fake = (void *)(uintptr_t)0x7f0000000000ull;
    CHECK(la_attn_fwd(NULL, fake, fake, fake, 1, 1, 16, 16, 64, 0, 0.125f, NULL, LA_BF16, NULL, 0, NULL) ==
              LA_ERR_INVALID, "NULL q accepted");
    CHECK(la_attn_fwd(fake, fake, fake, fake, 1, 1, 16, 16, 96, 0, 0.125f, NULL, LA_BF16, NULL, 0, NULL) ==
              LA_ERR_UNSUPPORTED, "D = 96 accepted");
    CHECK(la_attn_fwd(fake, fake, fake, fake, 1, 1, 16, 16, 64, 0, -1.0f, NULL, LA_BF16, NULL, 0, NULL) ==
              LA_ERR_INVALID, "negative scale accepted");
    CHECK(la_attn_fwd(fake, fake, fake, fake, 1, 1, 16, 16, 64, 0, 0.125f, NULL, LA_F32, NULL, 0, NULL) ==
              LA_ERR_WORKSPACE, "fp32 without workspace accepted");
    CHECK(la_workspace_size(LA_OP_ATTN_FWD, 1, 1, 16, 16, 96, LA_BF16) == (size_t)-1, "workspace size of D = 96");
    CHECK(strncmp(la_status_string(LA_ERR_TIMEOUT), "LA_ERR_TIMEOUT", 14) == 0, "status string");
    return failures;
}

/* bf16 causal B=2 H=3 S=200 D=64 with key padding, through la_attn_fwd */
static void bf16_causal(void) {
    const int B = 2, H = 3, S = 200, D = 64;
    const size_t n = (size_t)B * H * S * D;
    uint16_t *hq = malloc(n * 2), *hk = malloc(n * 2), *hv = malloc(n * 2), *ho = malloc(n * 2);
    double *want = malloc(n * 8), *got = malloc(n * 8);
    for (size_t i = 0; i < n; ++i) hq[i] = to_bf16((float)(2.0 * uniform()));
    for (size_t i = 0; i < n; ++i) hk[i] = to_bf16((float)(2.0 * uniform()));
    for (size_t i = 0; i < n; ++i) hv[i] = to_bf16((float)(2.0 * uniform()));
    const int32_t kv_len[2] = {200, 137};
    void *dq, *dk, *dv, *dout, *dkl;
    cudaMalloc(&dq, n * 2);
    cudaMalloc(&dk, n * 2);
    cudaMalloc(&dv, n * 2);
    cudaMalloc(&dout, n * 2);
    cudaMalloc(&dkl, sizeof kv_len);
    cudaMemcpy(dq, hq, n * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dk, hk, n * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dv, hv, n * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dkl, kv_len, sizeof kv_len, cudaMemcpyHostToDevice);
    const float scale = 0.125f;
    la_status st = la_attn_fwd(dq, dk, dv, dout, B, H, S, S, D, 1, scale, (const int32_t *)dkl, LA_BF16, NULL, 0, NULL);
    CHECK(st == LA_OK, "bf16 la_attn_fwd: %s", la_status_string(st));
    st = la_get_last_error(NULL);
    CHECK(st == LA_OK, "bf16 device status: %s", la_status_string(st));
    cudaMemcpy(ho, dout, n * 2, cudaMemcpyDeviceToHost);
    for (size_t i = 0; i < n; ++i) got[i] = from_bf16(ho[i]);
    oracle_attn(hq, hk, hv, ORC_BF16, want, B, H, S, S, D, 1, scale, kv_len);
    compare(got, want, n, 2e-2, 2e-2, "bf16 causal");
    cudaFree(dq), cudaFree(dk), cudaFree(dv), cudaFree(dout), cudaFree(dkl);
    free(hq), free(hk), free(hv), free(ho), free(want), free(got);
}

/* fp32 non-causal B=1 H=2 S_q=100 S_kv=300 D=128 with a caller workspace */
static void fp32_workspace(void) {
    const int B = 1, H = 2, S_q = 100, S_kv = 300, D = 128;
    const size_t nq = (size_t)B * H * S_q * D, nk = (size_t)B * H * S_kv * D;
    float *hq = malloc(nq * 4), *hk = malloc(nk * 4), *hv = malloc(nk * 4), *ho = malloc(nq * 4);
    double *want = malloc(nq * 8), *got = malloc(nq * 8);
    /* small-integer multiples of 1/8: exact in TF32, so the products see the inputs as stored */
    for (size_t i = 0; i < nq; ++i) hq[i] = (float)(floor(8.0 * uniform()) / 8.0);
    for (size_t i = 0; i < nk; ++i) hk[i] = (float)(floor(8.0 * uniform()) / 8.0);
    for (size_t i = 0; i < nk; ++i) hv[i] = (float)uniform();
    const size_t ws_bytes = la_workspace_size(LA_OP_ATTN_FWD, B, H, S_q, S_kv, D, LA_F32);
    CHECK(ws_bytes != (size_t)-1 && ws_bytes > 0, "fp32 workspace size");
    void *dq, *dk, *dv, *dout, *ws;
    cudaMalloc(&dq, nq * 4);
    cudaMalloc(&dk, nk * 4);
    cudaMalloc(&dv, nk * 4);
    cudaMalloc(&dout, nq * 4);
    cudaMalloc(&ws, ws_bytes);
    cudaMemcpy(dq, hq, nq * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dk, hk, nk * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dv, hv, nk * 4, cudaMemcpyHostToDevice);
    const float scale = 0.125f;
    la_status st = la_attn_fwd(dq, dk, dv, dout, B, H, S_q, S_kv, D, 0, scale, NULL, LA_F32, ws, ws_bytes, NULL);
    CHECK(st == LA_OK, "fp32 la_attn_fwd: %s", la_status_string(st));
    st = la_get_last_error(NULL);
    CHECK(st == LA_OK, "fp32 device status: %s", la_status_string(st));
    cudaMemcpy(ho, dout, nq * 4, cudaMemcpyDeviceToHost);
    for (size_t i = 0; i < nq; ++i) got[i] = ho[i];
    oracle_attn(hq, hk, hv, ORC_F32, want, B, H, S_q, S_kv, D, 0, scale, NULL);
    compare(got, want, nq, 1e-3, 1e-2, "fp32 with workspace");
    cudaFree(dq), cudaFree(dk), cudaFree(dv), cudaFree(dout), cudaFree(ws);
    free(hq), free(hk), free(hv), free(ho), free(want), free(got);
}

int oracle_layer_attn(const void *x, const void *W, const void *bias, int dt, double *o, int B, long long S,
                      int d_model, int H, int causal, const int32_t *kv_len);

static void *to_device(const void *h, size_t bytes) {
    void *d = NULL;
    cudaMalloc(&d, bytes);
    cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice);
    return d;
}

/* bf16 sublayer B=2 S=150 d_model=256 H=4 (causal) through la_layer_attn, then
 * the same on a weight prepared once (la_prepare_weight,
 * la_layer_attn_prepared): the oracle's sublayer, and bit for bit equal;
 * per-launch timing (la_profile_start / la_profile_stop) around the second */
static void bf16_sublayer(void) {
    const int B = 2, S = 150, dm = 256, H = 4;
    const size_t nx = (size_t)B * S * dm, nw = (size_t)dm * 3 * dm;
    uint16_t *hx = malloc(nx * 2), *hw = malloc(nw * 2), *hb = malloc(3 * dm * 2), *ho = malloc(nx * 2),
             *ho2 = malloc(nx * 2);
    double *want = malloc(nx * 8), *got = malloc(nx * 8);
    for (size_t i = 0; i < nx; ++i) hx[i] = to_bf16((float)(2.0 * uniform()));
    for (size_t i = 0; i < nw; ++i) hw[i] = to_bf16((float)(uniform() / 16.0));
    for (int i = 0; i < 3 * dm; ++i) hb[i] = to_bf16((float)(uniform() / 4.0));
    void *dx = to_device(hx, nx * 2), *dw = to_device(hw, nw * 2), *db = to_device(hb, 3 * dm * 2);
    void *dout, *dwp, *ws;
    cudaMalloc(&dout, nx * 2);
    cudaMalloc(&dwp, nw * 2);
    /* the block's size covers the sublayer and the prepared form */
    const size_t ws_bytes = la_workspace_size(LA_OP_LAYER_ATTN_LN, B, H, S, S, dm / H, LA_BF16);
    CHECK(ws_bytes != (size_t)-1, "sublayer workspace size");
    cudaMalloc(&ws, ws_bytes);
    la_status st = la_layer_attn(dx, dw, db, dout, B, S, dm, H, 1, NULL, LA_BF16, ws, ws_bytes, NULL);
    CHECK(st == LA_OK, "la_layer_attn: %s", la_status_string(st));
    cudaMemcpy(ho, dout, nx * 2, cudaMemcpyDeviceToHost);
    st = la_prepare_weight(dw, dwp, dm, 3 * dm, LA_BF16, NULL);
    CHECK(st == LA_OK, "la_prepare_weight: %s", la_status_string(st));
    CHECK(la_profile_start(64) == LA_OK, "la_profile_start");
    st = la_layer_attn_prepared(dx, NULL, NULL, 0.f, dwp, db, NULL, NULL, dout, B, S, dm, H, 1, NULL, LA_BF16, ws,
                                ws_bytes, NULL);
    CHECK(st == LA_OK, "la_layer_attn_prepared: %s", la_status_string(st));
    const char *names[64];
    float ms[64];
    const int nrec = la_profile_stop(names, ms, 64);
    CHECK(nrec >= 2, "profile: %d launches recorded", nrec);
    for (int i = 0; i < nrec; ++i) CHECK(names[i] != NULL && ms[i] > 0.f, "profile record %d", i);
    st = la_get_last_error(NULL);
    CHECK(st == LA_OK, "sublayer device status: %s", la_status_string(st));
    cudaMemcpy(ho2, dout, nx * 2, cudaMemcpyDeviceToHost);
    CHECK(memcmp(ho, ho2, nx * 2) == 0, "prepared sublayer differs from the sublayer");
    for (size_t i = 0; i < nx; ++i) got[i] = from_bf16(ho[i]);
    oracle_layer_attn(hx, hw, hb, ORC_BF16, want, B, S, dm, H, 1, NULL);
    compare(got, want, nx, 2e-2, 2e-2, "bf16 sublayer");
    cudaFree(dx), cudaFree(dw), cudaFree(db), cudaFree(dout), cudaFree(dwp), cudaFree(ws);
    free(hx), free(hw), free(hb), free(ho), free(ho2), free(want), free(got);
}

/* bf16 chunked mode: B=1 H=2 S=300 D=64 in windows of 128 (the last 44)
 * through la_attn_chunked on a caller-owned cache: the oracle's causal
 * attention over the whole sequence */
static void bf16_chunked(void) {
    const int B = 1, H = 2, S = 300, D = 64, C = 128;
    const size_t n = (size_t)B * H * S * D;
    uint16_t *hq = malloc(n * 2), *hk = malloc(n * 2), *hv = malloc(n * 2), *ho = malloc(n * 2);
    uint16_t *wq = malloc((size_t)B * H * C * D * 2), *wk = malloc((size_t)B * H * C * D * 2),
             *wv = malloc((size_t)B * H * C * D * 2), *wo = malloc((size_t)B * H * C * D * 2);
    double *want = malloc(n * 8), *got = malloc(n * 8);
    for (size_t i = 0; i < n; ++i) hq[i] = to_bf16((float)(2.0 * uniform()));
    for (size_t i = 0; i < n; ++i) hk[i] = to_bf16((float)(2.0 * uniform()));
    for (size_t i = 0; i < n; ++i) hv[i] = to_bf16((float)(2.0 * uniform()));
    la_kv_cache cache;
    cudaMalloc(&cache.k, n * 2);
    cudaMalloc(&cache.v, n * 2);
    cache.B = B, cache.H = H, cache.D = D, cache.S_max = S, cache.len = 0, cache.dtype = LA_BF16;
    const size_t ws_bytes = la_workspace_size(LA_OP_ATTN_CHUNKED, B, H, C, S, D, LA_BF16);
    void *ws = NULL, *dq, *dk, *dv, *dout;
    if (ws_bytes > 0) cudaMalloc(&ws, ws_bytes);
    const size_t wbytes = (size_t)B * H * C * D * 2;
    cudaMalloc(&dq, wbytes), cudaMalloc(&dk, wbytes), cudaMalloc(&dv, wbytes), cudaMalloc(&dout, wbytes);
    const float scale = 0.125f;
    for (int s0 = 0; s0 < S; s0 += C) {
        const int L = S - s0 < C ? S - s0 : C;
        for (int bh = 0; bh < B * H; ++bh)  /* the window's rows of each head, contiguous */
            for (int r = 0; r < L; ++r) {
                const size_t src = ((size_t)bh * S + s0 + r) * D, dst = ((size_t)bh * L + r) * D;
                memcpy(wq + dst, hq + src, D * 2), memcpy(wk + dst, hk + src, D * 2), memcpy(wv + dst, hv + src, D * 2);
            }
        const size_t lb = (size_t)B * H * L * D * 2;
        cudaMemcpy(dq, wq, lb, cudaMemcpyHostToDevice);
        cudaMemcpy(dk, wk, lb, cudaMemcpyHostToDevice);
        cudaMemcpy(dv, wv, lb, cudaMemcpyHostToDevice);
        la_status st = la_attn_chunked(dq, dk, dv, &cache, dout, L, 1, scale, ws, ws_bytes, NULL);
        CHECK(st == LA_OK, "la_attn_chunked at %d: %s", s0, la_status_string(st));
        CHECK(cache.len == s0 + L, "cache length %d after the window at %d", cache.len, s0);
        cudaMemcpy(wo, dout, lb, cudaMemcpyDeviceToHost);
        for (int bh = 0; bh < B * H; ++bh)
            for (int r = 0; r < L; ++r) memcpy(ho + ((size_t)bh * S + s0 + r) * D, wo + ((size_t)bh * L + r) * D, D * 2);
    }
    la_status st = la_get_last_error(NULL);
    CHECK(st == LA_OK, "chunked device status: %s", la_status_string(st));
    for (size_t i = 0; i < n; ++i) got[i] = from_bf16(ho[i]);
    oracle_attn(hq, hk, hv, ORC_BF16, want, B, H, S, S, D, 1, scale, NULL);
    compare(got, want, n, 2e-2, 2e-2, "bf16 chunked");
    cudaFree(cache.k), cudaFree(cache.v), cudaFree(dq), cudaFree(dk), cudaFree(dv), cudaFree(dout);
    if (ws) cudaFree(ws);
    free(hq), free(hk), free(hv), free(ho), free(wq), free(wk), free(wv), free(wo), free(want), free(got);
}

int main(int argc, char **argv) {
    rng_state = 0x9E3779B97F4A7C15ull;
    abi_checks();
    if (argc > 1 && strcmp(argv[1], "--abi") == 0) {
        printf(failures ? "abi checks failed\n" : "abi checks ok\n");
        return failures ? 1 : 0;
    }
    bf16_causal();
    fp32_workspace();
    bf16_sublayer();
    bf16_chunked();
    if (failures)
        printf("C caller: %d checks failed\n", failures);
    else
        printf("C caller ok\n");
    return failures ? 1 : 0;
}
