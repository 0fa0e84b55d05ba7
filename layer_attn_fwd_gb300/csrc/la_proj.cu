// la_proj.cu -- fused Q/K/V projection on sm_103a ("Roofline", sections What
// it does and How we built it: one x.Wqkv product instead of three).
//
//   y[M, 3d] = x[M, d] . Wqkv[d, 3d] + bqkv      (M = B*S rows)
//
// A persistent kernel, one CTA per SM, walks 128 x BNP tiles of y.  Each tile
// is accumulated in tensor memory by tcgen05.mma; the accumulator is double
// buffered, so the epilogue of one tile (bias, Q scale, split into heads)
// runs while the next tile's products are issued.  The epilogue scatters the
// tile straight into the head-major q, k, v [B, H, S, D] outputs, so the
// split into heads costs no extra pass.  The same kernel computes the
// sublayer's output projection y = o.Wo + bo: a row-major [M, d] output is the
// head-major layout with one batch entry and one head as wide as the row.
// Tiles are 128 rows by BNP columns, BNP the wide width or 128 (chosen per
// launch for the fewest waves).
//
//   warp 4        TMA: x tile (K-major) and weight tile through an NSP-stage
//                 ring.  bf16/fp16 read Wqkv itself (rows = K, columns = N:
//                 an MN-major operand).  TF32 products take K-major operands
//                 only, so fp32 reads Wqkv^T [3d, d], transposed beforehand.
//   warp 5        issues the MMAs (the warp runs the loop, one elected lane
//                 issues); commits free the stages.
//   warps 0..3    epilogue, thread r owns row r of the tile.
//   warps 6..9    (LN form only) LayerNorm in front of the projection
//                 ("Shape-Aware Attention", section What's next: fusing
//                 LayerNorm): thread r normalises row r of each x stage in
//                 shared memory, (x - mean_r) * rstd_r * gamma + beta with the
//                 row statistics of a stats pre-pass, rounds it to the
//                 operand type and hands the stage to the MMA warp, so the
//                 normalised activations never go through global memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

template <typename T>
struct PElem;
template <>
struct PElem<__nv_bfloat16> {
  static constexpr uint32_t ab = AB_BF16;
  static constexpr bool tf32 = false;
  static __device__ __forceinline__ float load(const void* p, int i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct PElem<__half> {
  static constexpr uint32_t ab = AB_F16;
  static constexpr bool tf32 = false;
  static __device__ __forceinline__ float load(const void* p, int i) {
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct PElem<float> {
  static constexpr uint32_t ab = AB_TF32;
  static constexpr bool tf32 = true;
  static __device__ __forceinline__ float load(const void* p, int i) {
    return reinterpret_cast<const float*>(p)[i];
  }
};

template <typename T, int BNP_, int NSP_, bool LN_ = false>
struct PCfg {
  static constexpr int BNP = BNP_, NSP = NSP_;
  static constexpr bool LN = LN_;
  static constexpr int E = sizeof(T);
  static constexpr int CW = 128 / E;           // elements per 128-byte row = K per stage
  static constexpr int A_STAGE = kTileM * 128; // x tile: 128 rows x 128 bytes
  static constexpr bool KMAJ = (E == 4);       // fp32: weight tile from Wqkv^T (K-major)
  static constexpr int B_CHUNK = KMAJ ? BNP * 128 : CW * 128;  // MN-major: CW weight rows x 128 bytes
  static constexpr int B_STAGE = BNP * CW * E;
  static constexpr int STG_BYTES = 32 * 128;   // one epilogue warp's 32 rows x 128 bytes
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = NSP * A_STAGE;
  static constexpr int OFF_STG = OFF_B + NSP * B_STAGE;
  static constexpr int OFF_BIAS = OFF_STG + 4 * STG_BYTES;  // each epilogue warp's bias slice (fp32)
  static constexpr int OFF_BAR = OFF_BIAS + 4 * BNP * 4;
  // full[NSP], empty[NSP], acc_full[2], acc_empty[2], mma_done, (LN) xf_full[NSP]
  static constexpr int NBAR = 2 * NSP + 5 + (LN ? NSP : 0);
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = 2 * BNP <= 256 ? 256 : 512;  // two accumulators (power of two)
  static constexpr int ROWS_PER_KSTEP = 32 / E;  // K rows consumed by one MMA
  static constexpr int THREADS = LN ? 320 : 192;
  static constexpr int WARP_TMA = 4, WARP_MMA = 5, WARP_XF = 6;
  static_assert(BNP % CW == 0 && BNP >= 32 && BNP <= 256 && BNP % 16 == 0, "tile width");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Packs CW values of one row (128 bytes) into eight 16-byte units.
template <typename T>
__device__ __forceinline__ uint4 pack_unit(const float* v, int u) {
  if constexpr (PElem<T>::tf32) {
    return make_uint4(__float_as_uint(v[4 * u]), __float_as_uint(v[4 * u + 1]), __float_as_uint(v[4 * u + 2]),
                      __float_as_uint(v[4 * u + 3]));
  } else {
    uint4 w;
    w.x = PElem<T>::pack2(v[8 * u + 0], v[8 * u + 1]);
    w.y = PElem<T>::pack2(v[8 * u + 2], v[8 * u + 3]);
    w.z = PElem<T>::pack2(v[8 * u + 4], v[8 * u + 5]);
    w.w = PElem<T>::pack2(v[8 * u + 6], v[8 * u + 7]);
    return w;
  }
}

// 16 bytes of x (CW / 8 values) normalised: (x - mu) * rs * gamma + beta,
// the LayerNorm kernel's arithmetic, rounded to the operand type (fp32: to
// TF32 to nearest, ties away, by adding half a TF32 ulp to the bit pattern;
// the kind::tf32 product reads only the top 19 bits; the copy into shared
// memory left x unrounded).
template <typename T>
__device__ __forceinline__ uint4 ln_unit(uint4 w, uint4 gw, uint4 bw, float mu, float rs);
template <>
__device__ __forceinline__ uint4 ln_unit<float>(uint4 w, uint4 gw, uint4 bw, float mu, float rs) {
  const float4 g = make_float4(__uint_as_float(gw.x), __uint_as_float(gw.y), __uint_as_float(gw.z), __uint_as_float(gw.w));
  const float4 b = make_float4(__uint_as_float(bw.x), __uint_as_float(bw.y), __uint_as_float(bw.z), __uint_as_float(bw.w));
  uint4 o;
  o.x = __float_as_uint(fmaf((__uint_as_float(w.x) - mu) * rs, g.x, b.x)) + 0x1000u;
  o.y = __float_as_uint(fmaf((__uint_as_float(w.y) - mu) * rs, g.y, b.y)) + 0x1000u;
  o.z = __float_as_uint(fmaf((__uint_as_float(w.z) - mu) * rs, g.z, b.z)) + 0x1000u;
  o.w = __float_as_uint(fmaf((__uint_as_float(w.w) - mu) * rs, g.w, b.w)) + 0x1000u;
  return o;
}
template <typename T>
__device__ __forceinline__ uint4 ln_unit_half(uint4 w, uint4 gw, uint4 bw, float mu, float rs) {
  const uint32_t xs[4] = {w.x, w.y, w.z, w.w}, gs[4] = {gw.x, gw.y, gw.z, gw.w}, bs[4] = {bw.x, bw.y, bw.z, bw.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    T x2[2], g2[2], b2[2];
    memcpy(x2, &xs[i], 4);
    memcpy(g2, &gs[i], 4);
    memcpy(b2, &bs[i], 4);
    const float y0 = fmaf((static_cast<float>(x2[0]) - mu) * rs, static_cast<float>(g2[0]), static_cast<float>(b2[0]));
    const float y1 = fmaf((static_cast<float>(x2[1]) - mu) * rs, static_cast<float>(g2[1]), static_cast<float>(b2[1]));
    o[i] = PElem<T>::pack2(y0, y1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
template <>
__device__ __forceinline__ uint4 ln_unit<__nv_bfloat16>(uint4 w, uint4 gw, uint4 bw, float mu, float rs) {
  return ln_unit_half<__nv_bfloat16>(w, gw, bw, mu, rs);
}
template <>
__device__ __forceinline__ uint4 ln_unit<__half>(uint4 w, uint4 gw, uint4 bw, float mu, float rs) {
  return ln_unit_half<__half>(w, gw, bw, mu, rs);
}

template <typename T, int BNP, int NSP, bool LN>
__global__ void __launch_bounds__(PCfg<T, BNP, NSP, LN>::THREADS, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                    const ProjArgs a) {
  using C = PCfg<T, BNP, NSP, LN>;
  constexpr bool TF32 = PElem<T>::tf32;
  constexpr int CW = C::CW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NSP;
  uint64_t* acc_full = empty + NSP;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* xf_full = mma_done + 1;  // (LN) stage s normalised in place, ready for the MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tn = (a.N + BNP - 1) / BNP;
  const int n_tiles = n_tn * ((a.M + kTileM - 1) / kTileM);
  const int n_k = a.K / CW;  // K = d_model, a multiple of 64

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSP; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrive per epilogue warp
    }
    mbar_init(mma_done, 1);
    if constexpr (LN)
      for (int s = 0; s < NSP; ++s) mbar_init(&xf_full[s], 4);  // one arrive per transform warp
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{a.err, abort_flag};
  // The set-up above overlaps the previous grid; nothing before the wait
  // reads or writes global memory the previous grid may touch.  The tensor
  // maps are kernel parameters, so their descriptors are fetched meanwhile.
  if (threadIdx.x == 0) pdl_trigger();
  if (warp == C::WARP_TMA && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  pdl_wait();

  if (warp == C::WARP_TMA) {
    int last[NSP];
#pragma unroll
    for (int s = 0; s < NSP; ++s) last[s] = -1;
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int tm = t / n_tn, tn = t - tm * n_tn;
        for (int kt = 0; kt < n_k; ++kt, ++it) {
          const int s = it % NSP, r = it / NSP;
          if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, ab, SITE_PROJ_EMPTY)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], C::A_STAGE + C::B_STAGE);
          tma_load_2d(&tm_x, &full[s], smem + C::OFF_A + s * C::A_STAGE, kt * CW, tm * kTileM, pol_x);
          if constexpr (C::KMAJ) {
            tma_load_2d(&tm_w, &full[s], smem + C::OFF_B + s * C::B_STAGE, kt * CW, tn * BNP, pol_w);
          } else {
            for (int c = 0; c < BNP / CW; ++c)
              tma_load_2d(&tm_w, &full[s], smem + C::OFF_B + s * C::B_STAGE + c * C::B_CHUNK, tn * BNP + c * CW,
                          kt * CW, pol_w);
          }
          last[s] = r;
        }
      }
    }
    __syncwarp();
    __syncthreads();
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < NSP; ++s)
        if (last[s] >= 0) mbar_wait_teardown(&full[s], last[s] & 1);
    }
    __syncwarp();
  } else if (warp == C::WARP_MMA) {
    // The whole warp runs the loop and waits (warp-uniform MMA operands); one
    // elected lane issues the MMAs and their commits.
    {
      const uint32_t idesc = idesc_make(PElem<T>::ab, kTileM, BNP, false, !C::KMAJ);
      const uint32_t sA = smem_u32(smem + C::OFF_A);
      const uint32_t sB = smem_u32(smem + C::OFF_B);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++lt) {
        const int accb = lt & 1, use = lt >> 1;
        if (use > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&acc_empty[accb], (use - 1) & 1, ab, SITE_PROJ_ACC_FREE))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + accb * BNP;
        for (int kt = 0; kt < n_k; ++kt, ++it) {
          const int s = it % NSP, r = it / NSP;
          if (!__all_sync(0xffffffffu, mbar_wait(LN ? &xf_full[s] : &full[s], r & 1, ab, SITE_PROJ_FULL))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc_sw128(sA + s * C::A_STAGE + kk * 32, 16, 1024);
              const uint64_t bd =
                  C::KMAJ ? sdesc_sw128(sB + s * C::B_STAGE + kk * 32, 16, 1024)
                          : sdesc_sw128(sB + s * C::B_STAGE + kk * C::ROWS_PER_KSTEP * 128, C::B_CHUNK, 1024);
              mma_ss<TF32>(d, ad, bd, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&empty[s]);
          }
          __syncwarp();
        }
        if (ok) {
          if (elect_one()) mma_commit(&acc_full[accb]);
          __syncwarp();
        }
      }
    }
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
      if (elect_one()) {  // the lane that issued the MMAs
        mma_commit(mma_done);
        mbar_wait_teardown(mma_done, 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  } else if (LN && warp >= C::WARP_XF) {
    // LayerNorm of each x stage in place (LN form).  Thread r owns row r of
    // the stage; its 128 bytes are eight 16-byte units stored at unit
    // position u ^ (r % 8) (the 128-byte swizzle the copy wrote).
    const int xr = (warp - C::WARP_XF) * 32 + lane;
    const T* gamma = reinterpret_cast<const T*>(a.ln_gamma);
    const T* beta = reinterpret_cast<const T*>(a.ln_beta);
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const int m = (t / n_tn) * kTileM + xr;
      float mu = 0.f, rs = 0.f;  // rows past the end (zero-filled) become beta; they are never stored
      if (m < a.M) {
        const float2 st = a.ln_stats[m];
        mu = st.x;
        rs = st.y;
      }
      for (int kt = 0; kt < n_k; ++kt, ++it) {
        const int s = it % NSP, r = it / NSP;
        uint4 gv[8], bv[8];  // this stage's gamma and beta, requested before the wait for the stage
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          gv[u] = __ldg(reinterpret_cast<const uint4*>(gamma + kt * CW + u * (CW / 8)));
          bv[u] = __ldg(reinterpret_cast<const uint4*>(beta + kt * CW + u * (CW / 8)));
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], r & 1, ab, SITE_PROJ_FULL))) { ok = false; break; }
        const uint32_t line = smem_u32(smem + C::OFF_A + s * C::A_STAGE) + xr * 128;
        // all eight loads first, then the arithmetic, then the stores (the
        // shared-memory accesses are ordered asm statements: interleaving
        // them unit by unit would serialise their latencies)
        uint4 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) xv[u] = lds128(line + ((u ^ (xr & 7)) << 4));
#pragma unroll
        for (int u = 0; u < 8; ++u) xv[u] = ln_unit<T>(xv[u], gv[u], bv[u], mu, rs);
#pragma unroll
        for (int u = 0; u < 8; ++u) sts128(line + ((u ^ (xr & 7)) << 4), xv[u]);
        fence_proxy_async_smem();  // the tensor cores read the stage through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&xf_full[s]);
      }
    }
    __syncwarp();
    __syncthreads();
  } else {
    // epilogue: thread owns row warp*32 + lane of the tile.  Per 128-byte
    // column chunk (CW columns, inside one head of one of q/k/v): TMEM ->
    // registers, + bias, x q_scale; then the warp's 32 rows go through a
    // swizzled 4 KB shared buffer so that every global store instruction
    // writes whole 128-byte row segments (four rows per instruction).
    // V^T for the fp32 sublayer is stored directly: there lanes hold
    // consecutive positions of one V^T row, which is already coalesced.
    float* sbias = reinterpret_cast<float*>(smem + C::OFF_BIAS) + warp * BNP;
    const uint32_t sbias_a = smem_u32(sbias);
    const uint32_t stg_a = smem_u32(smem + C::OFF_STG + warp * C::STG_BYTES);
    const int d_model = a.K;
    const int sub = lane >> 3, unit = lane & 7;  // row-in-4 and 16-byte unit this lane stores
    int lt = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
      const int tm = t / n_tn, tn = t - tm * n_tn;
      const int accb = lt & 1, use = lt >> 1;
      // the tile's bias slice, one private copy per warp (no barrier beyond the warp)
      __syncwarp();
      for (int i = lane; i < BNP; i += 32) {
        const int n = tn * BNP + i;
        sbias[i] = (a.bias != nullptr && n < a.N) ? PElem<T>::load(a.bias, n) : 0.f;
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[accb], use & 1, ab, SITE_PROJ_ACC))) break;
      tc_fence_after();
      const int m = tm * kTileM + warp * 32 + lane;
      const int bidx = m / a.S;
      const int srow = m - bidx * a.S;
      // element offset of this thread's row inside one [B, H, S, D] output, head 0;
      // ro[i]: the same for the row this lane stores in step i of each chunk
      const long long row_off = (static_cast<long long>(bidx) * a.H * a.S + srow) * a.D;
      long long ro[8];
      bool rok[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ro[i] = __shfl_sync(0xffffffffu, row_off, 4 * i + sub);
        rok[i] = tm * kTileM + warp * 32 + 4 * i + sub < a.M;
      }
      const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16) + accb * BNP;
#pragma unroll 1
      for (int c0 = 0; c0 < BNP; c0 += CW) {
        const int n0 = tn * BNP + c0;
        if (n0 >= a.N) break;  // warp-uniform
        float v[CW];
#pragma unroll
        for (int i = 0; i < CW / 4; ++i) {  // bias (same for every row): broadcast loads, issued first
          const float4 bb = lds128f(sbias_a + (c0 + 4 * i) * 4);
          v[4 * i] = bb.x;
          v[4 * i + 1] = bb.y;
          v[4 * i + 2] = bb.z;
          v[4 * i + 3] = bb.w;
        }
        const int which = n0 / d_model;
        const int hd = n0 - which * d_model;
        const int hh = hd / a.D;
        const int dd = hd - hh * a.D;
        const float mul = which == 0 ? a.q_scale : 1.f;
#pragma unroll
        for (int h = 0; h < CW / 32; ++h) {
          uint32_t acc[32];
          tmem_ld_x32(trow + c0 + 32 * h, acc);
#pragma unroll
          for (int c = 0; c < 32; ++c) v[32 * h + c] = (__uint_as_float(acc[c]) + v[32 * h + c]) * mul;
        }
        if (which == 2 && a.v_transposed) {
          // V^T [B, H, D, S_pad]: lanes hold consecutive rows, so each store is coalesced
          if (m < a.M) {
            T* out =
                reinterpret_cast<T*>(a.v) + ((static_cast<long long>(bidx) * a.H + hh) * a.D + dd) * a.S_pad + srow;
#pragma unroll
            for (int c = 0; c < CW; ++c)
              if (LA_IN_BOUNDS(out - reinterpret_cast<T*>(a.v) + c * a.S_pad, 1, a.v_elems, a.err))
                out[c * a.S_pad] = static_cast<T>(v[c]);
          }
        } else {
          // row `lane` of the buffer, 16-byte unit u at u ^ lane%8 (conflict-free both ways)
          __syncwarp();  // the previous chunk's reads of the buffer are done
#pragma unroll
          for (int u = 0; u < 8; ++u) sts128(stg_a + lane * 128 + ((u ^ (lane & 7)) << 4), pack_unit<T>(v, u));
          __syncwarp();
          T* out = reinterpret_cast<T*>(which == 0 ? a.q : (which == 1 ? a.k : a.v)) +
                   (static_cast<long long>(hh) * a.S * a.D + dd + unit * (16 / C::E));
          uint4 w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {  // row 4i + sub, this lane's 16-byte unit
            const int r = 4 * i + sub;
            w[i] = lds128(stg_a + r * 128 + ((unit ^ (r & 7)) << 4));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (rok[i] && LA_IN_BOUNDS(out - reinterpret_cast<T*>(which == 0 ? a.q : (which == 1 ? a.k : a.v)) + ro[i],
                                       16 / C::E, which == 2 ? a.v_elems : a.qk_elems, a.err))
              *reinterpret_cast<uint4*>(out + ro[i]) = w[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[accb]);
    }
    __syncwarp();
    __syncthreads();
  }
}

template <typename T, int BNP, int NSP, bool LN>
cudaError_t launch_p(const CUtensorMap& tx, const CUtensorMap& tw, const ProjArgs& a, cudaStream_t st) {
  using C = PCfg<T, BNP, NSP, LN>;
  auto kern = qkv_proj_kernel<T, BNP, NSP, LN>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tiles =
      static_cast<long long>((a.N + BNP - 1) / BNP) * ((a.M + kTileM - 1) / kTileM);
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  return launch_pdl(LN ? "qkv_proj_ln_kernel" : "qkv_proj_kernel", kern, dim3(grid), dim3(C::THREADS),
                    C::SMEM_BYTES, st, tx, tw, a);
}

template <typename T, int BNP, int NSP>
cudaError_t launch_p2(const CUtensorMap& tx, const CUtensorMap& tw, const ProjArgs& a, cudaStream_t st) {
  return a.ln_stats != nullptr ? launch_p<T, BNP, NSP, true>(tx, tw, a, st) : launch_p<T, BNP, NSP, false>(tx, tw, a, st);
}

}  // namespace

// Tile width: the wide tile (fp32 192, half 256 columns) unless the
// 128-column tile finishes sooner.  A tile's time grows with the bytes its
// k-steps move through shared memory (the 128-row x tile plus the block_n-row
// weight tile), so a launch costs about waves x (128 + block_n); ties keep the
// wide tile.  Every tile shape gives the same result.
bool proj_shape(la_dtype dt, long long M, long long N, int sms, ProjShape* s) {
  if (dt != LA_F32 && dt != LA_BF16 && dt != LA_F16) return false;
  const int e = dt == LA_F32 ? 4 : 2;
  const int wide = dt == LA_F32 ? 192 : 256;
  const long long m_tiles = (M + kTileM - 1) / kTileM;
  auto cost = [&](int bn) {
    const long long tiles = m_tiles * ((N + bn - 1) / bn);
    const long long waves = (tiles + sms - 1) / (sms > 0 ? sms : 1);
    return waves * (kTileM + bn);
  };
  s->block_n = cost(128) < cost(wide) ? 128 : wide;
  s->box_cols = 128 / e;
  s->box_k_rows = 128 / e;
  s->w_transposed = (dt == LA_F32);
  return true;
}

cudaError_t launch_proj(la_dtype dt, int block_n, const CUtensorMap& tx, const CUtensorMap& tw, const ProjArgs& a,
                        cudaStream_t st) {
  const bool narrow = block_n == 128;
  if (!narrow && block_n != (dt == LA_F32 ? 192 : 256)) return cudaErrorInvalidValue;
  switch (dt) {
    case LA_BF16:
      return narrow ? launch_p2<__nv_bfloat16, 128, 6>(tx, tw, a, st) : launch_p2<__nv_bfloat16, 256, 4>(tx, tw, a, st);
    case LA_F16: return narrow ? launch_p2<__half, 128, 6>(tx, tw, a, st) : launch_p2<__half, 256, 4>(tx, tw, a, st);
    case LA_F32: return narrow ? launch_p2<float, 128, 6>(tx, tw, a, st) : launch_p2<float, 192, 5>(tx, tw, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
