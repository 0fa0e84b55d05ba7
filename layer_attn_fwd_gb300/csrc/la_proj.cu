// la_proj.cu -- fused Q/K/V projection on sm_103a ("Roofline", sections What
// it does and How we built it: one x.Wqkv product instead of three).
//
//   y[M, 3d] = x[M, d] . Wqkv[d, 3d] + bqkv      (M = B*S rows)
//
// One CTA computes a 128 x BNP tile of y with tcgen05.mma (accumulator in
// tensor memory), then its epilogue adds the bias, scales the Q block and
// scatters the tile straight into the head-major q, k, v [B, H, S, D] outputs,
// so the split into heads costs no extra pass.
//
//   warp 4        TMA: x tile (K-major) and Wqkv tile (rows = K, columns = N,
//                 i.e. the B operand is MN-major) through an NSP-stage ring.
//                 TF32 products take K-major operands only, so for fp32 the
//                 weight is read from its transpose Wqkv^T [3d, d].
//   warp 5        one thread issues the MMAs; commits free the stages.
//   warps 0..3    epilogue, thread r owns row r of the tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

template <typename T, int BNP_, int NSP_>
struct PCfg {
  static constexpr int BNP = BNP_, NSP = NSP_;
  static constexpr int E = sizeof(T);
  static constexpr int CW = 128 / E;           // elements per 128-byte row = K per stage
  static constexpr int A_STAGE = kTileM * 128; // x tile: 128 rows x 128 bytes
  static constexpr bool WT = (E == 4);         // weight tile from Wqkv^T (K-major)
  static constexpr int B_CHUNK = WT ? BNP * 128 : CW * 128;  // MN-major: CW weight rows x 128 bytes
  static constexpr int B_STAGE = BNP * CW * E;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = NSP * A_STAGE;
  static constexpr int OFF_BAR = OFF_B + NSP * B_STAGE;
  static constexpr int NBAR = 2 * NSP + 2;     // full[NSP], empty[NSP], acc_full, mma_done
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_BIAS = OFF_MISC + 16;  // the tile's BNP bias values (fp32)
  static constexpr int SMEM_BYTES = OFF_BIAS + BNP * 4 + 1024;
  static constexpr int TMEM_COLS = BNP;
  static constexpr int ROWS_PER_KSTEP = 32 / E;  // K rows consumed by one MMA
  static constexpr int THREADS = 192;
  static constexpr int WARP_TMA = 4, WARP_MMA = 5;
  static_assert(BNP % CW == 0 && BNP >= 32 && BNP <= 256, "tile width");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <typename T>
__device__ __forceinline__ void store32(T* dst, const float (&v)[32]) {
  if constexpr (PElem<T>::tf32) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w;
      w.x = PElem<T>::pack2(v[8 * i + 0], v[8 * i + 1]);
      w.y = PElem<T>::pack2(v[8 * i + 2], v[8 * i + 3]);
      w.z = PElem<T>::pack2(v[8 * i + 4], v[8 * i + 5]);
      w.w = PElem<T>::pack2(v[8 * i + 6], v[8 * i + 7]);
      d4[i] = w;
    }
  }
}

template <typename T, int BNP, int NSP>
__global__ void __launch_bounds__(192, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                    const ProjArgs a) {
  using C = PCfg<T, BNP, NSP>;
  constexpr bool TF32 = PElem<T>::tf32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NSP;
  uint64_t* acc_full = empty + NSP;
  uint64_t* mma_done = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y;
  const int n_k = (a.K + C::CW - 1) / C::CW;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSP; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(mma_done, 1);
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

  if (warp == C::WARP_TMA) {
    int last[NSP];
#pragma unroll
    for (int s = 0; s < NSP; ++s) last[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      const uint64_t pol_x = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      for (int kt = 0; kt < n_k; ++kt) {
        const int s = kt % NSP, r = kt / NSP;
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, ab, SITE_PROJ_EMPTY)) break;
        mbar_arrive_expect_tx(&full[s], C::A_STAGE + C::B_STAGE);
        tma_load_2d(&tm_x, &full[s], smem + C::OFF_A + s * C::A_STAGE, kt * C::CW, tile_m * kTileM, pol_x);
        if constexpr (C::WT) {
          tma_load_2d(&tm_w, &full[s], smem + C::OFF_B + s * C::B_STAGE, kt * C::CW, tile_n * BNP, pol_w);
        } else {
          for (int c = 0; c < BNP / C::CW; ++c)
            tma_load_2d(&tm_w, &full[s], smem + C::OFF_B + s * C::B_STAGE + c * C::B_CHUNK,
                        tile_n * BNP + c * C::CW, kt * C::CW, pol_w);
        }
        last[s] = r;
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
    if (lane == 0) {
      const uint32_t idesc = idesc_make(PElem<T>::ab, kTileM, BNP, false, !C::WT);
      const uint32_t sA = smem_u32(smem + C::OFF_A);
      const uint32_t sB = smem_u32(smem + C::OFF_B);
      bool ok = true;
      for (int kt = 0; kt < n_k; ++kt) {
        const int s = kt % NSP, r = kt / NSP;
        if (!mbar_wait(&full[s], r & 1, ab, SITE_PROJ_FULL)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(sA + s * C::A_STAGE + kk * 32, 16, 1024);
          const uint64_t bd =
              C::WT ? sdesc_sw128(sB + s * C::B_STAGE + kk * 32, 16, 1024)
                    : sdesc_sw128(sB + s * C::B_STAGE + kk * C::ROWS_PER_KSTEP * 128, C::B_CHUNK, 1024);
          mma_ss<TF32>(tmem, ad, bd, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      if (ok) mma_commit(acc_full);
    }
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
      if (lane == 0) {
        mma_commit(mma_done);
        mbar_wait_teardown(mma_done, 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  } else {
    // epilogue: thread owns output row m; 32 columns at a time.  First stage
    // the tile's bias slice in shared memory while the main loop runs.
    float* sbias = reinterpret_cast<float*>(smem + C::OFF_BIAS);
    for (int i = threadIdx.x; i < BNP; i += 128) {
      const int n = tile_n * BNP + i;
      sbias[i] = (a.bias != nullptr && n < a.N) ? PElem<T>::load(a.bias, n) : 0.f;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps only
    const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, ab, SITE_PROJ_ACC));
    if (ok) {
      tc_fence_after();
      const int m = tile_m * kTileM + warp * 32 + lane;
      const int d_model = a.K;
      const int bidx = m / a.S;
      const int srow = m - bidx * a.S;
      const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BNP; c0 += 32) {
        const int n0 = tile_n * BNP + c0;
        if (n0 >= a.N) break;  // warp-uniform
        uint32_t acc[32];
        tmem_ld_x32(trow + c0, acc);
        const int which = n0 / d_model;
        const int hd = n0 - which * d_model;
        const int hh = hd / a.D;
        const int dd = hd - hh * a.D;
        const float mul = which == 0 ? a.q_scale : 1.f;
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          v[c] = (__uint_as_float(acc[c]) + sbias[c0 + c]) * mul;
        }
        if (m < a.M) {
          if (which == 2 && a.v_transposed) {
            // V^T [B, H, D, S_pad]: lanes hold consecutive rows, so each store is coalesced
            T* out = reinterpret_cast<T*>(a.v) + ((static_cast<long long>(bidx) * a.H + hh) * a.D + dd) * a.S_pad + srow;
#pragma unroll
            for (int c = 0; c < 32; ++c) out[c * a.S_pad] = static_cast<T>(v[c]);
          } else {
            T* out = reinterpret_cast<T*>(which == 0 ? a.q : (which == 1 ? a.k : a.v));
            store32<T>(out + ((static_cast<long long>(bidx) * a.H + hh) * a.S + srow) * a.D + dd, v);
          }
        }
      }
    }
    __syncthreads();
  }
}

template <typename T, int BNP, int NSP>
cudaError_t launch_p(const CUtensorMap& tx, const CUtensorMap& tw, const ProjArgs& a, cudaStream_t st) {
  using C = PCfg<T, BNP, NSP>;
  auto kern = qkv_proj_kernel<T, BNP, NSP>;
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
  dim3 grid((a.N + BNP - 1) / BNP, (a.M + kTileM - 1) / kTileM);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(tx, tw, a);
  return cudaGetLastError();
}

}  // namespace

bool proj_shape(la_dtype dt, ProjShape* s) {
  if (dt != LA_F32 && dt != LA_BF16 && dt != LA_F16) return false;
  const int e = dt == LA_F32 ? 4 : 2;
  s->block_n = 256;
  s->box_cols = 128 / e;
  s->box_k_rows = 128 / e;
  s->w_transposed = (dt == LA_F32);
  return true;
}

cudaError_t launch_proj(la_dtype dt, const CUtensorMap& tx, const CUtensorMap& tw, const ProjArgs& a,
                        cudaStream_t st) {
  switch (dt) {
    case LA_BF16: return launch_p<__nv_bfloat16, 256, 4>(tx, tw, a, st);
    case LA_F16: return launch_p<__half, 256, 4>(tx, tw, a, st);
    case LA_F32: return launch_p<float, 256, 4>(tx, tw, a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace la
