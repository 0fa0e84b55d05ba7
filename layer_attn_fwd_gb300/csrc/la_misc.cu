// la_misc.cu -- the memory-bound helpers of the path:
//   - split-KV merge: partial outputs O_s (each normalised by its own sum)
//     and their log2-sum-exp values lse_s combine as
//       o = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
//     the same rescaling algebra the online softmax applies tile by tile;
//   - key/value cache append for the chunked long-context mode ("Roofline",
//     section How we built it: windows against a growing key/value cache);
//   - a 32-bit batched transpose: the TF32 tensor cores take K-major operands
//     only, so fp32 V (and the fp32 projection weights) are presented
//     transposed;
//   - LayerNorm before the projection (the pre-norm block; "Shape-Aware
//     Attention", section What's next: fusing LayerNorm), statistics in fp32.
// All are plain coalesced streams with grids sized to the SM count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

__device__ __forceinline__ void store4(float* d, float a, float b, float c, float e) {
  *reinterpret_cast<float4*>(d) = make_float4(a, b, c, e);
}
__device__ __forceinline__ void store4(__nv_bfloat16* d, float a, float b, float c, float e) {
  __nv_bfloat162 x = __floats2bfloat162_rn(a, b), y = __floats2bfloat162_rn(c, e);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&x);
  w.y = *reinterpret_cast<uint32_t*>(&y);
  *reinterpret_cast<uint2*>(d) = w;
}
__device__ __forceinline__ void store4(__half* d, float a, float b, float c, float e) {
  __half2 x = __floats2half2_rn(a, b), y = __floats2half2_rn(c, e);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&x);
  w.y = *reinterpret_cast<uint32_t*>(&y);
  *reinterpret_cast<uint2*>(d) = w;
}

// One thread per (row, 4 consecutive columns).
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  const int vec = a.D / 4;
  const long long rows = static_cast<long long>(a.B) * a.H * a.S_q;
  const long long total = rows * vec;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = g / vec;
    const int c = static_cast<int>(g - row * vec) * 4;
    float M = -INFINITY;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, a.part_lse[s * rows + row]);
    float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f, wsum = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < a.splits; ++s) {
        const float w = ex2_approx(a.part_lse[s * rows + row] - M);
        const float4 o = *reinterpret_cast<const float4*>(a.part_o + (s * rows + row) * a.D + c);
        wsum += w;
        x0 = fmaf(w, o.x, x0);
        x1 = fmaf(w, o.y, x1);
        x2 = fmaf(w, o.z, x2);
        x3 = fmaf(w, o.w, x3);
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const long long bh = row / a.S_q;
    const long long i = row - bh * a.S_q;
    const long long b = bh / a.H, h = bh - b * a.H;
    T* dst = reinterpret_cast<T*>(a.o) + b * a.o_sb + h * a.o_sh + i * a.o_ss + c;
    if (LA_IN_BOUNDS(dst - reinterpret_cast<T*>(a.o), 4, a.o_elems, a.err)) store4(dst, x0 * inv, x1 * inv, x2 * inv, x3 * inv);
  }
}

// blockIdx.z selects k (0) or v (1) (a keys-only launch has one), blockIdx.y
// the (b, h) pair.  A pair's new rows are one contiguous run of per_head
// 16-byte vectors in the source and in the cache (rows at.. of its [S_max, D]
// block), so the copy needs no index arithmetic beyond the two bases; each
// thread keeps four 16-byte loads in flight.
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, uint8_t* k_dst,
                     uint8_t* v_dst, int per_head, long long dst_head_bytes, long long at_bytes) {
  const uint4* src = (blockIdx.z == 0 ? k_src : v_src) + static_cast<long long>(blockIdx.y) * per_head;
  uint4* dst = reinterpret_cast<uint4*>((blockIdx.z == 0 ? k_dst : v_dst) + blockIdx.y * dst_head_bytes + at_bytes);
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < per_head; i += 4 * step) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * step < per_head) w[u] = src[i + u * step];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * step < per_head) dst[i + u * step] = w[u];
  }
}

// dst[b][c][r] = src[b][r][c] for 4-byte elements; source rows are C long
// and batches src_batch apart; destination rows are ld_dst long (>= R) and
// batches dst_batch apart.  64x64 tiles through shared memory: each thread
// keeps four 16-byte loads in flight, and both sides are coalesced.  vec:
// every row start on both sides is 16-byte aligned (C, ld_dst and the batch
// strides multiples of 4, bases 16-byte aligned), so 4-wide accesses are
// used wherever a group of four lies inside the matrix.
__global__ void __launch_bounds__(256)
    transpose32_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst, int R, int C, long long ld_dst,
                       long long src_batch, long long dst_batch, int vec) {
  __shared__ uint32_t tile[64][65];
  pdl_trigger();  // the consumer launched next may be scheduled now; it waits for this grid to finish
  const int r0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  const long long b = blockIdx.z;
  const uint32_t* s = src + b * src_batch;
  uint32_t* d = dst + b * dst_batch;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16
  uint32_t v[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty + 16 * i, c = c0 + 4 * tx;
    const uint32_t* p = s + static_cast<long long>(r) * C + c;
    if (r < R && vec && c + 3 < C) {
      const uint4 w = *reinterpret_cast<const uint4*>(p);
      v[i][0] = w.x, v[i][1] = w.y, v[i][2] = w.z, v[i][3] = w.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[i][k] = (r < R && c + k < C) ? p[k] : 0u;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) tile[ty + 16 * i][4 * tx + k] = v[i][k];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c0 + ty + 16 * i, r = r0 + 4 * tx;  // destination row c, columns r .. r+3
    if (c >= C) continue;
    uint32_t* p = d + static_cast<long long>(c) * ld_dst + r;
    const uint32_t w0 = tile[4 * tx][ty + 16 * i], w1 = tile[4 * tx + 1][ty + 16 * i];
    const uint32_t w2 = tile[4 * tx + 2][ty + 16 * i], w3 = tile[4 * tx + 3][ty + 16 * i];
    if (vec && r + 3 < R) {
      *reinterpret_cast<uint4*>(p) = make_uint4(w0, w1, w2, w3);
    } else {
      if (r < R) p[0] = w0;
      if (r + 1 < R) p[1] = w1;
      if (r + 2 < R) p[2] = w2;
      if (r + 3 < R) p[3] = w3;
    }
  }
  // Under programmatic serialization this grid may run beside the one before
  // it; waiting for that grid before exiting keeps the stream's order for the
  // grids after this one.  A no-op for an ordinary launch.
  pdl_wait();
}

// 16 bytes of T <-> fp32 values.
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void unpack(const uint4& w, float* v) {
    v[0] = __uint_as_float(w.x), v[1] = __uint_as_float(w.y), v[2] = __uint_as_float(w.z), v[3] = __uint_as_float(w.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  // a bf16 value is the upper half of the fp32 with the same bits
  static __device__ __forceinline__ void unpack(const uint4& w, float* v) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) v[2 * i] = __uint_as_float(u[i] << 16), v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      memcpy(&u[i], &h, 4);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
};
template <>
struct Vec16<__half> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4& w, float* v) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h;
      memcpy(&h, &u[i], 4);
      const float2 f = __half22float2(h);
      v[2 * i] = f.x, v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      memcpy(&u[i], &h, 4);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
};

// Sum over aligned groups of G lanes (G a power of two <= 32).
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// LayerNorm of rows of d elements (d a multiple of 64), one group of LPR
// lanes per row (a warp takes 32 / LPR rows at once): the mean, then the
// mean squared deviation from it, both in fp32; then
// y = (x - mean) / sqrt(var + eps) * gamma + beta, rounded to T.  16-byte
// accesses; rows 16-byte aligned.  A row of up to LPR * FPL values is loaded
// once (all of a lane's loads issued together) and kept unpacked in
// registers; gamma and beta, the same for every row, are read when the
// output is formed.  Longer rows take three passes (the later two hit L1).
// Every lane of a warp runs the same number of loop trips (rows past the end
// skip their loads and stores), so the group sums see whole warps.
// STATS: only the row statistics (mean, 1 / sqrt(var + eps)) are written, to
// stats[row], for a projection that normalises its input tiles as it loads
// them; the arithmetic of the statistics is the same.
template <typename T, int FPL, int LPR, bool STATS>
__global__ void __launch_bounds__(256, 3)
    layernorm_kernel(const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
                     T* __restrict__ y, float2* __restrict__ stats, long long M, int d, float eps) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  constexpr int NVL = FPL / E;  // 16-byte vectors a lane holds
  constexpr int RPW = 32 / LPR;  // rows per warp
  pdl_trigger();  // the next grid may be scheduled now; it waits for this one to finish
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & (LPR - 1);        // lane within the row's group
  const int grp = (threadIdx.x & 31) / LPR;        // the warp's row this lane works on
  const int nv = d / E;
  const float inv_d = 1.f / static_cast<float>(d);
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  const uint4* b4 = reinterpret_cast<const uint4*>(beta);
  const long long stride = static_cast<long long>(gridDim.x) * 8 * RPW;
  for (long long r0 = (blockIdx.x * 8LL + warp) * RPW; r0 < M; r0 += stride) {
    const long long r = r0 + grp;
    const bool live = r < M;
    const long long rr = live ? r : r0;  // a dead group reads the warp's first row and stores nothing
    const uint4* xr = reinterpret_cast<const uint4*>(x + rr * d);
    uint4* yr = reinterpret_cast<uint4*>(y + rr * d);
    if (nv <= LPR * NVL) {
      uint4 w[NVL];
#pragma unroll
      for (int j = 0; j < NVL; ++j)
        if (lane + LPR * j < nv) w[j] = xr[lane + LPR * j];
      float v[NVL][E];
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < NVL; ++j) {
        if (lane + LPR * j < nv) {
          V::unpack(w[j], v[j]);
#pragma unroll
          for (int e = 0; e < E; ++e) s += v[j][e];
        }
      }
      const float mu = group_sum<LPR>(s) * inv_d;
      float q = 0.f;
#pragma unroll
      for (int j = 0; j < NVL; ++j)
        if (lane + LPR * j < nv)
#pragma unroll
          for (int e = 0; e < E; ++e) {
            v[j][e] -= mu;
            q = fmaf(v[j][e], v[j][e], q);
          }
      const float rstd = 1.f / sqrtf(group_sum<LPR>(q) * inv_d + eps);
      if constexpr (STATS) {
        if (live && lane == 0) stats[r] = make_float2(mu, rstd);
        continue;
      }
#pragma unroll
      for (int j = 0; j < NVL; ++j) {
        const int i = lane + LPR * j;
        if (live && i < nv) {
          float g[E], b[E];
          V::unpack(g4[i], g);
          V::unpack(b4[i], b);
#pragma unroll
          for (int e = 0; e < E; ++e) v[j][e] = fmaf(v[j][e] * rstd, g[e], b[e]);
          yr[i] = V::pack(v[j]);
        }
      }
    } else {
      float v[E];
      float s = 0.f;
      for (int i = lane; i < nv; i += LPR) {
        V::unpack(xr[i], v);
#pragma unroll
        for (int e = 0; e < E; ++e) s += v[e];
      }
      const float mu = group_sum<LPR>(s) * inv_d;
      float q = 0.f;
      for (int i = lane; i < nv; i += LPR) {
        V::unpack(xr[i], v);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float t = v[e] - mu;
          q = fmaf(t, t, q);
        }
      }
      const float rstd = 1.f / sqrtf(group_sum<LPR>(q) * inv_d + eps);
      if constexpr (STATS) {
        if (live && lane == 0) stats[r] = make_float2(mu, rstd);
        continue;
      }
      for (int i = lane; i < nv && live; i += LPR) {
        float g[E], b[E];
        V::unpack(xr[i], v);
        V::unpack(g4[i], g);
        V::unpack(b4[i], b);
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = fmaf((v[e] - mu) * rstd, g[e], b[e]);
        yr[i] = V::pack(v);
      }
    }
  }
  // Under programmatic serialization this grid may run beside the one before
  // it; waiting for that grid before exiting keeps the stream's order for the
  // grids after this one.  A no-op for an ordinary launch.
  pdl_wait();
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

}  // namespace

cudaError_t launch_combine(la_dtype dt, const CombineArgs& a, cudaStream_t st) {
  const long long total = static_cast<long long>(a.B) * a.H * a.S_q * (a.D / 4);
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int cap = sm_count() * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  switch (dt) {
    case LA_F32: return launch("combine_kernel", combine_kernel<float>, dim3(grid), dim3(256), 0, st, false, a);
    case LA_BF16: return launch("combine_kernel", combine_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st, false, a);
    case LA_F16: return launch("combine_kernel", combine_kernel<__half>, dim3(grid), dim3(256), 0, st, false, a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_transpose32(const void* src, long long src_batch, void* dst, long long ld_dst, long long batches,
                               int R, int C, cudaStream_t st, bool pdl) {
  if (batches == 0 || R == 0 || C == 0) return cudaSuccess;
  if (batches > 65535 || (C + 63) / 64 > 65535) return cudaErrorInvalidValue;
  const long long dst_batch = static_cast<long long>(C) * ld_dst;
  const int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (reinterpret_cast<uintptr_t>(dst) % 16 == 0) &&
                  C % 4 == 0 && ld_dst % 4 == 0 && src_batch % 4 == 0 && dst_batch % 4 == 0;
  dim3 grid((R + 63) / 64, (C + 63) / 64, static_cast<unsigned>(batches));
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
  uint32_t* d = reinterpret_cast<uint32_t*>(dst);
  return launch("transpose32_kernel", transpose32_kernel, grid, dim3(256), 0, st, pdl, s, d, R, C, ld_dst, src_batch,
                dst_batch, vec);
}

// Row values each lane keeps in registers (within 80 registers, so three
// blocks share an SM): rows of up to 32 x 16 fp32 or 32 x 32 half-precision
// values take the single-pass form.
constexpr int kLnFloatsPerLaneF32 = 16, kLnFloatsPerLaneHalf = 32;

template <typename T, int FPL>
cudaError_t launch_ln(const void* x, const void* gamma, const void* beta, void* y, float2* stats, long long M, int d,
                      float eps, cudaStream_t st, bool pdl) {
  // Half a warp per row when the row fits in registers that way: twice the
  // rows per warp, so a launch of a few thousand rows runs in one wave.
  const bool half_warp = d / Vec16<T>::N <= 16 * (FPL / Vec16<T>::N);
  const int rows_per_block = half_warp ? 16 : 8;
  const long long want = (M + rows_per_block - 1) / rows_per_block;
  const int cap = sm_count() * 8;
  const dim3 grid(static_cast<unsigned>(want < cap ? want : cap));
  const T* xx = static_cast<const T*>(x);
  const T* gg = static_cast<const T*>(gamma);
  const T* bb = static_cast<const T*>(beta);
  T* yy = static_cast<T*>(y);
  if (stats != nullptr) {
    auto k = half_warp ? layernorm_kernel<T, FPL, 16, true> : layernorm_kernel<T, FPL, 32, true>;
    return launch("layernorm_stats_kernel", k, grid, dim3(256), 0, st, pdl, xx, gg, bb, yy, stats, M, d, eps);
  }
  auto k = half_warp ? layernorm_kernel<T, FPL, 16, false> : layernorm_kernel<T, FPL, 32, false>;
  return launch("layernorm_kernel", k, grid, dim3(256), 0, st, pdl, xx, gg, bb, yy, stats, M, d, eps);
}

cudaError_t launch_layernorm(la_dtype dt, const void* x, const void* gamma, const void* beta, void* y, long long M,
                             int d, float eps, cudaStream_t st, bool pdl, float2* stats) {
  if (M == 0) return cudaSuccess;
  switch (dt) {
    case LA_F32: return launch_ln<float, kLnFloatsPerLaneF32>(x, gamma, beta, y, stats, M, d, eps, st, pdl);
    case LA_BF16:
      return launch_ln<__nv_bfloat16, kLnFloatsPerLaneHalf>(x, gamma, beta, y, stats, M, d, eps, st, pdl);
    case LA_F16: return launch_ln<__half, kLnFloatsPerLaneHalf>(x, gamma, beta, y, stats, M, d, eps, st, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_append(const void* k_src, const void* v_src, void* k_dst, void* v_dst, int B, int H,
                             int rows, int D, int S_max, int at, int elem_bytes, cudaStream_t st) {
  const int vec_per_row = D * elem_bytes / 16;
  const long long per_head = static_cast<long long>(rows) * vec_per_row;
  const long long pairs = static_cast<long long>(B) * H;
  if (per_head == 0 || pairs == 0) return cudaSuccess;
  if (per_head > 0x7fffffffLL || pairs > 65535) return cudaErrorInvalidValue;
  // enough blocks per pair for about four waves of the whole grid, each
  // thread moving four vectors a pass
  const long long per_pair_want = (per_head + 1023) / 1024;
  const long long cap = (static_cast<long long>(sm_count()) * 32 + pairs - 1) / pairs;
  const long long bx = per_pair_want < cap ? per_pair_want : (cap > 0 ? cap : 1);
  dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(pairs), v_src != nullptr ? 2 : 1);  // keys only without v
  const long long row_bytes = static_cast<long long>(D) * elem_bytes;
  return launch("kv_append_kernel", kv_append_kernel, grid, dim3(256), 0, st, false,
                reinterpret_cast<const uint4*>(k_src), reinterpret_cast<const uint4*>(v_src),
                reinterpret_cast<uint8_t*>(k_dst), reinterpret_cast<uint8_t*>(v_dst), static_cast<int>(per_head),
                static_cast<long long>(S_max) * row_bytes, static_cast<long long>(at) * row_bytes);
}

}  // namespace la
