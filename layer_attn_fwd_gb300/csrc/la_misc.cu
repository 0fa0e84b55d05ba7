// la_misc.cu -- the memory-bound helpers of the path:
//   - split-KV merge: partial outputs O_s (each normalised by its own sum)
//     and their log2-sum-exp values lse_s combine as
//       o = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
//     the same rescaling algebra the online softmax applies tile by tile;
//   - key/value cache append for the chunked long-context mode ("Roofline",
//     section How we built it: windows against a growing key/value cache);
//   - a 32-bit batched transpose: the TF32 tensor cores take K-major operands
//     only, so fp32 V (and the fp32 projection weight) are presented
//     transposed.
// All are plain coalesced streams with grids sized to the SM count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "la_device.cuh"
#include "la_internal.h"

// The attention's work-ticket counters: per slot a ticket count and a count
// of CTAs done drawing, both zero between launches (the last CTA of a launch
// to finish drawing resets them).  Launches take the slots in turn, so that
// launches that may run at the same time (on other streams) rarely share one.
__device__ unsigned long long la_counters[2 * 64];

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
    store4(dst, x0 * inv, x1 * inv, x2 * inv, x3 * inv);
  }
}

// blockIdx.y selects k (0) or v (1).
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, uint8_t* k_dst,
                     uint8_t* v_dst, long long n_vec, int vec_per_row, int rows, long long dst_head_bytes,
                     long long at_bytes) {
  const uint4* src = blockIdx.y == 0 ? k_src : v_src;
  uint8_t* dst = blockIdx.y == 0 ? k_dst : v_dst;
  const long long row_bytes = static_cast<long long>(vec_per_row) * 16;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < n_vec;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = g / vec_per_row;  // row over all (b, h)
    const long long c = g - r * vec_per_row;
    const long long bh = r / rows;
    const long long rr = r - bh * rows;
    *reinterpret_cast<uint4*>(dst + bh * dst_head_bytes + at_bytes + rr * row_bytes + c * 16) = src[g];
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

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

}  // namespace

cudaError_t counter_slot(unsigned long long** ctr) {
  constexpr int kDev = 64, kSlots = 64;
  static std::mutex mu;
  static unsigned long long* addr[kDev] = {};
  static int next_slot[kDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, la_counters);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<unsigned long long*>(p);
  }
  const int slot = next_slot[dev];
  next_slot[dev] = (slot + 1) % kSlots;
  *ctr = addr[dev] + 2 * slot;
  return cudaSuccess;
}

cudaError_t launch_combine(la_dtype dt, const CombineArgs& a, cudaStream_t st) {
  const long long total = static_cast<long long>(a.B) * a.H * a.S_q * (a.D / 4);
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int cap = sm_count() * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  switch (dt) {
    case LA_F32: combine_kernel<float><<<grid, 256, 0, st>>>(a); break;
    case LA_BF16: combine_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(a); break;
    case LA_F16: combine_kernel<__half><<<grid, 256, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
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
  if (pdl) return launch_pdl(transpose32_kernel, grid, dim3(256), 0, st, s, d, R, C, ld_dst, src_batch, dst_batch, vec);
  transpose32_kernel<<<grid, 256, 0, st>>>(s, d, R, C, ld_dst, src_batch, dst_batch, vec);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k_src, const void* v_src, void* k_dst, void* v_dst, int B, int H,
                             int rows, int D, int S_max, int at, int elem_bytes, cudaStream_t st) {
  const int vec_per_row = D * elem_bytes / 16;
  const long long n_vec = static_cast<long long>(B) * H * rows * vec_per_row;
  if (n_vec == 0) return cudaSuccess;
  const long long want = (n_vec + 255) / 256;
  const int cap = sm_count() * 4;
  dim3 grid(static_cast<unsigned>(want < cap ? want : cap), 2);
  const long long row_bytes = static_cast<long long>(D) * elem_bytes;
  kv_append_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(k_src),
                                         reinterpret_cast<const uint4*>(v_src), reinterpret_cast<uint8_t*>(k_dst),
                                         reinterpret_cast<uint8_t*>(v_dst), n_vec, vec_per_row, rows,
                                         static_cast<long long>(S_max) * row_bytes,
                                         static_cast<long long>(at) * row_bytes);
  return cudaGetLastError();
}

}  // namespace la
