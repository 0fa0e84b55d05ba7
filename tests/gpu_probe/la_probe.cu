// Test-only probe library: runs single device helpers of the attention
// kernels on arrays so the GPU tests can check them against references.
#include "la_device.cuh"

namespace {
__global__ void ex2_kernel(const float* x, float* poly, float* mufu, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    poly[i] = la::ex2_poly(x[i]);
    mufu[i] = la::ex2_approx(x[i]);
  }
}
}  // namespace

extern "C" int probe_ex2(const float* x, float* poly, float* mufu, int n) {
  if (n <= 0) return 0;
  ex2_kernel<<<(n + 255) / 256, 256>>>(x, poly, mufu, n);
  return static_cast<int>(cudaDeviceSynchronize());
}
