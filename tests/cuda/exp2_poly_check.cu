// Test-only kernel: evaluates the kernels' polynomial exp2 (exp2_poly2 from
// sm103_ptx.cuh) and CUDA's exp2f on the same inputs, for tests/test_exp2_poly.py.
#include <cuda_runtime.h>
#include "sm103_ptx.cuh"

__global__ void exp2_pair(const float* x, float* poly, float* ref, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i + 1 >= n) return;
  const float2 p = fa::exp2_poly2(make_float2(x[i], x[i + 1]));
  poly[i] = p.x;
  poly[i + 1] = p.y;
  ref[i] = exp2f(x[i]);
  ref[i + 1] = exp2f(x[i + 1]);
}

extern "C" int exp2_poly_check(const float* x, float* poly, float* ref, int n) {
  exp2_pair<<<(n / 2 + 255) / 256, 256>>>(x, poly, ref, n);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 1;
}
