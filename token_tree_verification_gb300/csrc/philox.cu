// Step R exposed on its own: the uniforms the verification and expansion
// kernels draw, for arbitrary counters, so that a caller (and the test-suite)
// can check the device generator against an independent implementation.
//
// Generator: Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11), key
// (seed, 0); uniform = top 24 bits of the first output word times 2^-24.
#include "common.cuh"

namespace spec {

__global__ void philox_uniforms_kernel(uint64_t seed, const int64_t *__restrict__ ctr, int n,
                                       float *__restrict__ u) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  U64x4 c;
#pragma unroll
  for (int w = 0; w < 4; ++w) c.w[w] = static_cast<uint64_t>(ctr[4 * static_cast<size_t>(i) + w]);
  const U64x4 r = philox4x64_10(c, seed, 0);
  u[i] = static_cast<float>(r.w[0] >> 40) * (1.0f / 16777216.0f);
}

}  // namespace spec

extern "C" int spec_philox_uniforms(uint64_t seed, const int64_t *counters, int n, float *u,
                                    void *stream) {
  if (n < 0) return SPEC_ERR_SHAPE;
  if (n == 0) return SPEC_OK;
  if (!counters || !u) return SPEC_ERR_NULL;
  const int threads = 256;
  const int blocks = (n + threads - 1) / threads;
  spec::philox_uniforms_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      seed, counters, n, u);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
