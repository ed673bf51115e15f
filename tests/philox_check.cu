// philox_check.cu -- test harness (not part of the library): evaluates the
// library's device Philox4x32-10 (svw_device.cuh) and CUDA's own
// curand_Philox4x32_10 on the same counters and keys, for the three-way check
// against the oracle in test_gpu_philox.py.
#include <cstdint>
#include <cuda_runtime.h>
#include <curand_philox4x32_x.h>

#include "../serving_vocab_wide_gb300/csrc/svw_device.cuh"

__global__ void philox_pairs(const uint32_t *ctr, const uint64_t *seed, int n, uint32_t *lib_w0, float *lib_u,
                             uint32_t *cur) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = make_uint4(ctr[3 * i], ctr[3 * i + 1], ctr[3 * i + 2], 0u);
  const uint2 k = make_uint2(static_cast<uint32_t>(seed[i]), static_cast<uint32_t>(seed[i] >> 32));
  const uint4 r = curand_Philox4x32_10(c, k);
  cur[4 * i] = r.x;
  cur[4 * i + 1] = r.y;
  cur[4 * i + 2] = r.z;
  cur[4 * i + 3] = r.w;
  lib_w0[i] = svw::philox_word0(seed[i], c.x, c.y, c.z);
  lib_u[i] = svw::philox_uniform(seed[i], c.x, c.y, c.z);
}

// host arrays in, host arrays out; returns a cudaError_t
extern "C" int philox_check(const uint32_t *ctr, const uint64_t *seed, int n, uint32_t *lib_w0, float *lib_u,
                            uint32_t *cur) {
  uint32_t *dctr = nullptr, *dw0 = nullptr, *dcur = nullptr;
  uint64_t *dseed = nullptr;
  float *du = nullptr;
  cudaError_t e = cudaMalloc(&dctr, 3 * sizeof(uint32_t) * n);
  if (e == cudaSuccess) e = cudaMalloc(&dseed, sizeof(uint64_t) * n);
  if (e == cudaSuccess) e = cudaMalloc(&dw0, sizeof(uint32_t) * n);
  if (e == cudaSuccess) e = cudaMalloc(&du, sizeof(float) * n);
  if (e == cudaSuccess) e = cudaMalloc(&dcur, 4 * sizeof(uint32_t) * n);
  if (e == cudaSuccess) e = cudaMemcpy(dctr, ctr, 3 * sizeof(uint32_t) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(dseed, seed, sizeof(uint64_t) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    philox_pairs<<<(n + 255) / 256, 256>>>(dctr, dseed, n, dw0, du, dcur);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(lib_w0, dw0, sizeof(uint32_t) * n, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(lib_u, du, sizeof(float) * n, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(cur, dcur, 4 * sizeof(uint32_t) * n, cudaMemcpyDeviceToHost);
  cudaFree(dctr);
  cudaFree(dseed);
  cudaFree(dw0);
  cudaFree(du);
  cudaFree(dcur);
  return static_cast<int>(e);
}
