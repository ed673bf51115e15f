// lengthhead.cu -- the adaptive length head: forward and label.
//
// "AdaFlash: Taming Variance in Diffusion Speculative Decoding", "Algorithm
// 3: Adaptive Length Head, Forward Pass" ("AdaFlash：基于在策略蒸馏扩散草稿器的
// 自适应投机解码" §2.2), per request i with drafter hidden states h_i (k x H):
//   h'_p = SiLU(W1 h_i[p] + b1)   (W1: H' x H)    -- a dense contraction
//   hbar = mean_p h'_p
//   a_hat = sigmoid(w2 . hbar + b2),  k_hat = clamp(floor(gamma a_hat k), 1, k)
// and "Online Update of the Length Head, Derived": a* = accept_len / L,
// loss = (a_hat - a*)^2.
//
// GPU design.  The projection of all N k positions is one plain GEMM
// ([N k, H] x [H, H'], bf16 in, fp32 out), run by cuBLASLt on the caller's
// workspace (no device allocation; plans cached per shape and device).  One
// kernel then does everything else per request: bias, SiLU, the mean over the
// k positions, the dot with w2, the sigmoid and the clamp.
#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace svw {

namespace {

constexpr int kHeadThreads = 256;

// per request: SiLU(Y + b1), mean over positions, dot w2, sigmoid, clamp
__global__ void __launch_bounds__(kHeadThreads) length_head_epilogue(const float *Y, const float *b1,
                                                                     const float *w2, float b2, int32_t k,
                                                                     int32_t Hp, float gamma, float *a_hat,
                                                                     int32_t *k_hat) {
  __shared__ float red[kHeadThreads / 32];
  const int32_t i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float part = 0.f;
  for (int j = tid; j < Hp; j += kHeadThreads) {
    const float bj = __ldg(b1 + j);
    float s = 0.f;
    // eight positions' loads in flight at once; the sum stays sequential over p
    for (int p0 = 0; p0 < k; p0 += 8) {
      float y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        y[u] = (p0 + u < k) ? __ldg(Y + (static_cast<int64_t>(i) * k + p0 + u) * Hp + j) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p0 + u < k) {
          const float g = y[u] + bj;
          s += g / (1.f + expf(-g));  // SiLU
        }
    }
    part = fmaf(__ldg(w2 + j), s / static_cast<float>(k), part);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) red[warp] = part;
  __syncthreads();
  if (tid == 0) {
    float z = b2;
    for (int w = 0; w < kHeadThreads / 32; ++w) z += red[w];
    const float a = 1.f / (1.f + expf(-z));
    float kh = floorf(gamma * a * static_cast<float>(k));
    kh = fminf(fmaxf(kh, 1.f), static_cast<float>(k));
    a_hat[i] = a;
    k_hat[i] = static_cast<int32_t>(kh);
  }
}

__global__ void length_label_kernel(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                                    float *a_star, float *loss) {
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const int32_t L = __ldg(cu + i + 1) - __ldg(cu + i);
  const int32_t acc = __ldg(accept_len + i);
  if (acc < 0 || L < 1) {
    a_star[i] = __int_as_float(0x7fffffff);
    if (loss) loss[i] = __int_as_float(0x7fffffff);
    return;
  }
  const float as = static_cast<float>(acc) / static_cast<float>(L);
  a_star[i] = as;
  if (loss) {
    const float d = __ldg(a_hat + i) - as;
    loss[i] = d * d;
  }
}

// cuBLASLt plans, one per (device, shape); created once, never freed
struct GemmPlan {
  int dev;
  int32_t M, H, Hp;
  cublasLtMatmulDesc_t op;
  cublasLtMatrixLayout_t a, b, c;
  cublasLtMatmulAlgo_t algo;
  size_t ws;
};
std::mutex g_mu;
cublasLtHandle_t g_handle = nullptr;
GemmPlan g_plans[32];
int g_nplans = 0;

// Y (row-major [M, Hp], fp32) = X (row-major [M, H], bf16) * W1^T (W1 row-major [Hp, H], bf16).
// In cuBLASLt's column-major terms: Y^T [Hp, M] = W1' [Hp, H] * X^T [H, M],
// with W1' = (W1 viewed column-major [H, Hp])^T.
const GemmPlan *get_plan(int dev, int32_t M, int32_t H, int32_t Hp, size_t max_ws) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int q = 0; q < g_nplans; ++q)
    if (g_plans[q].dev == dev && g_plans[q].M == M && g_plans[q].H == H && g_plans[q].Hp == Hp &&
        g_plans[q].ws <= max_ws)
      return &g_plans[q];
  if (g_nplans >= 32) return nullptr;
  if (!g_handle && cublasLtCreate(&g_handle) != CUBLAS_STATUS_SUCCESS) return nullptr;
  GemmPlan p{};
  p.dev = dev;
  p.M = M;
  p.H = H;
  p.Hp = Hp;
  if (cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return nullptr;
  const cublasOperation_t tA = CUBLAS_OP_T, tB = CUBLAS_OP_N;
  cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSA, &tA, sizeof(tA));
  cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSB, &tB, sizeof(tB));
  if (cublasLtMatrixLayoutCreate(&p.a, CUDA_R_16BF, H, Hp, H) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&p.b, CUDA_R_16BF, H, M, H) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&p.c, CUDA_R_32F, Hp, M, Hp) != CUBLAS_STATUS_SUCCESS)
    return nullptr;
  cublasLtMatmulPreference_t pref;
  if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) return nullptr;
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &max_ws, sizeof(max_ws));
  cublasLtMatmulHeuristicResult_t res[1];
  int found = 0;
  const cublasStatus_t st =
      cublasLtMatmulAlgoGetHeuristic(g_handle, p.op, p.a, p.b, p.c, p.c, pref, 1, res, &found);
  cublasLtMatmulPreferenceDestroy(pref);
  if (st != CUBLAS_STATUS_SUCCESS || found < 1) return nullptr;
  p.algo = res[0].algo;
  p.ws = res[0].workspaceSize;
  g_plans[g_nplans] = p;
  return &g_plans[g_nplans++];
}

}  // namespace

size_t length_head_gemm_bytes(int32_t N, int32_t k, int32_t Hp) {
  return (static_cast<size_t>(N) * k * Hp * sizeof(float) + 255) / 256 * 256;
}

int launch_length_head(const void *hidden, const void *w1, const float *b1, const float *w2, float b2, int32_t N,
                       int32_t k, int32_t H, int32_t Hp, float gamma, float *a_hat, int32_t *k_hat,
                       void *workspace, size_t workspace_bytes, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const size_t ybytes = length_head_gemm_bytes(N, k, Hp);
  char *ws = static_cast<char *>(workspace);
  float *Y = reinterpret_cast<float *>(ws);
  const GemmPlan *p = get_plan(dev, N * k, H, Hp, workspace_bytes - ybytes);
  if (!p) return 2;
  const float alpha = 1.f, beta = 0.f;
  void *tm = timer_before("length_head_gemm", st);
  const cublasStatus_t s = cublasLtMatmul(g_handle, p->op, &alpha, w1, p->a, hidden, p->b, &beta, Y, p->c, Y, p->c,
                                          &p->algo, ws + ybytes, p->ws, st);
  timer_after(tm, st);
  if (s != CUBLAS_STATUS_SUCCESS) return 3;
  tm = timer_before("length_head_epilogue", st);
  length_head_epilogue<<<N, kHeadThreads, 0, st>>>(Y, b1, w2, b2, k, Hp, gamma, a_hat, k_hat);
  timer_after(tm, st);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_length_label(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                        float *a_star, float *loss, cudaStream_t st) {
  length_label_kernel<<<(N + 255) / 256, 256, 0, st>>>(accept_len, cu, a_hat, N, a_star, loss);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace svw
