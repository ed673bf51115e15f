// fused.cu -- per-request step of spec_verify_opd (verification and the OPD
// loss on the same batch in one pass over the logits).
//
// The OPD fast kernel has already reduced every draft row together with its
// target row (in log2 units log2 p = y k - Ct and log2 q - log2 p =
// (z - y) k - dC; the target argmax x*) and every bonus row (Ct, argmax).
// What verification still needs per request is what "Speculative Decoding:
// The Basic Idea" steps 3-4 ("AdaFlash: Taming Variance in Diffusion
// Speculative Decoding") and "DFlash 阅读笔记" §5.1-§5.2 define on top of the
// two softmaxes: the accept test at each drafted token, the leftmost
// rejection and the next token.  One CTA per request (at T > 0 a cluster of
// CTAs): warp 0 of CTA 0 (lane j tests position j) decides, then at T > 0 the
// cluster draws the next token by inverse CDF (svw_sample.cuh).
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"
#include "svw_sample.cuh"

namespace svw {

namespace {

constexpr int kFThreads = 512;  // one CTA (or, at T > 0, a cluster of CTAs) per request

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kFThreads) fused_finalize(FusedArgs a) {
  using E = Elem<DT>;
  __shared__ int32_t s_js;
  __shared__ float s_nT, s_nD;
  __shared__ uint32_t s_draw[4];  // the draw's inputs from CTA 0 of the cluster: js, nT, nD, resid
  __shared__ SampleSmem<kFThreads> ssm;
  extern __shared__ float sample_w[];  // T > 0: the draw's warp totals
  // at T > 0 a cluster of CL CTAs serves request i: warp 0 of CTA 0 tests,
  // then all of them draw the next token (one slice of the row each)
  const int CL = GREEDY ? 1 : static_cast<int>(cluster_size());
  const int rank = GREEDY ? 0 : static_cast<int>(cluster_rank());
  const int lane = threadIdx.x & 31;
  const int32_t i = blockIdx.x / CL;
  if (rank != 0) {
    // the other CTAs of the cluster only draw (they read no output of the stream kernel)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else if (threadIdx.x >= 32) {
    // warps 1.. only take part in the draw
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (GREEDY) return;
  } else {
    // ---- inputs only: overlaps the end of the fast kernel ----
    const int64_t c_i = __ldg(a.cu + i), c_e = __ldg(a.cu + i + 1);
    const bool len_ok = (c_e - c_i >= 1 && c_e - c_i <= a.max_len && c_i >= 0 && c_e <= a.total_rows);
    const int32_t L = len_ok ? static_cast<int32_t>(c_e - c_i) : 0;
    const int64_t t0 = c_i + i, d0 = c_i;
    int32_t x = 0;
    bool tok_ok = true;
    float yx = 0.f, zx = 0.f, u = 0.f;
    if (lane < L) {
      x = __ldg(a.tokens + d0 + lane);
      tok_ok = (x >= 0 && static_cast<int64_t>(x) < a.V);
      if (tok_ok && !GREEDY) {
        yx = E::load(a.target, (t0 + lane) * a.V + x);
        zx = E::load(a.draft, (d0 + lane) * a.V + x);
        u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(lane), 0u);
      }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // row constants and CSR flags are complete
    // the fix-up grid that follows reads only the fast kernel's output: it may start now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    int csr_bad = 0;
    for (int b = lane; b < a.csr_grid; b += 32) csr_bad |= __ldcg(a.csr_bad + b);
    float Ct = 0.f, dC = 0.f;
    int32_t xs = -1;
    bool row_bad = false;
    if (lane < L) {
      const float4 rc = __ldcg(a.rowc + d0 + lane);
      Ct = rc.x;
      dC = rc.y;
      xs = __float_as_int(rc.z);
      row_bad = !(Ct == Ct);
    }
    // the bonus row: merge the fast kernel's per-CTA partials (lane q <- CTA q)
    float bm = -INFINITY, bs = 0.f;
    int32_t bidx = INT32_MAX, bflag = 0;
    if (len_ok && lane < a.bparts) {
      const float4 q = __ldcg(a.bpart + static_cast<int64_t>(i) * kBonusParts + lane);
      bm = q.x;
      bs = q.y;
      bidx = __float_as_int(q.z);
      bflag = __float_as_int(q.w);
    }
    float bM = bm;
  #pragma unroll
    for (int o = kBonusParts / 2; o > 0; o >>= 1) bM = fmaxf(bM, __shfl_xor_sync(0xffffffffu, bM, o));
    float bS = (bm == -INFINITY) ? bs * 0.f : bs * ex2((bm - bM) * a.k);
  #pragma unroll
    for (int o = kBonusParts / 2; o > 0; o >>= 1) bS += __shfl_xor_sync(0xffffffffu, bS, o);
    // the butterfly spans lanes 0 .. kBonusParts - 1: every lane takes lane 0's merge
    bM = __shfl_sync(0xffffffffu, bM, 0);
    bS = __shfl_sync(0xffffffffu, bS, 0);
    const int32_t bx = static_cast<int32_t>(__reduce_min_sync(
        0xffffffffu, static_cast<uint32_t>((lane < kBonusParts && bm == bM) ? bidx : INT32_MAX)));
    const bool bonus_bad = len_ok && (__any_sync(0xffffffffu, bflag != 0) || !(bS > 0.f && bS <= FLT_MAX) ||
                                      bx == INT32_MAX);
    const float4 br = make_float4(fmaf(bM, a.k, lg2(bS)), __int_as_float(bx), 0.f, 0.f);
    const bool bad = !len_ok || __any_sync(0xffffffffu, csr_bad != 0 || !tok_ok || row_bad) || bonus_bad;
    if (bad) {
      if (lane == 0) {
        a.accept_len[i] = -1;
        a.next_token[i] = -1;
        s_js = -1;
        if (a.status) atomicOr(a.status, SVW_DEV_BAD_INPUT);
      }
    } else {
      bool acc = true;
      if (lane < L) {
        if (GREEDY) {
          acc = (x == xs);
        } else if (zx == -INFINITY) {
          acc = true;  // q(x) = 0: accept
        } else {
          // log2 p(x) - log2 q(x) = (y_x - z_x) k + dC (the logit difference is exact)
          const float dl = __fmaf_rn(__fsub_rn(yx, zx), a.k, dC);
          acc = u < ((dl >= 0.f) ? 1.f : ex2(dl));
        }
      }
      const unsigned rej = __ballot_sync(0xffffffffu, !acc);
      const int32_t js = rej ? (__ffs(rej) - 1) : L;
      const int src = (js < L) ? js : 0;
      const int32_t xs_js = __shfl_sync(0xffffffffu, xs, src);
      const float Ct_js = __shfl_sync(0xffffffffu, Ct, src);
      const float Cd_js = Ct_js + __shfl_sync(0xffffffffu, dC, src);
      if (lane == 0) {
        a.accept_len[i] = js;
        if (GREEDY) a.next_token[i] = (js < L) ? xs_js : __float_as_int(br.y);
        s_js = js;
        // the draw's offsets: log2 p = y k - Ct, log2 q = z k - Cd
        s_nT = -((js < L) ? Ct_js : br.x);
        s_nD = -Cd_js;
      }
    }
  }
  if (GREEDY) return;
  __syncthreads();
  // the draw's inputs to every CTA of the cluster
  if (rank == 0 && threadIdx.x < static_cast<unsigned>(CL)) {
    const int32_t js = s_js;
    const int32_t L = __ldg(a.cu + i + 1) - __ldg(a.cu + i);
    const uint32_t v[4] = {static_cast<uint32_t>(js), __float_as_uint(s_nT), __float_as_uint(s_nD),
                           (js >= 0 && js < L) ? 1u : 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q) st_cluster_b32(mapa_shared(smem_u32(&s_draw[q]), threadIdx.x), v[q]);
  }
  cluster_barrier();
  const int32_t js = static_cast<int32_t>(s_draw[0]);
  if (js < 0) return;  // the same in every CTA of the cluster
  // ---- the next token by inverse CDF: [p - q]_+ at row js, or p at the bonus row ----
  const int64_t c_i = __ldg(a.cu + i);
  RowConst rc;
  rc.k = a.k;
  rc.resid = s_draw[3] != 0;
  rc.nT = __uint_as_float(s_draw[1]);
  rc.nD = __uint_as_float(s_draw[2]);
  const char *trow = static_cast<const char *>(a.target) + (c_i + i + js) * a.V * E::kSize;
  const char *drow = rc.resid ? static_cast<const char *>(a.draft) + (c_i + js) * a.V * E::kSize : nullptr;
  const float w = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(js), 1u);
  const int32_t tok = cluster_sample<DT, true, kFThreads>(trow, drow, a.V, rc, w, ssm, sample_w, CL, rank);
  if (threadIdx.x == 0 && tok >= 0) a.next_token[i] = tok;
}

// at T > 0 a cluster of CL CTAs per request (draw_cluster), each with the
// draw's dynamic shared memory
template <int DT>
cudaError_t launch_t(const FusedArgs &a, bool greedy, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  int cl = 1;
  size_t smem = 0;
  if (!greedy) {
    cl = draw_cluster(a.N);
    smem = sample_dyn_bytes(a.V, cl, kFThreads);
    e = cudaFuncSetAttribute(fused_finalize<DT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(a.N) * static_cast<unsigned>(cl), 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = greedy ? 1 : 2;
  void *tm = timer_before("fused_finalize", st);
  e = greedy ? cudaLaunchKernelEx(&cfg, fused_finalize<DT, true>, a)
             : cudaLaunchKernelEx(&cfg, fused_finalize<DT, false>, a);
  timer_after(tm, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_finalize(const FusedArgs &a, int dtype, bool greedy, cudaStream_t st) {
  return (dtype == SVW_BF16) ? launch_t<1>(a, greedy, st) : launch_t<0>(a, greedy, st);
}

}  // namespace svw
