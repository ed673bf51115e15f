// opd.cu -- fused OPD loss forward + backward on sm_103a.
//
// Method ("AdaFlash: Taming Variance in Diffusion Speculative Decoding",
// "The Reverse-KL + Hard-Label Mixture Loss, Derived" and "Algorithm 2:
// Entry-Wise Clipped Reverse-KL"), per draft row paired with a target row:
//   t_v = q_v (lq_v - lp_v);  loss = sum_v clamp(t_v, -c, c) - lambda lq[x*]
//   dz_v = gs/T (q_v (a_v - S) + lambda (q_v - [v = x*])),
//   a_v = [-c < t_v < c] (lq_v - lp_v + 1),  S = sum_v q_v a_v.
// The gradient needs two row-wide reductions (the two log-sum-exps, then S)
// before any dz_v can be written, so the row must stay on chip between them.
//
// GPU design.  A thread-block cluster of CL CTAs (CL <= 8) owns one row at a
// time; CTA r of the cluster holds vocabulary slice [r*SL, (r+1)*SL) of both
// the target and the draft row in shared memory.
//   * The slices arrive by 1-D bulk asynchronous copies (cp.async.bulk, one
//     per tensor per CTA, completion counted on an mbarrier); with two stages
//     the next row's copies are in flight while the current row computes, so
//     HBM sees each logit byte once.
//   * Pass A (max, argmax, sum of exp2 for both rows) -> CTA partial -> DSMEM
//     exchange across the cluster (barrier.cluster) -> every CTA merges the
//     CL partials in rank order (identical results everywhere).
//   * Pass B (clamped terms, S) -> second exchange.
//   * Pass C writes dz with 16-byte streaming stores.
// Every wait on a bulk copy is bounded by a clock deadline; on expiry the CTA
// records SVW_DEV_TIMEOUT, stops issuing copies and keeps joining the cluster
// barriers so that no peer can hang.
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace cg = cooperative_groups;

namespace svw {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

struct OpdSmem {
  unsigned long long mbar[2];
  float red[kWarps][4];
  float redv[kWarps];
  int32_t redi[kWarps];
  float partA[8];  // mt, st, md, sd, amax value, amax index (bits), abort, -
  float partB[4];  // rkl, S, abort, -
  int32_t abort;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait: false if the deadline passed first
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         unsigned long long *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// target row paired with draft row r, or -1 if r lies outside its request's
// CSR range (bad offsets)
__device__ __forceinline__ int64_t target_row_of(const OpdArgs &a, int64_t r) {
  if (!a.has_bonus) return r;
  int32_t lo = 0, hi = a.N - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(a.cu + mid)) <= r) lo = mid;
    else hi = mid - 1;
  }
  const int64_t c0 = __ldg(a.cu + lo), c1 = __ldg(a.cu + lo + 1);
  if (!(c0 <= r && r < c1)) return -1;
  return r + lo;
}

template <int DT, bool BULK, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) opd_kernel(OpdArgs a, int32_t SL, int32_t slice_bytes) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ OpdSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nclusters = gridDim.x / CL;
  const int64_t cid = blockIdx.x / CL;
  const int64_t V = a.V;
  const int64_t lo = static_cast<int64_t>(rank) * SL;
  const int64_t n = max(static_cast<int64_t>(0), min(static_cast<int64_t>(SL), V - lo));
  const float k = a.k;

  unsigned char *tbuf[2], *dbuf[2];
  for (int s = 0; s < 2; ++s) {
    const int ss = (STAGES == 2) ? s : 0;
    tbuf[s] = dyn + static_cast<size_t>(ss) * 2 * slice_bytes;
    dbuf[s] = tbuf[s] + slice_bytes;
  }

  if (tid == 0) {
    mbar_init(&sm.mbar[0], 1);
    mbar_init(&sm.mbar[1], 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  // thread 0 starts the copies of row r into stage s
  auto issue = [&](int64_t r, int s) {
    const int64_t tr = target_row_of(a, r);
    if (!BULK) return;
    if (sm.abort) return;
    const uint32_t bytes = static_cast<uint32_t>(n * E::kSize);
    if (tr >= 0 && bytes > 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&sm.mbar[s], 2 * bytes);
      bulk_g2s(tbuf[s], static_cast<const char *>(a.target) + (tr * V + lo) * E::kSize, bytes,
               &sm.mbar[s]);
      bulk_g2s(dbuf[s], static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize, bytes,
               &sm.mbar[s]);
    } else {
      mbar_arrive(&sm.mbar[s]);
    }
  };

  int64_t it = 0;
  if (STAGES == 2 && cid < a.R && tid == 0) issue(cid, 0);
  for (int64_t r = cid; r < a.R; r += nclusters, ++it) {
    const int s = (STAGES == 2) ? static_cast<int>(it & 1) : 0;
    const uint32_t parity = static_cast<uint32_t>(((STAGES == 2) ? (it >> 1) : it) & 1);
    if (tid == 0) {
      if (STAGES == 2) {
        if (r + nclusters < a.R) issue(r + nclusters, s ^ 1);
      } else {
        issue(r, 0);
      }
    }
    const int64_t tr = target_row_of(a, r);
    const bool valid = (tr >= 0);
    if (BULK) {
      if (!sm.abort) {
        if (!mbar_wait_bounded(&sm.mbar[s], parity)) {
          if (tid == 0 && a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
          sm.abort = 1;
        }
      }
      __syncthreads();
    } else {
      // scalar fill (rows not 16-byte pitched): plain loads into shared memory
      if (valid) {
        const char *ts = static_cast<const char *>(a.target) + (tr * V + lo) * E::kSize;
        const char *ds = static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize;
        for (int64_t v = tid; v < n; v += kThreads) {
          if (DT == 1) {
            reinterpret_cast<unsigned short *>(tbuf[s])[v] = __ldg(reinterpret_cast<const unsigned short *>(ts) + v);
            reinterpret_cast<unsigned short *>(dbuf[s])[v] = __ldg(reinterpret_cast<const unsigned short *>(ds) + v);
          } else {
            reinterpret_cast<float *>(tbuf[s])[v] = __ldg(reinterpret_cast<const float *>(ts) + v);
            reinterpret_cast<float *>(dbuf[s])[v] = __ldg(reinterpret_cast<const float *>(ds) + v);
          }
        }
      }
      __syncthreads();
    }
    const bool work = valid && !sm.abort;
    const unsigned char *T = tbuf[s];
    const unsigned char *D = dbuf[s];
    const int64_t nvec = n / EPV;      // whole 16-byte vectors of the slice
    const int64_t ntail = n - nvec * EPV;

    // ---------------- pass A: max / argmax / sum-exp of both rows ----------------
    float mt = -INFINITY, md = -INFINITY, st = 0.f, sd = 0.f;
    int32_t ai = INT32_MAX;
    float av = -INFINITY;
    if (work) {
      auto visit_max = [&](float y, float z, int64_t v) {
        if (y > av || (ai == INT32_MAX && y == y)) {
          av = y;
          ai = static_cast<int32_t>(v);
        }
        mt = fmaxf(mt, y);
        md = fmaxf(md, z);
      };
      for (int64_t vi = tid; vi < nvec; vi += kThreads) {
        float y[EPV], z[EPV];
        E::unpack(*reinterpret_cast<const uint4 *>(T + vi * 16), y);
        E::unpack(*reinterpret_cast<const uint4 *>(D + vi * 16), z);
#pragma unroll
        for (int e = 0; e < EPV; ++e) visit_max(y[e], z[e], lo + vi * EPV + e);
      }
      if (tid == 0)
        for (int64_t v = nvec * EPV; v < n; ++v) {
          const float y = E::load_plain(T, v), z = E::load_plain(D, v);
          visit_max(y, z, lo + v);
        }
      const float mtr = (mt == -INFINITY) ? 0.f : mt;
      const float mdr = (md == -INFINITY) ? 0.f : md;
      for (int64_t vi = tid; vi < nvec; vi += kThreads) {
        float y[EPV], z[EPV];
        E::unpack(*reinterpret_cast<const uint4 *>(T + vi * 16), y);
        E::unpack(*reinterpret_cast<const uint4 *>(D + vi * 16), z);
        float ps = 0.f, qs = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          ps = __fadd_rn(ps, ex2(__fmul_rn(__fsub_rn(y[e], mtr), k)));
          qs = __fadd_rn(qs, ex2(__fmul_rn(__fsub_rn(z[e], mdr), k)));
        }
        st = __fadd_rn(st, ps);
        sd = __fadd_rn(sd, qs);
      }
      if (tid == 0)
        for (int64_t v = nvec * EPV; v < n; ++v) {
          st = __fadd_rn(st, ex2(__fmul_rn(__fsub_rn(E::load_plain(T, v), mtr), k)));
          sd = __fadd_rn(sd, ex2(__fmul_rn(__fsub_rn(E::load_plain(D, v), mdr), k)));
        }
    }
    (void)ntail;
    // block reduction of (mt, st), (md, sd), (av, ai)
    warp_lse(mt, st, k);
    warp_lse(md, sd, k);
    warp_amax(av, ai);
    if (lane == 0) {
      sm.red[warp][0] = mt;
      sm.red[warp][1] = st;
      sm.red[warp][2] = md;
      sm.red[warp][3] = sd;
      sm.redv[warp] = av;
      sm.redi[warp] = ai;
    }
    __syncthreads();
    if (warp == 0) {
      float a0 = -INFINITY, a1 = 0.f, a2 = -INFINITY, a3 = 0.f, vv = -INFINITY;
      int32_t ii = INT32_MAX;
      if (lane < kWarps) {
        a0 = sm.red[lane][0];
        a1 = sm.red[lane][1];
        a2 = sm.red[lane][2];
        a3 = sm.red[lane][3];
        vv = sm.redv[lane];
        ii = sm.redi[lane];
      }
      warp_lse(a0, a1, k);
      warp_lse(a2, a3, k);
      warp_amax(vv, ii);
      if (lane == 0) {
        sm.partA[0] = a0;
        sm.partA[1] = a1;
        sm.partA[2] = a2;
        sm.partA[3] = a3;
        sm.partA[4] = vv;
        sm.partA[5] = __int_as_float(ii);
        sm.partA[6] = sm.abort ? 1.f : 0.f;
      }
    }
    cluster.sync();
    // merge the CL partials in rank order (same result in every CTA)
    float Mt = -INFINITY, St = 0.f, Md = -INFINITY, Sd = 0.f, Av = -INFINITY;
    int32_t Ai = INT32_MAX;
    bool any_abort = false;
    for (int q = 0; q < CL; ++q) {
      const float *pa = cluster.map_shared_rank(sm.partA, q);
      lse_combine(Mt, St, pa[0], pa[1], k);
      lse_combine(Md, Sd, pa[2], pa[3], k);
      amax_combine(Av, Ai, pa[4], __float_as_int(pa[5]));
      any_abort |= (pa[6] != 0.f);
    }
    const bool row_ok = valid && !any_abort && (St > 0.f && St <= FLT_MAX) && (Sd > 0.f && Sd <= FLT_MAX);
    const float lt = lg2(St), ld = lg2(Sd);
    const float c = a.clip_c;

    // ---------------- pass B: clamped reverse-KL terms and S ----------------
    float rkl = 0.f, S = 0.f;
    auto term = [&](float y, float z, float &qv, float &qa, float &tcl) {
      const float lp = __fsub_rn(__fmul_rn(__fsub_rn(y, Mt), k), lt);  // log2 p
      const float lq = __fsub_rn(__fmul_rn(__fsub_rn(z, Md), k), ld);  // log2 q
      qv = ex2(lq);
      if (qv == 0.f) {
        qa = 0.f;
        tcl = 0.f;
        return;
      }
      const float d = __fmul_rn(__fsub_rn(lq, lp), kLn2);  // ln q - ln p
      const float t = __fmul_rn(qv, d);
      tcl = fminf(fmaxf(t, -c), c);
      qa = (t > -c && t < c) ? __fmul_rn(qv, __fadd_rn(d, 1.f)) : 0.f;
    };
    if (row_ok) {
      for (int64_t vi = tid; vi < nvec; vi += kThreads) {
        float y[EPV], z[EPV];
        E::unpack(*reinterpret_cast<const uint4 *>(T + vi * 16), y);
        E::unpack(*reinterpret_cast<const uint4 *>(D + vi * 16), z);
        float r1 = 0.f, s1 = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          float qv, qa, tcl;
          term(y[e], z[e], qv, qa, tcl);
          r1 = __fadd_rn(r1, tcl);
          s1 = __fadd_rn(s1, qa);
        }
        rkl = __fadd_rn(rkl, r1);
        S = __fadd_rn(S, s1);
      }
      if (tid == 0)
        for (int64_t v = nvec * EPV; v < n; ++v) {
          float qv, qa, tcl;
          term(E::load_plain(T, v), E::load_plain(D, v), qv, qa, tcl);
          rkl = __fadd_rn(rkl, tcl);
          S = __fadd_rn(S, qa);
        }
    }
    rkl = warp_sum(rkl);
    S = warp_sum(S);
    if (lane == 0) {
      sm.red[warp][0] = rkl;
      sm.red[warp][1] = S;
    }
    __syncthreads();
    if (warp == 0) {
      float r1 = (lane < kWarps) ? sm.red[lane][0] : 0.f;
      float s1 = (lane < kWarps) ? sm.red[lane][1] : 0.f;
      r1 = warp_sum(r1);
      s1 = warp_sum(s1);
      if (lane == 0) {
        sm.partB[0] = r1;
        sm.partB[1] = s1;
      }
    }
    cluster.sync();
    float RKL = 0.f, SS = 0.f;
    for (int q = 0; q < CL; ++q) {
      const float *pb = cluster.map_shared_rank(sm.partB, q);
      RKL = __fadd_rn(RKL, pb[0]);
      SS = __fadd_rn(SS, pb[1]);
    }

    if (rank == 0 && tid == 0) {
      float out = __int_as_float(0x7fffffff);
      if (row_ok) {
        const float zx = E::load(a.draft, r * V + Ai);
        const float lqx = __fsub_rn(__fmul_rn(__fsub_rn(zx, Md), k), ld);
        out = __fadd_rn(RKL, __fmul_rn(a.lambda_ce, __fmul_rn(-lqx, kLn2)));
      } else if (a.status && !any_abort) {
        atomicOr(a.status, SVW_DEV_BAD_INPUT);
      }
      a.loss[r] = out;
    }

    // ---------------- pass C: gradient wrt the draft logits ----------------
    if (a.dlogits != nullptr && valid && !any_abort) {
      const float gsT = __fmul_rn(a.grad_scale, a.invT);
      const float lam = a.lambda_ce;
      float *out = a.dlogits + r * V + lo;
      auto grad = [&](float y, float z, int64_t v) -> float {
        if (!row_ok) return __int_as_float(0x7fffffff);
        float qv, qa, tcl;
        term(y, z, qv, qa, tcl);
        float g = __fadd_rn(__fsub_rn(qa, __fmul_rn(qv, SS)), __fmul_rn(lam, qv));
        if (v == Ai) g = __fsub_rn(g, lam);
        return __fmul_rn(gsT, g);
      };
      if (BULK) {
        for (int64_t vi = tid; vi < nvec; vi += kThreads) {
          float y[EPV], z[EPV], g[EPV];
          E::unpack(*reinterpret_cast<const uint4 *>(T + vi * 16), y);
          E::unpack(*reinterpret_cast<const uint4 *>(D + vi * 16), z);
#pragma unroll
          for (int e = 0; e < EPV; ++e) g[e] = grad(y[e], z[e], lo + vi * EPV + e);
#pragma unroll
          for (int h = 0; h < EPV / 4; ++h)
            st_stream(out + vi * EPV + 4 * h, g[4 * h], g[4 * h + 1], g[4 * h + 2], g[4 * h + 3]);
        }
      } else {
        for (int64_t v = tid; v < n; v += kThreads) out[v] = grad(E::load_plain(T, v), E::load_plain(D, v), lo + v);
      }
    }
    __syncthreads();  // stage s fully consumed before it is refilled
  }
  cluster.sync();  // peers may still read this CTA's partials
}

struct OpdPlan {
  int CL;
  int SL;
  int slice_bytes;
  int stages;
  size_t smem;
};

OpdPlan plan_opd(int64_t V, int esize) {
  OpdPlan p{};
  const int64_t row_bytes = V * esize * 2;
  int64_t CL = (row_bytes + 32767) / 32768;
  if (CL < 1) CL = 1;
  if (CL > kMaxCluster) CL = kMaxCluster;
  int64_t SL = (V + CL - 1) / CL;
  SL = (SL + 7) / 8 * 8;
  p.CL = static_cast<int>(CL);
  p.SL = static_cast<int>(SL);
  p.slice_bytes = static_cast<int>((SL * esize + 127) / 128 * 128);
  const size_t stage = static_cast<size_t>(p.slice_bytes) * 2;
  const size_t cap = 200 * 1024;
  if (2 * stage <= cap) p.stages = 2;
  else if (stage <= cap) p.stages = 1;
  else p.stages = 0;
  p.smem = stage * (p.stages == 2 ? 2 : 1);
  return p;
}

template <int DT, bool BULK, int STAGES>
cudaError_t launch_opd_t(const OpdArgs &a, const OpdPlan &p, cudaStream_t st) {
  auto kern = opd_kernel<DT, BULK, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(p.smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent clusters: as many as can be co-resident (cached per shape)
  struct Entry {
    int dev, CL;
    size_t smem;
    int n;
  };
  static Entry cache[32];
  static int ncache = 0;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int maxc = 0;
  for (int q = 0; q < ncache; ++q)
    if (cache[q].dev == dev && cache[q].CL == p.CL && cache[q].smem == p.smem) maxc = cache[q].n;
  if (maxc == 0) {
    cfg.gridDim = dim3(p.CL * 1024, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (maxc <= 0) return cudaErrorInvalidConfiguration;
    if (ncache < 32) cache[ncache++] = Entry{dev, p.CL, p.smem, maxc};
  }
  int64_t nclusters = maxc;
  if (nclusters > a.R) nclusters = a.R;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * p.CL), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, a, p.SL, p.slice_bytes);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool opd_supported(int64_t V, int esize) { return plan_opd(V, esize).stages > 0; }

cudaError_t launch_opd(const OpdArgs &a, int dtype, bool bulk, cudaStream_t st) {
  const int esize = (dtype == SVW_BF16) ? 2 : 4;
  const OpdPlan p = plan_opd(a.V, esize);
  if (p.stages == 0) return cudaErrorInvalidValue;
  if (dtype == SVW_BF16) {
    if (bulk) return p.stages == 2 ? launch_opd_t<1, true, 2>(a, p, st) : launch_opd_t<1, true, 1>(a, p, st);
    return launch_opd_t<1, false, 1>(a, p, st);
  }
  if (bulk) return p.stages == 2 ? launch_opd_t<0, true, 2>(a, p, st) : launch_opd_t<0, true, 1>(a, p, st);
  return launch_opd_t<0, false, 1>(a, p, st);
}

}  // namespace svw
