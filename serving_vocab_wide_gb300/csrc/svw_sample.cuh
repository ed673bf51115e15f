// svw_sample.cuh -- inverse-CDF draw of the next token by a thread-block
// cluster.
//
// "DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.2 eq. (7) and Algorithm 1
// (and "AdaFlash: Taming Variance in Diffusion Speculative Decoding",
// "Speculative Decoding: The Basic Idea" step 4): after the first rejection
// the next token is drawn from the normalised residual [p - q]_+ of that row,
// or from p of the bonus row when every drafted token passed.  The draw is an
// inverse CDF in vocabulary order: the smallest v with C_v > w Z, where C is
// the prefix sum of the weights, Z their total and w the request's uniform.
//
// The row is cut into one slice per CTA of the cluster, so a request's row
// pair streams through several SMs at once (and a batch of requests spreads
// evenly over the GPU); each CTA keeps its slice's round and warp totals on
// chip, the slice totals are exchanged, and only the crossing warp's 32
// groups are read a second time.  Rounding can leave a
// level without a crossing (or w Z can round up to Z): then the last entry
// with positive weight of the slice (or row) is taken -- such draws are within
// float rounding of a CDF boundary.  A rejected row whose residual rounds to
// zero mass is drawn from p.
#pragma once

#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "svw_device.cuh"

namespace svw {

// log2 p = y k + nT, log2 q = z k + nD (one rounding each)
struct RowConst {
  float k, nT, nD;
  bool resid;
};

// [p - q]_+ from log2 p and log2 q (both exp2 evaluated, then a select: the
// same value as sample_weight's)
__device__ __forceinline__ float resid_weight(float lp, float lq) {
  const float d = fmaxf(__fsub_rn(ex2(lp), ex2(lq)), 0.f);
  return (lq < lp) ? d : 0.f;
}

// [p - q]_+ (resid) or p
__device__ __forceinline__ float sample_weight(float y, float z, const RowConst &c) {
  const float lp = __fmaf_rn(y, c.k, c.nT);
  if (!c.resid) return ex2(lp);
  const float lq = __fmaf_rn(z, c.k, c.nD);
  if (!(lq < lp)) return 0.f;
  return fmaxf(__fsub_rn(ex2(lp), ex2(lq)), 0.f);
}

// raw logits of group g (entries 8g .. 8g+7, -inf at v >= V)
template <int DT, bool VEC>
__device__ __forceinline__ void sample_load_group(const char *row, int64_t g, int64_t V, float (&x)[8]) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  const int64_t v0 = g * 8;
  if (VEC) {
#pragma unroll
    for (int h = 0; h < 8 / EPV; ++h) {
      const int64_t vv = v0 + h * EPV;
      if (vv < V) {
        E::unpack(ld_vec(row + vv * E::kSize), x + h * EPV);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) x[h * EPV + e] = -INFINITY;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (v0 + e < V) ? E::load(row, v0 + e) : -INFINITY;
  }
}

// the 8 weights of group g and their sequential sum a_g (0 at g >= NG, the
// end of the row or of the caller's slice)
template <int DT, bool VEC>
__device__ __forceinline__ float sample_group(const char *trow, const char *drow, int64_t g, int64_t NG,
                                              int64_t V, const RowConst &c, float (&w)[8]) {
  float a = 0.f;
  if (g >= NG) {
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = 0.f;
    return a;
  }
  float y[8], z[8];
  sample_load_group<DT, VEC>(trow, g, V, y);
  if (c.resid) sample_load_group<DT, VEC>(drow, g, V, z);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = sample_weight(y[e], c.resid ? z[e] : 0.f, c);
    a = __fadd_rn(a, w[e]);
  }
  return a;
}

// inclusive prefix over the warp's lanes (fixed shuffle tree)
__device__ __forceinline__ float warp_scan_incl(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, y);
  }
  return x;
}

// shared memory of cluster_sample
constexpr int kMaxSampleCluster = 8;
// The warp totals of a CTA's slice (round-major, NT / 32 per round) live in
// dynamic shared memory: sample_dyn_bytes() per CTA.
template <int NT>
struct SampleSmem {
  static constexpr int kMaxRounds = ((1 << 20) / 8 + NT - 1) / NT;  // V <= 2^20
  float R[kMaxRounds];  // round totals of this CTA's slice
  float Zs[kMaxSampleCluster];    // slice totals of the cluster, one per CTA (pushed by every peer)
  int32_t lg[kMaxSampleCluster];  // last group with positive weight, per slice (-1: none)
  int32_t lastg;                  // this CTA's
  int32_t rs, ws, degenerate, spick;
  float t, Pr, Qw;
};

// dynamic shared memory of cluster_sample for rows of V entries cut into CL
// slices: the warp totals of a slice
__host__ __device__ inline size_t sample_dyn_bytes(int64_t V, int CL, int NT) {
  const int64_t NG = (V + 7) / 8, P = (NG + CL - 1) / CL, nR = (P + NT - 1) / NT;
  return static_cast<size_t>(nR) * (NT / 32) * sizeof(float);
}

// The next token drawn from row trow (and drow when rc.resid) by the CL CTAs
// of a thread-block cluster, NT threads each; wu: the request's uniform in
// [0, 1).  CTA `rank` streams groups [rank P, (rank + 1) P) of the row (P =
// ceil(NG / CL)); the slice totals are exchanged through distributed shared
// memory, the crossing slice is found by every CTA alike, and only the CTA
// that owns it resolves the round, lane and entry levels.  Returns the token
// in the CTA that drew it, -1 in the others (every thread of a CTA returns
// the same).  Every CTA of the cluster must call it with the same arguments
// (but its own rank); it ends with no peer access outstanding.
//
// Prefix definition (fp32, each level a fixed order of adds): groups of 8
// entries (sequential), warps of 32 groups (shuffle scan), rounds of NT / 32
// warps (sequential), the rounds of a slice (sequential), the CL slices
// (sequential): C_v = fl(P_s + fl(P_r + fl(Q_w + fl(E_{l-1} + part_k)))).
template <int DT, bool VEC, int NT>
__device__ __noinline__ int32_t cluster_sample(const char *trow, const char *drow, int64_t V, RowConst rc, float wu,
                                               SampleSmem<NT> &sm, float *Wt, int CL, int rank) {
  constexpr int NW = NT / 32;
  constexpr int B = (DT == 1) ? 4 : 2;  // rounds whose loads are in flight together
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t NG = (V + 7) / 8;
  const int64_t P = (NG + CL - 1) / CL;
  const int64_t gs = min(NG, static_cast<int64_t>(rank) * P), ge = min(NG, gs + P);
  const int nR = static_cast<int>((ge - gs + NT - 1) / NT);
  for (int attempt = 0; attempt < 2; ++attempt) {
    // ---- one pass over the slice: group sums, warp scans, warp totals ----
    if (tid == 0) sm.lastg = -1;
    int32_t lastg = -1;
    for (int r0 = 0; r0 < nR; r0 += B) {
      float ag[B];
      if (VEC && DT == 1) {
        // every load of the B rounds in flight before any arithmetic
        constexpr uint32_t ninf = 0xff80ff80u;
        uint4 ry[B], rz[B];
#pragma unroll
        for (int b = 0; b < B; ++b) {
          const int64_t g = gs + static_cast<int64_t>(r0 + b) * NT + tid;
          const bool in = (r0 + b < nR) && g < ge;
          ry[b] = in ? ld_vec(trow + g * 16) : make_uint4(ninf, ninf, ninf, ninf);
          rz[b] = (in && rc.resid) ? ld_vec(drow + g * 16) : make_uint4(ninf, ninf, ninf, ninf);
        }
        // log2 p and log2 q two entries at a time (f32x2); the weights and
        // the group's sum as sample_weight and sample_group form them
        const float2 k2 = make_float2(rc.k, rc.k), nT2 = make_float2(rc.nT, rc.nT), nD2 = make_float2(rc.nD, rc.nD);
#pragma unroll
        for (int b = 0; b < B; ++b) {
          const int64_t g = gs + static_cast<int64_t>(r0 + b) * NT + tid;
          const uint32_t wy[4] = {ry[b].x, ry[b].y, ry[b].z, ry[b].w};
          const uint32_t wz[4] = {rz[b].x, rz[b].y, rz[b].z, rz[b].w};
          float a = 0.f;
          if (rc.resid) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 lp = __ffma2_rn(bf16x2_f2(wy[h]), k2, nT2);
              const float2 lq = __ffma2_rn(bf16x2_f2(wz[h]), k2, nD2);
              a = __fadd_rn(a, resid_weight(lp.x, lq.x));
              a = __fadd_rn(a, resid_weight(lp.y, lq.y));
            }
          } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 lp = __ffma2_rn(bf16x2_f2(wy[h]), k2, nT2);
              a = __fadd_rn(a, ex2(lp.x));
              a = __fadd_rn(a, ex2(lp.y));
            }
          }
          ag[b] = a;
          if (a > 0.f) lastg = static_cast<int32_t>(g);
        }
      } else {
#pragma unroll
        for (int b = 0; b < B; ++b) {
          float w[8];
          const int64_t g = gs + static_cast<int64_t>(r0 + b) * NT + tid;
          ag[b] = (r0 + b < nR) ? sample_group<DT, VEC>(trow, drow, g, ge, V, rc, w) : 0.f;
          if (ag[b] > 0.f) lastg = static_cast<int32_t>(g);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float W = warp_scan_incl(ag[b]);
        if (lane == 31 && r0 + b < nR) Wt[(r0 + b) * NW + warp] = W;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastg = max(lastg, __shfl_xor_sync(0xffffffffu, lastg, o));
    __syncthreads();
    if (lane == 0) atomicMax(&sm.lastg, lastg);
    // round totals (sequential over warps), one round per thread
    for (int r = tid; r < nR; r += NT) {
      float R = 0.f;
      for (int w = 0; w < NW; ++w) R = __fadd_rn(R, Wt[r * NW + w]);
      sm.R[r] = R;
    }
    __syncthreads();
    // the slice total and last positive group, pushed to every CTA of the cluster
    if (warp == 0) {
      float Zs = 0.f;
      if (lane == 0)
        for (int r = 0; r < nR; ++r) Zs = __fadd_rn(Zs, sm.R[r]);
      Zs = __shfl_sync(0xffffffffu, Zs, 0);
      if (lane < CL) {
        st_cluster_b32(mapa_shared(smem_u32(&sm.Zs[rank]), lane), __float_as_uint(Zs));
        st_cluster_b32(mapa_shared(smem_u32(&sm.lg[rank]), lane), static_cast<uint32_t>(sm.lastg));
      }
    }
    cluster_barrier();
    if (tid == 0) {
      float Z = 0.f;
      for (int q = 0; q < CL; ++q) Z = __fadd_rn(Z, sm.Zs[q]);
      sm.degenerate = (rc.resid && !(Z > 0.f)) ? 1 : 0;
      const float t = __fmul_rn(wu, Z);
      // the crossing slice (the same in every CTA), then, in its owner, the round and warp
      int ss = -1, rs = -1, ws = -1;
      float Ps = 0.f, Pr = 0.f, Qw = 0.f, Pacc = 0.f;
      for (int q = 0; q < CL && ss < 0; ++q) {
        const float P2 = __fadd_rn(Pacc, sm.Zs[q]);
        if (P2 > t) {
          ss = q;
          Ps = Pacc;
        }
        Pacc = P2;
      }
      int spick = -1;  // the CTA that returns the token
      if (ss < 0) {
        // no crossing after rounding (w Z rounded up to Z): the last entry of
        // the row with positive weight, in the slice that holds it
        for (int q = 0; q < CL; ++q)
          if (sm.lg[q] >= 0) spick = q;
      } else {
        spick = ss;
      }
      if (ss == rank) {
        float Pq = Ps;
        for (int r = 0; r < nR && rs < 0; ++r) {
          const float P2 = __fadd_rn(Pq, sm.R[r]);
          if (P2 > t) {
            rs = r;
            Pr = Pq;
          }
          Pq = P2;
        }
        if (rs >= 0) {
          float Q = 0.f;
          for (int w = 0; w < NW && ws < 0; ++w) {
            const float Q2 = __fadd_rn(Q, Wt[rs * NW + w]);
            if (__fadd_rn(Pr, Q2) > t) {
              ws = w;
              Qw = Q;
            }
            Q = Q2;
          }
        }
      }
      sm.t = t;
      sm.rs = rs;
      sm.ws = ws;
      sm.Pr = Pr;
      sm.Qw = Qw;
      sm.spick = spick;
    }
    __syncthreads();
    if (sm.degenerate) {
      // no residual mass after rounding: draw from p at that row instead;
      // every peer has read this CTA's slice totals before they are rewritten
      rc.resid = false;
      cluster_barrier();
      continue;
    }
    if (sm.spick != rank) return -1;
    int32_t pick = -1;
    if (warp == 0) {
      const int rs = sm.rs, ws = sm.ws;
      const int64_t glast = sm.lastg;
      if (rs >= 0 && ws >= 0) {
        // lane and entry levels: lane l recomputes group l of the crossing warp
        const float t = sm.t, Pr = sm.Pr, Qw = sm.Qw;
        const int64_t g = gs + static_cast<int64_t>(rs) * NT + ws * 32 + lane;
        float w[8];
        const float ag = sample_group<DT, VEC>(trow, drow, g, ge, V, rc, w);
        const float E = warp_scan_incl(ag);
        const float Ex = __shfl_up_sync(0xffffffffu, E, 1);
        const float Eprev = (lane == 0) ? 0.f : Ex;
        const unsigned cross = __ballot_sync(0xffffffffu, __fadd_rn(Pr, __fadd_rn(Qw, E)) > t);
        if (cross) {
          const int l = __ffs(cross) - 1;
          if (lane == l) {
            float part = 0.f;
            int32_t lastpos = -1;
            for (int e = 0; e < 8; ++e) {
              part = __fadd_rn(part, w[e]);
              if (w[e] > 0.f) lastpos = static_cast<int32_t>(g * 8 + e);
              if (pick < 0 && __fadd_rn(Pr, __fadd_rn(Qw, __fadd_rn(Eprev, part))) > t)
                pick = static_cast<int32_t>(g * 8 + e);
            }
            if (pick < 0) pick = lastpos;  // rounding between the lane and entry levels
          }
          pick = __shfl_sync(0xffffffffu, pick, l);
        }
      }
      if (pick < 0 && glast >= 0 && lane == 0) {
        // no crossing inside the slice after rounding: its last entry with positive weight
        float w[8];
        sample_group<DT, VEC>(trow, drow, glast, ge, V, rc, w);
        for (int e = 0; e < 8; ++e)
          if (w[e] > 0.f) pick = static_cast<int32_t>(glast * 8 + e);
      }
      if (lane == 0) sm.rs = pick;
    }
    __syncthreads();
    return sm.rs;
  }
  return -1;  // not reached: p always has mass
}

}  // namespace svw
