// verify.cu -- batched speculative verification on sm_103a.
//
// Method ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.1, §5.2 eqs. (6)-(8),
// Algorithm 1; "AdaFlash: Taming Variance in Diffusion Speculative Decoding",
// "Speculative Decoding: The Basic Idea" steps 3-4):
//   accept x_j iff u_j < min(1, p_j(x_j)/q_j(x_j)); keep the leftmost-rejection
//   prefix; draw one token from [p - q]_+ at the rejected row or from p at the
//   bonus row.  Greedy (T = 0): accept iff x_j is the target argmax.
//
// GPU design.  The work is an HBM-bound stream over every logit row of the
// batch (sum_i (2 L_i + 1) rows of V, or L_i + 1 target rows when greedy).
//   * Each row is cut into C chunks (C <= 32, ~30 KB each); a (row, chunk)
//     pair is one work item.  Items are numbered request-major, so a
//     request's items are processed close together in time.
//   * A persistent grid (SMs x resident CTAs) walks the items.  A CTA loads its
//     chunk with 16-byte streaming loads (8 in flight per thread), reduces it
//     to (max, sum 2^((x - max) log2e / T)) -- or (max, argmax) when greedy --
//     and writes one Partial.
//   * A per-request arrival counter elects the CTA that finishes the request's
//     last item; that CTA (no waiting anywhere) merges the partials into row
//     log-sum-exps, evaluates every accept test in one warp (ballot + ffs gives
//     the leftmost rejection), and draws the next token with the block-wide
//     inverse-CDF sampler below while the request's rows are still in L2.
//
// Inverse-CDF sampler (one row, or one target/draft row pair).  Weights
// w_v = [p_v - q_v]_+ (or p_v).  The prefix sum C_v is defined hierarchically
// so that it is exactly reproducible and exactly monotone:
//   groups of 8 consecutive entries (sequential sum a_g), thread spans of GPT
//   consecutive groups (sequential running sum R), and the 256 span totals
//   (sequential exclusive prefix E_tau, computed by one thread);
//   C_v = fl(E_tau + fl(R_before_group + partial_k)).
// next = smallest v with C_v > w * Z (Z = E_256).  Every level is a
// sequential fp32 sum of non-negative terms, so C is non-decreasing and equal
// at every level boundary; the first crossing always has w_v > 0.
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace svw {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMinBlocks = 4;
constexpr int kUnroll = 8;               // 16-byte loads in flight per thread
constexpr int kMaxGroupsPerThread = 512;  // sampler span cap: V <= 256 * 512 * 8
constexpr int kMaxRows = 2 * SVW_MAX_LEN + 1;

struct Smem {
  float red_m[kWarps];
  float red_s[kWarps];
  int32_t red_i[kWarps];
  int32_t red_n[kWarps];
  int32_t last;
  // finalisation
  float row_m[kMaxRows];
  float row_l[kMaxRows];
  int32_t row_idx[kMaxRows];
  int32_t row_bad[kMaxRows];
  int32_t acc_len;
  int32_t bad;
  // sampler
  float span_tot[kThreads];
  float E[kThreads + 1];
  int32_t span_last[kThreads];
  float grp[kMaxGroupsPerThread];
  float Z;
  float t;
  int32_t tau_star;
  int32_t result;
  int32_t redo;
};

__device__ __forceinline__ Partial ldcg_partial(const Partial *p) {
  const float4 v = __ldcg(reinterpret_cast<const float4 *>(p));
  Partial r;
  r.m = v.x;
  r.s = v.y;
  r.idx = __float_as_int(v.z);
  r.nan = __float_as_int(v.w);
  return r;
}

// ---------------------------------------------------------------------------
// chunk reductions (the HBM stream)
// ---------------------------------------------------------------------------

// (max, sum 2^((x - max) k)) of elements [0, n) of a chunk, this thread's share
template <int DT, bool VEC>
__device__ __forceinline__ void chunk_lse(const char *p0, int64_t n, float k, float &m, float &s) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  m = -INFINITY;
  s = 0.f;
  if (VEC) {
    const int64_t nvec = n / EPV;  // whole vectors: V is a multiple of EPV on this path
    for (int64_t b = threadIdx.x; b < nvec; b += (int64_t)kUnroll * kThreads) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t vi = b + (int64_t)u * kThreads;
        if (vi < nvec) w[u] = ld_stream(p0 + vi * 16);
      }
      float mb = -INFINITY;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t vi = b + (int64_t)u * kThreads;
        if (vi < nvec) {
          float x[EPV];
          E::unpack(w[u], x);
#pragma unroll
          for (int e = 0; e < EPV; ++e) mb = fmaxf(mb, x[e]);
        }
      }
      const float mref = (mb == -INFINITY) ? 0.f : mb;
      float sb = 0.f;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t vi = b + (int64_t)u * kThreads;
        if (vi < nvec) {
          float x[EPV];
          E::unpack(w[u], x);
          float e[EPV];
#pragma unroll
          for (int q = 0; q < EPV; ++q) e[q] = ex2(__fmul_rn(__fsub_rn(x[q], mref), k));
          float v;
          if (EPV == 8)
            v = __fadd_rn(__fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3])),
                          __fadd_rn(__fadd_rn(e[4], e[5]), __fadd_rn(e[6], e[7])));
          else
            v = __fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3]));
          sb = __fadd_rn(sb, v);
        }
      }
      lse_combine(m, s, mb, sb, k);
    }
  } else {
    float mb = -INFINITY;
    for (int64_t v = threadIdx.x; v < n; v += kThreads) mb = fmaxf(mb, E::load(p0, v));
    const float mref = (mb == -INFINITY) ? 0.f : mb;
    float sb = 0.f;
    for (int64_t v = threadIdx.x; v < n; v += kThreads)
      sb = __fadd_rn(sb, ex2(__fmul_rn(__fsub_rn(E::load(p0, v), mref), k)));
    lse_combine(m, s, mb, sb, k);
  }
}

// (max, smallest argmax, any-NaN) of elements [0, n); v0 = chunk's first index
template <int DT, bool VEC>
__device__ __forceinline__ void chunk_amax(const char *p0, int64_t n, int64_t v0, float &best,
                                           int32_t &idx, int32_t &nan) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  best = -INFINITY;
  idx = INT32_MAX;
  nan = 0;
  auto visit = [&](float x, int64_t v) {
    nan |= (x != x);
    if (x > best || (idx == INT32_MAX && x == x)) {
      best = x;
      idx = static_cast<int32_t>(v);
    }
  };
  if (VEC) {
    const int64_t nvec = n / EPV;
    for (int64_t b = threadIdx.x; b < nvec; b += (int64_t)kUnroll * kThreads) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t vi = b + (int64_t)u * kThreads;
        if (vi < nvec) w[u] = ld_stream(p0 + vi * 16);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t vi = b + (int64_t)u * kThreads;
        if (vi < nvec) {
          float x[EPV];
          E::unpack(w[u], x);
#pragma unroll
          for (int e = 0; e < EPV; ++e) visit(x[e], v0 + vi * EPV + e);
        }
      }
    }
  } else {
    for (int64_t v = threadIdx.x; v < n; v += kThreads) visit(E::load(p0, v), v0 + v);
  }
}

// ---------------------------------------------------------------------------
// inverse-CDF sampler
// ---------------------------------------------------------------------------
struct RowConst {
  float Mt, lt, Md, ld, k;
};

// weight of one entry: [p - q]_+ (resid) or p, from raw logits
__device__ __forceinline__ float weight(float y, float z, bool resid, const RowConst &c) {
  const float lp = __fsub_rn(__fmul_rn(__fsub_rn(y, c.Mt), c.k), c.lt);  // log2 p
  if (!resid) return ex2(lp);
  const float lq = __fsub_rn(__fmul_rn(__fsub_rn(z, c.Md), c.k), c.ld);  // log2 q
  if (!(lq < lp)) return 0.f;
  return fmaxf(__fsub_rn(ex2(lp), ex2(lq)), 0.f);
}

// the 8 raw logits of group g (entries 8g .. 8g+7; -inf beyond V)
template <int DT, bool VEC>
__device__ __forceinline__ void load_group(const char *row, int64_t g, int64_t V, float (&x)[8]) {
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

// weights of group g and their sequential sum
template <int DT, bool VEC>
__device__ __forceinline__ float group_weights(const char *trow, const char *drow, bool resid,
                                               int64_t g, int64_t V, const RowConst &c,
                                               float (&w)[8]) {
  float y[8], z[8];
  load_group<DT, VEC>(trow, g, V, y);
  if (resid) load_group<DT, VEC>(drow, g, V, z);
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = weight(y[e], resid ? z[e] : 0.f, resid, c);
    a = __fadd_rn(a, w[e]);
  }
  return a;
}

// One token by inverse CDF; whole block participates; returns on all threads.
template <int DT, bool VEC>
__device__ __noinline__ int32_t sample_token(const char *trow, const char *drow, int64_t V, const RowConst &c,
                                float wu, Smem &sm) {
  const int tid = threadIdx.x;
  const int64_t NG = (V + 7) / 8;
  const int64_t GPT = (NG + kThreads - 1) / kThreads;
  bool resid = (drow != nullptr);
  for (int attempt = 0; attempt < 2; ++attempt) {
    // pass 1: span totals
    const int64_t g0 = (int64_t)tid * GPT, g1 = min(NG, g0 + GPT);
    float R = 0.f;
    int32_t last = -1;
    if (VEC) {
      using E = Elem<DT>;
      constexpr int EPV = E::kPerVec;
      constexpr int VPG = 8 / EPV;             // 16-byte vectors per group per tensor
      constexpr int GU = (DT == 1) ? 4 : 2;   // groups whose loads are in flight together
      for (int64_t g = g0; g < g1; g += GU) {
        uint4 ty[GU][VPG], tz[GU][VPG];
#pragma unroll
        for (int u = 0; u < GU; ++u)
#pragma unroll
          for (int h = 0; h < VPG; ++h) {
            const int64_t vv = (g + u) * 8 + h * EPV;
            if (g + u < g1 && vv < V) {
              ty[u][h] = ld_vec(trow + vv * E::kSize);
              if (resid) tz[u][h] = ld_vec(drow + vv * E::kSize);
            }
          }
#pragma unroll
        for (int u = 0; u < GU; ++u) {
          if (g + u < g1) {
            float y[8], z[8];
#pragma unroll
            for (int h = 0; h < VPG; ++h) {
              const int64_t vv = (g + u) * 8 + h * EPV;
              if (vv < V) {
                E::unpack(ty[u][h], y + h * EPV);
                if (resid) E::unpack(tz[u][h], z + h * EPV);
              } else {
#pragma unroll
                for (int e = 0; e < EPV; ++e) y[h * EPV + e] = z[h * EPV + e] = -INFINITY;
              }
            }
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float w = weight(y[e], resid ? z[e] : 0.f, resid, c);
              a = __fadd_rn(a, w);
              if (w > 0.f) last = static_cast<int32_t>((g + u) * 8 + e);
            }
            R = __fadd_rn(R, a);
          }
        }
      }
    } else {
      for (int64_t g = g0; g < g1; ++g) {
        float w[8];
        const float a = group_weights<DT, VEC>(trow, drow, resid, g, V, c, w);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (w[e] > 0.f) last = static_cast<int32_t>(g * 8 + e);
        R = __fadd_rn(R, a);
      }
    }
    sm.span_tot[tid] = R;
    sm.span_last[tid] = last;
    __syncthreads();
    if (tid == 0) {
      float E = 0.f;
      sm.E[0] = 0.f;
      for (int s = 0; s < kThreads; ++s) {
        E = __fadd_rn(E, sm.span_tot[s]);
        sm.E[s + 1] = E;
      }
      sm.Z = E;
      sm.redo = (resid && !(E > 0.f)) ? 1 : 0;  // no residual mass: fall back to p
      sm.t = __fmul_rn(wu, E);
      sm.tau_star = INT32_MAX;
    }
    __syncthreads();
    if (!sm.redo) break;
    resid = false;
    __syncthreads();
  }
  // first span whose end prefix exceeds t
  const float t = sm.t;
  if (sm.E[tid + 1] > t) atomicMin(&sm.tau_star, tid);
  __syncthreads();
  const int32_t ts = sm.tau_star;
  if (ts == INT32_MAX) {
    // t rounded up to Z: the last entry with positive weight
    if (tid == 0) {
      int32_t lastv = -1;
      for (int s = 0; s < kThreads; ++s) lastv = max(lastv, sm.span_last[s]);
      sm.result = lastv;
    }
    __syncthreads();
    return sm.result;
  }
  // pass 2: group sums of the crossing span (one group per thread, in parallel)
  const int64_t g0 = (int64_t)ts * GPT, g1 = min(NG, g0 + GPT);
  for (int64_t g = g0 + tid; g < g1; g += kThreads) {
    float w[8];
    sm.grp[g - g0] = group_weights<DT, VEC>(trow, drow, resid, g, V, c, w);
  }
  __syncthreads();
  if (tid == 0) {
    const float Es = sm.E[ts];
    float R = 0.f;
    int32_t pick = -1;
    for (int64_t g = g0; g < g1 && pick < 0; ++g) {
      const float R2 = __fadd_rn(R, sm.grp[g - g0]);
      if (__fadd_rn(Es, R2) > t) {
        float w[8];
        group_weights<DT, VEC>(trow, drow, resid, g, V, c, w);
        float part = 0.f;
        for (int e = 0; e < 8; ++e) {
          part = __fadd_rn(part, w[e]);
          if (__fadd_rn(Es, __fadd_rn(R, part)) > t) {
            pick = static_cast<int32_t>(g * 8 + e);
            break;
          }
        }
      }
      R = R2;
    }
    if (pick < 0) pick = sm.span_last[ts];  // unreachable by construction
    sm.result = pick;
  }
  __syncthreads();
  return sm.result;
}

// ---------------------------------------------------------------------------
// per-request finalisation (run by the CTA that completes the request)
// ---------------------------------------------------------------------------
template <int DT, bool VEC, bool GREEDY>
__device__ __noinline__ void finalize(const VerifyArgs &a, int32_t i, int64_t c_i, int32_t L, Smem &sm) {
  using E = Elem<DT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t0 = c_i + i, d0 = c_i;
  const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
  // merge chunk partials of each row (one warp per row, one lane per chunk)
  for (int r = warp; r < nrows; r += kWarps) {
    const int64_t prow = (r <= L) ? (t0 + r) : (a.rows_t + d0 + (r - L - 1));
    if (GREEDY) {
      float v = -INFINITY;
      int32_t idx = INT32_MAX, nan = 0;
      if (lane < a.C) {
        const Partial p = ldcg_partial(a.part + prow * a.C + lane);
        v = p.m;
        idx = p.idx;
        nan = p.nan;
      }
      warp_amax(v, idx);
      nan = __any_sync(0xffffffffu, nan);
      if (lane == 0) {
        sm.row_idx[r] = idx;
        sm.row_bad[r] = nan;
      }
    } else {
      float m = -INFINITY, s = 0.f;
      if (lane < a.C) {
        const Partial p = ldcg_partial(a.part + prow * a.C + lane);
        m = p.m;
        s = p.s;
      }
      warp_lse(m, s, a.k);
      if (lane == 0) {
        sm.row_m[r] = m;
        sm.row_l[r] = lg2(s);
        sm.row_bad[r] = !(s > 0.f && s <= FLT_MAX);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    int bad = 0;
    for (int r = lane; r < nrows; r += 32) bad |= sm.row_bad[r];
    bad = __any_sync(0xffffffffu, bad);
    bool acc = true;
    if (lane < L) {
      const int32_t x = __ldg(a.tokens + d0 + lane);
      if (GREEDY) {
        acc = (x == sm.row_idx[lane]);
      } else {
        // log2(p(x)/q(x)) from raw logits and row log-sum-exps
        const float yx = E::load(a.target, (t0 + lane) * a.V + x);
        const float zx = E::load(a.draft, (d0 + lane) * a.V + x);
        float thr;
        if (zx == -INFINITY) {
          thr = 1.f;  // q(x) = 0: accept
        } else {
          const float dl = __fsub_rn(
              __fmul_rn(__fsub_rn(__fsub_rn(yx, sm.row_m[lane]), __fsub_rn(zx, sm.row_m[L + 1 + lane])),
                        a.k),
              __fsub_rn(sm.row_l[lane], sm.row_l[L + 1 + lane]));
          thr = (dl >= 0.f) ? 1.f : ex2(dl);
        }
        const float u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(lane), 0u);
        acc = (u < thr);
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !acc);
    if (lane == 0) {
      sm.acc_len = rej ? (__ffs(rej) - 1) : L;
      sm.bad = bad;
    }
  }
  __syncthreads();
  if (sm.bad) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, SVW_DEV_BAD_INPUT);
    return;  // outputs keep the -1 written by the prologue
  }
  const int32_t js = sm.acc_len;
  int32_t tok;
  if (GREEDY) {
    tok = sm.row_idx[js];
  } else {
    RowConst c;
    c.Mt = sm.row_m[js];
    c.lt = sm.row_l[js];
    c.Md = (js < L) ? sm.row_m[L + 1 + js] : 0.f;
    c.ld = (js < L) ? sm.row_l[L + 1 + js] : 0.f;
    c.k = a.k;
    const float wu = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(js), 1u);
    const char *trow = static_cast<const char *>(a.target) + (t0 + js) * a.V * E::kSize;
    const char *drow =
        (js < L) ? static_cast<const char *>(a.draft) + (d0 + js) * a.V * E::kSize : nullptr;
    tok = sample_token<DT, VEC>(trow, drow, a.V, c, wu, sm);
  }
  if (threadIdx.x == 0) {
    a.accept_len[i] = js;
    a.next_token[i] = tok;
  }
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------

// Validates the CSR offsets and tokens, resets per-call state, writes the -1
// defaults.  One CTA; runs before the main kernel on the same stream.
__global__ void __launch_bounds__(1024) verify_prologue(VerifyArgs a) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int bad = 0;
  if (threadIdx.x == 0 &&
      (__ldg(a.cu) != 0 || static_cast<int64_t>(__ldg(a.cu + a.N)) != a.total_rows))
    bad |= 2;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const int32_t c0 = __ldg(a.cu + i), c1 = __ldg(a.cu + i + 1);
    const int32_t L = c1 - c0;
    if (L < 0) bad |= 2;
    bool ok = (L >= 1 && L <= a.max_len && c0 >= 0 && static_cast<int64_t>(c1) <= a.total_rows);
    if (ok)
      for (int j = 0; j < L; ++j) {
        const int32_t x = __ldg(a.tokens + c0 + j);
        if (x < 0 || static_cast<int64_t>(x) >= a.V) ok = false;
      }
    a.req_ok[i] = ok ? 1 : 0;
    a.counters[i] = 0;
    a.accept_len[i] = -1;
    a.next_token[i] = -1;
    if (!ok) bad |= 1;
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  if (threadIdx.x == 0) {
    *a.global_ok = (s_bad & 2) ? 0 : 1;
    if (s_bad && a.status) atomicOr(a.status, SVW_DEV_BAD_INPUT);
  }
}

template <bool GREEDY>
__device__ __forceinline__ int32_t find_request(const VerifyArgs &a, int64_t item) {
  int32_t lo = 0, hi = a.N - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    const int64_t cm = __ldg(a.cu + mid);
    const int64_t off = static_cast<int64_t>(a.C) * (GREEDY ? (cm + mid) : (2 * cm + mid));
    if (off <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int DT, bool VEC, bool GREEDY>
__global__ void __launch_bounds__(kThreads, kMinBlocks) verify_main(VerifyArgs a) {
  using E = Elem<DT>;
  __shared__ Smem sm;
  if (*a.global_ok == 0) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t item = blockIdx.x; item < a.total_items; item += gridDim.x) {
    const int32_t i = find_request<GREEDY>(a, item);
    const int64_t c_i = __ldg(a.cu + i);
    const int32_t L = __ldg(a.cu + i + 1) - static_cast<int32_t>(c_i);
    const int64_t off = static_cast<int64_t>(a.C) * (GREEDY ? (c_i + i) : (2 * c_i + i));
    const int64_t local = item - off;
    const int32_t rl = static_cast<int32_t>(local / a.C);
    const int32_t chunk = static_cast<int32_t>(local - static_cast<int64_t>(rl) * a.C);
    const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
    if (!a.req_ok[i] || rl >= nrows) continue;  // uniform across the block

    int64_t prow;
    const char *rowp;
    if (GREEDY || rl <= L) {
      const int64_t tr = c_i + i + rl;
      rowp = static_cast<const char *>(a.target) + tr * a.V * E::kSize;
      prow = tr;
    } else {
      const int64_t dr = c_i + (rl - L - 1);
      rowp = static_cast<const char *>(a.draft) + dr * a.V * E::kSize;
      prow = a.rows_t + dr;
    }
    const int64_t c0 = static_cast<int64_t>(chunk) * a.chunk_len;
    const int64_t n = min(static_cast<int64_t>(a.chunk_len), a.V - c0);
    const char *p0 = rowp + c0 * E::kSize;

    Partial res;
    if (GREEDY) {
      float v;
      int32_t idx, nan;
      chunk_amax<DT, VEC>(p0, n, c0, v, idx, nan);
      warp_amax(v, idx);
      nan = __any_sync(0xffffffffu, nan);
      if (lane == 0) {
        sm.red_m[warp] = v;
        sm.red_i[warp] = idx;
        sm.red_n[warp] = nan;
      }
      __syncthreads();
      if (warp == 0) {
        v = (lane < kWarps) ? sm.red_m[lane] : -INFINITY;
        idx = (lane < kWarps) ? sm.red_i[lane] : INT32_MAX;
        nan = (lane < kWarps) ? sm.red_n[lane] : 0;
        warp_amax(v, idx);
        nan = __any_sync(0xffffffffu, nan);
      }
      res.m = v;
      res.s = 0.f;
      res.idx = idx;
      res.nan = nan;
    } else {
      float m, s;
      chunk_lse<DT, VEC>(p0, n, a.k, m, s);
      warp_lse(m, s, a.k);
      if (lane == 0) {
        sm.red_m[warp] = m;
        sm.red_s[warp] = s;
      }
      __syncthreads();
      if (warp == 0) {
        m = (lane < kWarps) ? sm.red_m[lane] : -INFINITY;
        s = (lane < kWarps) ? sm.red_s[lane] : 0.f;
        warp_lse(m, s, a.k);
      }
      res.m = m;
      res.s = s;
      res.idx = 0;
      res.nan = 0;
    }
    if (threadIdx.x == 0) {
      a.part[prow * a.C + chunk] = res;
      __threadfence();
      const int32_t prev = atomicAdd(a.counters + i, 1);
      sm.last = (prev == a.C * nrows - 1) ? 1 : 0;
    }
    __syncthreads();
    if (sm.last) {
      __threadfence();
      finalize<DT, VEC, GREEDY>(a, i, c_i, L, sm);
    }
    __syncthreads();
  }
}

template <int DT, bool VEC, bool GREEDY>
cudaError_t launch_main(const VerifyArgs &a, cudaStream_t st) {
  static int grid_cache[128] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = (dev >= 0 && dev < 128) ? grid_cache[dev] : 0;
  if (grid == 0) {
    int nsm = 0, occ = 0;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, verify_main<DT, VEC, GREEDY>, kThreads, 0);
    if (e != cudaSuccess) return e;
    grid = nsm * (occ > 0 ? occ : 1);
    if (dev >= 0 && dev < 128) grid_cache[dev] = grid;
  }
  const int64_t blocks = a.total_items < grid ? a.total_items : grid;
  verify_main<DT, VEC, GREEDY><<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

ChunkPlan plan_chunks(int64_t V, int esize) {
  const int64_t target = (esize == 2) ? 16384 : 8192;
  int64_t C = (V + target - 1) / target;
  if (C < 1) C = 1;
  if (C > 32) C = 32;
  int64_t len = (V + C - 1) / C;
  len = (len + 7) / 8 * 8;
  C = (V + len - 1) / len;
  return ChunkPlan{static_cast<int32_t>(C), static_cast<int32_t>(len)};
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

VerifyLayout verify_layout(int32_t N, int64_t total_rows, int64_t V, int esize) {
  const ChunkPlan p = plan_chunks(V, esize);
  VerifyLayout l;
  const size_t rows = static_cast<size_t>(total_rows + N) + static_cast<size_t>(total_rows);
  l.part_off = 0;
  l.counters_off = align256(rows * static_cast<size_t>(p.C) * sizeof(Partial));
  l.req_ok_off = l.counters_off + align256(static_cast<size_t>(N) * 4);
  l.global_ok_off = l.req_ok_off + align256(static_cast<size_t>(N) * 4);
  l.total = l.global_ok_off + 256;
  return l;
}

cudaError_t launch_verify(const VerifyArgs &a, int dtype, bool vec, bool greedy, cudaStream_t st) {
  verify_prologue<<<1, 1024, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dtype == SVW_BF16) {
    if (vec) return greedy ? launch_main<1, true, true>(a, st) : launch_main<1, true, false>(a, st);
    return greedy ? launch_main<1, false, true>(a, st) : launch_main<1, false, false>(a, st);
  }
  if (vec) return greedy ? launch_main<0, true, true>(a, st) : launch_main<0, true, false>(a, st);
  return greedy ? launch_main<0, false, true>(a, st) : launch_main<0, false, false>(a, st);
}

}  // namespace svw
