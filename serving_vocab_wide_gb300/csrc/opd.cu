// opd.cu -- fused OPD loss forward + backward on sm_103a.
//
// Method ("AdaFlash: Taming Variance in Diffusion Speculative Decoding",
// "The Reverse-KL + Hard-Label Mixture Loss, Derived" and "Algorithm 2:
// Entry-Wise Clipped Reverse-KL"), per draft row paired with a target row:
//   t_v = q_v (lq_v - lp_v);  loss = sum_v clamp(t_v, -c, c) - lambda lq[x*]
//   dz_v = gs/T (q_v (a_v - S) + lambda (q_v - [v = x*])),
//   a_v = [-c < t_v < c] (lq_v - lp_v + 1),  S = sum_v q_v a_v.
// The gradient needs two row-wide reductions (the two log-sum-exps, then S)
// before any dz_v can be written, so the row stays on chip between them.
//
// GPU design.  A thread-block cluster of CL CTAs (CL <= 8) owns one row at a
// time; CTA r of the cluster holds vocabulary slice [r*SL, (r+1)*SL) of both
// the target and the draft row in shared memory (76 KB at V = 151936 bf16,
// so two CTAs of different clusters share an SM and overlap one's copies
// with the other's arithmetic).
//   * The slices arrive by 1-D bulk asynchronous copies (cp.async.bulk, one
//     per tensor per CTA, completion counted on an mbarrier): HBM sees each
//     logit byte once.
//   * Pass A: packed bf16 max, then sum of exp2 for both rows -> CTA partial
//     -> DSMEM exchange (barrier.cluster) -> every CTA merges the CL partials
//     in rank order, so all CTAs hold identical row constants.
//   * Pass B: clamped terms and S; the threads holding the row maximum look
//     up the first argmax index -> second exchange.
//   * Pass C: dz with 16-byte streaming stores.
// In log2 units: A = log2 q = z k - Cd, Bp = log2 p = y k - Ct, d2 = A - Bp,
// t/ln2 = q d2, q(d + 1) = t + q; the per-entry arithmetic runs on f32x2
// pairs.  Entries whose term is clipped, or undefined (q = 0 against an
// infinite log ratio, a term of 0), take a scalar slow path.
// Every wait on a bulk copy is bounded by a clock deadline; on expiry the CTA
// records SVW_DEV_TIMEOUT, stops issuing copies and keeps joining the cluster
// barriers so that no peer can hang.
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace cg = cooperative_groups;

namespace svw {

namespace {

constexpr int kMaxWarps = 32;
constexpr int kMaxCluster = 8;

struct OpdSmem {
  unsigned long long mbar[2];
  float red[kMaxWarps][4];
  int32_t redi[kMaxWarps];
  float partA[8];  // this CTA's mt, st, md, sd, abort
  float partB[4];  // this CTA's rkl (log2 units), S, argmax candidate (bits)
  float rowA[8];   // merged over the cluster: Mt, St, Md, Sd, any abort
  float rowB[4];   // merged over the cluster: rkl, S, argmax (bits)
  int64_t tr[2];   // target row of the row in each stage (-1: outside its request)
  int32_t abort;
};

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

// max over a 16-byte vector (packed bf16 pairs or 4 floats) folded into m
template <int DT>
__device__ __forceinline__ float vec_max(const uint4 &w, float m) {
  if (DT == 1) {
    const float2 f = bf16x2_f2(bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w)));
    return fmaxf(m, fmaxf(f.x, f.y));
  }
  return fmaxf(fmaxf(m, fmaxf(__uint_as_float(w.x), __uint_as_float(w.y))),
               fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
}

// the elements of a 16-byte vector as float pairs, in index order
template <int DT>
struct Pairs {
  static constexpr int kN = (DT == 1) ? 4 : 2;
  float2 p[kN];
  __device__ __forceinline__ explicit Pairs(const uint4 &w) {
    if (DT == 1) {
      p[0] = bf16x2_f2(w.x);
      p[1] = bf16x2_f2(w.y);
      p[2] = bf16x2_f2(w.z);
      p[3] = bf16x2_f2(w.w);
    } else {
      p[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
      p[kN - 1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
  }
};

// one entry's contribution when its term is clipped or undefined (rare):
// NaN arises only from q = 0 against an infinite log ratio, whose term is 0
__device__ __forceinline__ void term_slow(float t2, float q, float c2, float &rkl2, float &S) {
  if (t2 != t2) return;
  if (fabsf(t2) < c2) {
    rkl2 += t2;
    S += fmaf(t2, kLn2, q);
  } else {
    rkl2 += (t2 > 0.f) ? c2 : -c2;
  }
}

// NT threads per CTA; STAGES = 1: one slice buffer, two CTAs per SM overlap
// each other's copies; STAGES = 2: the next row's slices are prefetched into
// the second buffer while the current row is processed (one CTA per SM).
template <int DT, bool BULK, int NT, int STAGES>
__global__ void __launch_bounds__(NT, (STAGES == 1 ? 2 : 1)) opd_kernel(OpdArgs a, int32_t SL, int32_t slice_bytes) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int kThreads = NT;
  constexpr int kWarps = NT / 32;
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
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(SL), V - lo)));
  const int nvec = n / EPV;  // whole 16-byte vectors (the bulk path has no tail)
  const float k = a.k;

  if (tid == 0) {
    mbar_init(&sm.mbar[0], 1);
    mbar_init(&sm.mbar[1], 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // thread 0: start the bulk copies of row r's slices into stage s
  auto issue = [&](int64_t r, int s) {
    const int64_t t = target_row_of(a, r);
    sm.tr[s] = t;
    unsigned char *tb = dyn + static_cast<size_t>(s) * 2 * slice_bytes;
    const uint32_t bytes = static_cast<uint32_t>(n) * E::kSize;
    if (!sm.abort && t >= 0 && bytes > 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&sm.mbar[s], 2 * bytes);
      bulk_g2s(tb, static_cast<const char *>(a.target) + (t * V + lo) * E::kSize, bytes, &sm.mbar[s]);
      bulk_g2s(tb + slice_bytes, static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize, bytes,
               &sm.mbar[s]);
    } else {
      mbar_arrive(&sm.mbar[s]);
    }
  };
  int pf_stage = -1;  // thread 0: stage of a prefetch still in flight
  uint32_t pf_parity = 0;
  if (BULK && STAGES == 2 && tid == 0 && cid < a.R) issue(cid, 0);

  for (int64_t r = cid, it = 0; r < a.R; r += nclusters, ++it) {
    const int s = (STAGES == 2) ? static_cast<int>(it & 1) : 0;
    const uint32_t parity = static_cast<uint32_t>(((STAGES == 2) ? (it >> 1) : it) & 1);
    unsigned char *tbuf = dyn + static_cast<size_t>(s) * 2 * slice_bytes;
    unsigned char *dbuf = tbuf + slice_bytes;
    const uint32_t tb = smem_u32(tbuf), db = smem_u32(dbuf);
    // ---- fill the slices ----
    if (BULK) {
      if (tid == 0) {
        if (STAGES == 2) {
          pf_stage = -1;
          if (r + nclusters < a.R) {
            issue(r + nclusters, s ^ 1);
            pf_stage = s ^ 1;
            pf_parity = static_cast<uint32_t>(((it + 1) >> 1) & 1);
          }
        } else {
          issue(r, 0);
        }
      }
      if (!sm.abort && !mbar_wait_bounded(&sm.mbar[s], parity)) {
        if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        sm.abort = 1;
      }
      __syncthreads();
    } else {
      if (tid == 0) sm.tr[s] = target_row_of(a, r);
      __syncthreads();
      const int64_t t = sm.tr[s];
      if (t >= 0) {
        const char *ts = static_cast<const char *>(a.target) + (t * V + lo) * E::kSize;
        const char *ds = static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize;
        for (int v = tid; v < n; v += kThreads) {
          if (DT == 1) {
            reinterpret_cast<unsigned short *>(tbuf)[v] = __ldg(reinterpret_cast<const unsigned short *>(ts) + v);
            reinterpret_cast<unsigned short *>(dbuf)[v] = __ldg(reinterpret_cast<const unsigned short *>(ds) + v);
          } else {
            reinterpret_cast<float *>(tbuf)[v] = __ldg(reinterpret_cast<const float *>(ts) + v);
            reinterpret_cast<float *>(dbuf)[v] = __ldg(reinterpret_cast<const float *>(ds) + v);
          }
        }
      }
      __syncthreads();
    }
    const bool valid = (sm.tr[s] >= 0);
    const bool work = valid && !sm.abort;

    // ---------------- pass A: maxima, then sums of exp2 ----------------
    float mt = -INFINITY, md = -INFINITY, st = 0.f, sd = 0.f;
    if (work) {
      for (int vi = tid; vi < nvec; vi += kThreads) {
        mt = vec_max<DT>(lds128(tb + vi * 16), mt);
        md = vec_max<DT>(lds128(db + vi * 16), md);
      }
      if (!BULK && tid == 0)
        for (int v = nvec * EPV; v < n; ++v) {
          mt = fmaxf(mt, E::load_plain(tbuf, v));
          md = fmaxf(md, E::load_plain(dbuf, v));
        }
      const float nmt = (mt == -INFINITY) ? 0.f : -mt * k;
      const float nmd = (md == -INFINITY) ? 0.f : -md * k;
      const float2 kk = make_float2(k, k), nt2 = make_float2(nmt, nmt), nd2 = make_float2(nmd, nmd);
      float2 at = make_float2(0.f, 0.f), ad = make_float2(0.f, 0.f);
      for (int vi = tid; vi < nvec; vi += kThreads) {
        const Pairs<DT> y(lds128(tb + vi * 16)), z(lds128(db + vi * 16));
#pragma unroll
        for (int h = 0; h < Pairs<DT>::kN; ++h) {
          const float2 ey = __ffma2_rn(y.p[h], kk, nt2);
          const float2 ez = __ffma2_rn(z.p[h], kk, nd2);
          at = __fadd2_rn(at, make_float2(ex2(ey.x), ex2(ey.y)));
          ad = __fadd2_rn(ad, make_float2(ex2(ez.x), ex2(ez.y)));
        }
      }
      st = at.x + at.y;
      sd = ad.x + ad.y;
      if (!BULK && tid == 0)
        for (int v = nvec * EPV; v < n; ++v) {
          st += ex2(fmaf(E::load_plain(tbuf, v), k, nmt));
          sd += ex2(fmaf(E::load_plain(dbuf, v), k, nmd));
        }
    }
    const float my_mt = mt;  // this thread's target maximum (argmax lookup below)
    warp_lse(mt, st, k);
    warp_lse(md, sd, k);
    if (lane == 0) {
      sm.red[warp][0] = mt;
      sm.red[warp][1] = st;
      sm.red[warp][2] = md;
      sm.red[warp][3] = sd;
    }
    __syncthreads();
    if (warp == 0) {
      float a0 = -INFINITY, a1 = 0.f, a2 = -INFINITY, a3 = 0.f;
      if (lane < kWarps) {
        a0 = sm.red[lane][0];
        a1 = sm.red[lane][1];
        a2 = sm.red[lane][2];
        a3 = sm.red[lane][3];
      }
      warp_lse(a0, a1, k);
      warp_lse(a2, a3, k);
      if (lane == 0) {
        sm.partA[0] = a0;
        sm.partA[1] = a1;
        sm.partA[2] = a2;
        sm.partA[3] = a3;
        sm.partA[4] = sm.abort ? 1.f : 0.f;
      }
    }
    cluster.sync();
    // one warp gathers the CL partials (lane q <- rank q) and merges them in
    // rank order; every CTA computes the same constants
    if (warp == 0) {
      float v0 = -INFINITY, v1 = 0.f, v2 = -INFINITY, v3 = 0.f, v4 = 0.f;
      if (lane < CL) {
        const float *pa = cluster.map_shared_rank(sm.partA, lane);
        v0 = pa[0];
        v1 = pa[1];
        v2 = pa[2];
        v3 = pa[3];
        v4 = pa[4];
      }
      float M0 = -INFINITY, S0 = 0.f, M1 = -INFINITY, S1 = 0.f, ab = 0.f;
      for (int q = 0; q < CL; ++q) {
        lse_combine(M0, S0, __shfl_sync(0xffffffffu, v0, q), __shfl_sync(0xffffffffu, v1, q), k);
        lse_combine(M1, S1, __shfl_sync(0xffffffffu, v2, q), __shfl_sync(0xffffffffu, v3, q), k);
        ab += __shfl_sync(0xffffffffu, v4, q);
      }
      if (lane == 0) {
        sm.rowA[0] = M0;
        sm.rowA[1] = S0;
        sm.rowA[2] = M1;
        sm.rowA[3] = S1;
        sm.rowA[4] = ab;
      }
    }
    __syncthreads();
    const float Mt = sm.rowA[0], St = sm.rowA[1], Md = sm.rowA[2], Sd = sm.rowA[3];
    const bool any_abort = sm.rowA[4] != 0.f;
    const bool row_ok = valid && !any_abort && (St > 0.f && St <= FLT_MAX) && (Sd > 0.f && Sd <= FLT_MAX);
    const float Ct = fmaf(Mt, k, lg2(St));  // log2 p = y k - Ct
    const float Cd = fmaf(Md, k, lg2(Sd));  // log2 q = z k - Cd
    const float c2 = a.clip_c * kLog2e;     // clip bound in log2 units of t
    float rkl = 0.f, S = 0.f;
    int32_t cand = INT32_MAX;

    // ---------------- pass B: clamped terms, S, argmax ----------------
    if (row_ok) {
      const float2 kk = make_float2(k, k), nkk = make_float2(-k, -k);
      const float2 nCd = make_float2(-Cd, -Cd), Ct2 = make_float2(Ct, Ct), l2 = make_float2(kLn2, kLn2);
      float2 r2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
      for (int vi = tid; vi < nvec; vi += kThreads) {
        const Pairs<DT> y(lds128(tb + vi * 16)), z(lds128(db + vi * 16));
#pragma unroll
        for (int h = 0; h < Pairs<DT>::kN; ++h) {
          const float2 A = __ffma2_rn(z.p[h], kk, nCd);    // log2 q
          const float2 q = make_float2(ex2(A.x), ex2(A.y));
          const float2 d = __fadd2_rn(A, __ffma2_rn(y.p[h], nkk, Ct2));  // log2 q - log2 p
          const float2 t = __fmul2_rn(q, d);               // t / ln 2
          if (fabsf(t.x) < c2 && fabsf(t.y) < c2) {
            r2 = __fadd2_rn(r2, t);
            s2 = __fadd2_rn(__ffma2_rn(t, l2, s2), q);
          } else {
            term_slow(t.x, q.x, c2, r2.x, s2.x);
            term_slow(t.y, q.y, c2, r2.y, s2.y);
          }
        }
      }
      rkl = r2.x + r2.y;
      S = s2.x + s2.y;
      if (!BULK && tid == 0)
        for (int v = nvec * EPV; v < n; ++v) {
          const float y = E::load_plain(tbuf, v), z = E::load_plain(dbuf, v);
          const float A = fmaf(z, k, -Cd);
          const float q = ex2(A);
          term_slow(q * (A - fmaf(y, k, -Ct)), q, c2, rkl, S);
        }
      // first index holding the row maximum (only threads that saw it look)
      if (my_mt == Mt) {
        for (int vi = tid; vi < nvec && cand == INT32_MAX; vi += kThreads) {
          float y[EPV];
          E::unpack(lds128(tb + vi * 16), y);
          for (int e = 0; e < EPV; ++e)
            if (y[e] == Mt) {
              cand = static_cast<int32_t>(lo + vi * EPV + e);
              break;
            }
        }
        if (!BULK && tid == 0 && cand == INT32_MAX)
          for (int v = nvec * EPV; v < n; ++v)
            if (E::load_plain(tbuf, v) == Mt) {
              cand = static_cast<int32_t>(lo + v);
              break;
            }
      }
    }
    rkl = warp_sum(rkl);
    S = warp_sum(S);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    if (lane == 0) {
      sm.red[warp][0] = rkl;
      sm.red[warp][1] = S;
      sm.redi[warp] = cand;
    }
    __syncthreads();
    if (warp == 0) {
      float r1 = (lane < kWarps) ? sm.red[lane][0] : 0.f;
      float s1 = (lane < kWarps) ? sm.red[lane][1] : 0.f;
      int32_t c1 = (lane < kWarps) ? sm.redi[lane] : INT32_MAX;
      r1 = warp_sum(r1);
      s1 = warp_sum(s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c1 = min(c1, __shfl_xor_sync(0xffffffffu, c1, o));
      if (lane == 0) {
        sm.partB[0] = r1;
        sm.partB[1] = s1;
        sm.partB[2] = __int_as_float(c1);
      }
    }
    cluster.sync();
    if (warp == 0) {
      float v0 = 0.f, v1 = 0.f;
      int32_t v2 = INT32_MAX;
      if (lane < CL) {
        const float *pb = cluster.map_shared_rank(sm.partB, lane);
        v0 = pb[0];
        v1 = pb[1];
        v2 = __float_as_int(pb[2]);
      }
      float R0 = 0.f, S0 = 0.f;
      int32_t X = INT32_MAX;
      for (int q = 0; q < CL; ++q) {
        R0 += __shfl_sync(0xffffffffu, v0, q);
        S0 += __shfl_sync(0xffffffffu, v1, q);
        X = min(X, __shfl_sync(0xffffffffu, v2, q));
      }
      if (lane == 0) {
        sm.rowB[0] = R0;
        sm.rowB[1] = S0;
        sm.rowB[2] = __int_as_float(X);
      }
    }
    __syncthreads();
    const float RKL2 = sm.rowB[0], SS = sm.rowB[1];
    const int32_t xs = __float_as_int(sm.rowB[2]);
    if (rank == 0 && tid == 0) {
      float out = __int_as_float(0x7fffffff);
      if (row_ok && xs != INT32_MAX) {
        const float zx = E::load(a.draft, r * V + xs);
        // loss = sum clamp(t) + lambda * (-lq[x*]);  t = ln2 * t2, lq = ln2 * A
        out = kLn2 * (RKL2 - a.lambda_ce * fmaf(zx, k, -Cd));
      } else if (a.status && !any_abort) {
        atomicOr(a.status, SVW_DEV_BAD_INPUT);
      }
      a.loss[r] = out;
    }

    // ---------------- pass C: gradient wrt the draft logits ----------------
    // dz = gsT (qa + q (lambda - S)) - gsT lambda [v = x*], qa = t + q when
    // |t| < c else 0; in log2 units dz = t2 gsT ln2 + q gsT (lambda - S + 1).
    if (a.dlogits != nullptr && valid && !any_abort) {
      const float gsT = a.grad_scale * a.invT;
      const float gL0 = gsT * (a.lambda_ce - SS);
      const float gL1 = gsT * (a.lambda_ce - SS + 1.f);
      const float nan = __int_as_float(0x7fffffff);
      float *out = a.dlogits + r * V + lo;
      if (BULK) {
        const float2 kk = make_float2(k, k), nkk = make_float2(-k, -k);
        const float2 nCd = make_float2(-Cd, -Cd), Ct2 = make_float2(Ct, Ct);
        const float2 gl = make_float2(gsT * kLn2, gsT * kLn2), g1 = make_float2(gL1, gL1);
        for (int vi = tid; vi < nvec; vi += kThreads) {
          const Pairs<DT> y(lds128(tb + vi * 16)), z(lds128(db + vi * 16));
          float g[EPV];
#pragma unroll
          for (int h = 0; h < Pairs<DT>::kN; ++h) {
            const float2 A = __ffma2_rn(z.p[h], kk, nCd);
            const float2 q = make_float2(ex2(A.x), ex2(A.y));
            const float2 t = __fmul2_rn(q, __fadd2_rn(A, __ffma2_rn(y.p[h], nkk, Ct2)));
            float2 gg = __ffma2_rn(t, gl, __fmul2_rn(q, g1));
            if (!(fabsf(t.x) < c2 && fabsf(t.y) < c2)) {
              if (!(fabsf(t.x) < c2)) gg.x = q.x * gL0;
              if (!(fabsf(t.y) < c2)) gg.y = q.y * gL0;
            }
            g[2 * h] = gg.x;
            g[2 * h + 1] = gg.y;
          }
          const int off = static_cast<int>(xs - (lo + vi * EPV));
          if (off >= 0 && off < EPV) {
#pragma unroll
            for (int e = 0; e < EPV; ++e)
              if (e == off) g[e] -= gsT * a.lambda_ce;
          }
          if (!row_ok) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) g[e] = nan;
          }
#pragma unroll
          for (int h = 0; h < EPV / 4; ++h)
            st_stream(out + vi * EPV + 4 * h, g[4 * h], g[4 * h + 1], g[4 * h + 2], g[4 * h + 3]);
        }
      } else {
        for (int v = tid; v < n; v += kThreads) {
          const float y = E::load_plain(tbuf, v), z = E::load_plain(dbuf, v);
          const float A = fmaf(z, k, -Cd);
          const float q = ex2(A);
          const float t = q * (A - fmaf(y, k, -Ct));
          float g = (fabsf(t) < c2) ? fmaf(t, gsT * kLn2, q * gL1) : q * gL0;
          if (lo + v == xs) g -= gsT * a.lambda_ce;
          out[v] = row_ok ? g : nan;
        }
      }
    }
    __syncthreads();  // the slices are fully consumed before the next copy
  }
  if (BULK && STAGES == 2 && tid == 0 && sm.abort && pf_stage >= 0)
    mbar_wait_bounded(&sm.mbar[pf_stage], pf_parity);  // let a copy still in flight land
  cluster.sync();  // peers may still read this CTA's partials
}

// Register-resident variant (16-byte-pitched rows).  Each thread owns the
// 16-byte vectors tid + j*NT (j < VPT) of both slices: as soon as a row's bulk
// copies land, every thread moves its vectors from shared memory into
// registers and the buffer is handed straight back to the next row's copies,
// so the next row streams in while this row's three passes run from registers.
template <int DT, int NT, int VPT>
__global__ void __launch_bounds__(NT, 2) opd_reg_kernel(OpdArgs a, int32_t SL, int32_t slice_bytes) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int kWarps = NT / 32;
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
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(SL), V - lo)));
  const int nvec = n / EPV;  // V is a multiple of EPV on this path: no tail
  const int nj = (tid < nvec) ? min(VPT, (nvec - tid + NT - 1) / NT) : 0;  // my vectors
  const float k = a.k;
  unsigned char *tbuf = dyn;
  unsigned char *dbuf = dyn + slice_bytes;
  const uint32_t tb = smem_u32(tbuf), db = smem_u32(dbuf);

  if (tid == 0) {
    mbar_init(&sm.mbar[0], 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](int64_t r) {
    const int64_t t = target_row_of(a, r);
    sm.tr[0] = t;
    const uint32_t bytes = static_cast<uint32_t>(n) * E::kSize;
    if (!sm.abort && t >= 0 && bytes > 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&sm.mbar[0], 2 * bytes);
      bulk_g2s(tbuf, static_cast<const char *>(a.target) + (t * V + lo) * E::kSize, bytes, &sm.mbar[0]);
      bulk_g2s(dbuf, static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize, bytes, &sm.mbar[0]);
    } else {
      mbar_arrive(&sm.mbar[0]);
    }
  };
  if (tid == 0 && cid < a.R) issue(cid);
  bool issued_next = false;  // thread 0: a copy for a later row is in flight

  for (int64_t r = cid, it = 0; r < a.R; r += nclusters, ++it) {
    if (!sm.abort && !mbar_wait_bounded(&sm.mbar[0], static_cast<uint32_t>(it & 1))) {
      if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
      sm.abort = 1;
    }
    const bool valid = (sm.tr[0] >= 0);
    uint4 ty[VPT], tz[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
      if (j < nj) {
        ty[j] = lds128(tb + (tid + j * NT) * 16);
        tz[j] = lds128(db + (tid + j * NT) * 16);
      }
    __syncthreads();  // the buffer is free: stream the next row in
    if (tid == 0) {
      issued_next = false;
      if (r + nclusters < a.R) {
        issue(r + nclusters);
        issued_next = true;
      }
    }
    const bool work = valid && !sm.abort;

    // ---------------- pass A: maxima, then sums of exp2 ----------------
    float mt = -INFINITY, md = -INFINITY, st = 0.f, sd = 0.f;
    if (work) {
#pragma unroll
      for (int j = 0; j < VPT; ++j)
        if (j < nj) {
          mt = vec_max<DT>(ty[j], mt);
          md = vec_max<DT>(tz[j], md);
        }
      const float nmt = (mt == -INFINITY) ? 0.f : -mt * k;
      const float nmd = (md == -INFINITY) ? 0.f : -md * k;
      const float2 kk = make_float2(k, k), nt2 = make_float2(nmt, nmt), nd2 = make_float2(nmd, nmd);
      float2 at = make_float2(0.f, 0.f), ad = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < VPT; ++j)
        if (j < nj) {
          const Pairs<DT> y(ty[j]), z(tz[j]);
#pragma unroll
          for (int h = 0; h < Pairs<DT>::kN; ++h) {
            const float2 ey = __ffma2_rn(y.p[h], kk, nt2);
            const float2 ez = __ffma2_rn(z.p[h], kk, nd2);
            at = __fadd2_rn(at, make_float2(ex2(ey.x), ex2(ey.y)));
            ad = __fadd2_rn(ad, make_float2(ex2(ez.x), ex2(ez.y)));
          }
        }
      st = at.x + at.y;
      sd = ad.x + ad.y;
    }
    const float my_mt = mt;
    warp_lse(mt, st, k);
    warp_lse(md, sd, k);
    if (lane == 0) {
      sm.red[warp][0] = mt;
      sm.red[warp][1] = st;
      sm.red[warp][2] = md;
      sm.red[warp][3] = sd;
    }
    __syncthreads();
    if (warp == 0) {
      float a0 = -INFINITY, a1 = 0.f, a2 = -INFINITY, a3 = 0.f;
      if (lane < kWarps) {
        a0 = sm.red[lane][0];
        a1 = sm.red[lane][1];
        a2 = sm.red[lane][2];
        a3 = sm.red[lane][3];
      }
      warp_lse(a0, a1, k);
      warp_lse(a2, a3, k);
      if (lane == 0) {
        sm.partA[0] = a0;
        sm.partA[1] = a1;
        sm.partA[2] = a2;
        sm.partA[3] = a3;
        sm.partA[4] = sm.abort ? 1.f : 0.f;
      }
    }
    cluster.sync();
    if (warp == 0) {
      float v0 = -INFINITY, v1 = 0.f, v2 = -INFINITY, v3 = 0.f, v4 = 0.f;
      if (lane < CL) {
        const float *pa = cluster.map_shared_rank(sm.partA, lane);
        v0 = pa[0];
        v1 = pa[1];
        v2 = pa[2];
        v3 = pa[3];
        v4 = pa[4];
      }
      float M0 = -INFINITY, S0 = 0.f, M1 = -INFINITY, S1 = 0.f, ab = 0.f;
      for (int q = 0; q < CL; ++q) {
        lse_combine(M0, S0, __shfl_sync(0xffffffffu, v0, q), __shfl_sync(0xffffffffu, v1, q), k);
        lse_combine(M1, S1, __shfl_sync(0xffffffffu, v2, q), __shfl_sync(0xffffffffu, v3, q), k);
        ab += __shfl_sync(0xffffffffu, v4, q);
      }
      if (lane == 0) {
        sm.rowA[0] = M0;
        sm.rowA[1] = S0;
        sm.rowA[2] = M1;
        sm.rowA[3] = S1;
        sm.rowA[4] = ab;
      }
    }
    __syncthreads();
    const float Mt = sm.rowA[0], St = sm.rowA[1], Md = sm.rowA[2], Sd = sm.rowA[3];
    const bool any_abort = sm.rowA[4] != 0.f;
    const bool row_ok = valid && !any_abort && (St > 0.f && St <= FLT_MAX) && (Sd > 0.f && Sd <= FLT_MAX);
    const float Ct = fmaf(Mt, k, lg2(St));  // log2 p = y k - Ct
    const float Cd = fmaf(Md, k, lg2(Sd));  // log2 q = z k - Cd
    const float c2 = a.clip_c * kLog2e;     // clip bound in log2 units of t
    float rkl = 0.f, S = 0.f;
    int32_t cand = INT32_MAX;

    // ---------------- pass B: clamped terms, S, argmax ----------------
    if (row_ok) {
      const float2 kk = make_float2(k, k), nkk = make_float2(-k, -k);
      const float2 nCd = make_float2(-Cd, -Cd), Ct2 = make_float2(Ct, Ct), l2 = make_float2(kLn2, kLn2);
      float2 r2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < VPT; ++j)
        if (j < nj) {
          const Pairs<DT> y(ty[j]), z(tz[j]);
#pragma unroll
          for (int h = 0; h < Pairs<DT>::kN; ++h) {
            const float2 A = __ffma2_rn(z.p[h], kk, nCd);                    // log2 q
            const float2 q = make_float2(ex2(A.x), ex2(A.y));
            const float2 d = __fadd2_rn(A, __ffma2_rn(y.p[h], nkk, Ct2));  // log2 q - log2 p
            const float2 t = __fmul2_rn(q, d);                               // t / ln 2
            if (fabsf(t.x) < c2 && fabsf(t.y) < c2) {
              r2 = __fadd2_rn(r2, t);
              s2 = __fadd2_rn(__ffma2_rn(t, l2, s2), q);
            } else {
              term_slow(t.x, q.x, c2, r2.x, s2.x);
              term_slow(t.y, q.y, c2, r2.y, s2.y);
            }
          }
        }
      rkl = r2.x + r2.y;
      S = s2.x + s2.y;
      if (my_mt == Mt) {  // first index holding the row maximum
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j < nj && cand == INT32_MAX) {
            float y[EPV];
            E::unpack(ty[j], y);
#pragma unroll
            for (int e = 0; e < EPV; ++e)
              if (cand == INT32_MAX && y[e] == Mt) cand = static_cast<int32_t>(lo + (tid + j * NT) * EPV + e);
          }
      }
    }
    rkl = warp_sum(rkl);
    S = warp_sum(S);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    if (lane == 0) {
      sm.red[warp][0] = rkl;
      sm.red[warp][1] = S;
      sm.redi[warp] = cand;
    }
    __syncthreads();
    if (warp == 0) {
      float r1 = (lane < kWarps) ? sm.red[lane][0] : 0.f;
      float s1 = (lane < kWarps) ? sm.red[lane][1] : 0.f;
      int32_t c1 = (lane < kWarps) ? sm.redi[lane] : INT32_MAX;
      r1 = warp_sum(r1);
      s1 = warp_sum(s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c1 = min(c1, __shfl_xor_sync(0xffffffffu, c1, o));
      if (lane == 0) {
        sm.partB[0] = r1;
        sm.partB[1] = s1;
        sm.partB[2] = __int_as_float(c1);
      }
    }
    cluster.sync();
    if (warp == 0) {
      float v0 = 0.f, v1 = 0.f;
      int32_t v2 = INT32_MAX;
      if (lane < CL) {
        const float *pb = cluster.map_shared_rank(sm.partB, lane);
        v0 = pb[0];
        v1 = pb[1];
        v2 = __float_as_int(pb[2]);
      }
      float R0 = 0.f, S0 = 0.f;
      int32_t X = INT32_MAX;
      for (int q = 0; q < CL; ++q) {
        R0 += __shfl_sync(0xffffffffu, v0, q);
        S0 += __shfl_sync(0xffffffffu, v1, q);
        X = min(X, __shfl_sync(0xffffffffu, v2, q));
      }
      if (lane == 0) {
        sm.rowB[0] = R0;
        sm.rowB[1] = S0;
        sm.rowB[2] = __int_as_float(X);
      }
    }
    __syncthreads();
    const float RKL2 = sm.rowB[0], SS = sm.rowB[1];
    const int32_t xs = __float_as_int(sm.rowB[2]);
    if (rank == 0 && tid == 0) {
      float out = __int_as_float(0x7fffffff);
      if (row_ok && xs != INT32_MAX) {
        const float zx = E::load(a.draft, r * V + xs);
        out = kLn2 * (RKL2 - a.lambda_ce * fmaf(zx, k, -Cd));
      } else if (a.status && !any_abort) {
        atomicOr(a.status, SVW_DEV_BAD_INPUT);
      }
      a.loss[r] = out;
    }

    // ---------------- pass C: gradient wrt the draft logits ----------------
    if (a.dlogits != nullptr && valid && !any_abort) {
      const float gsT = a.grad_scale * a.invT;
      const float gL0 = gsT * (a.lambda_ce - SS);
      const float gL1 = gsT * (a.lambda_ce - SS + 1.f);
      const float nan = __int_as_float(0x7fffffff);
      float *out = a.dlogits + r * V + lo;
      const float2 kk = make_float2(k, k), nkk = make_float2(-k, -k);
      const float2 nCd = make_float2(-Cd, -Cd), Ct2 = make_float2(Ct, Ct);
      const float2 gl = make_float2(gsT * kLn2, gsT * kLn2), g1 = make_float2(gL1, gL1);
#pragma unroll
      for (int j = 0; j < VPT; ++j)
        if (j < nj) {
          const int vi = tid + j * NT;
          const Pairs<DT> y(ty[j]), z(tz[j]);
          float g[EPV];
#pragma unroll
          for (int h = 0; h < Pairs<DT>::kN; ++h) {
            const float2 A = __ffma2_rn(z.p[h], kk, nCd);
            const float2 q = make_float2(ex2(A.x), ex2(A.y));
            const float2 t = __fmul2_rn(q, __fadd2_rn(A, __ffma2_rn(y.p[h], nkk, Ct2)));
            float2 gg = __ffma2_rn(t, gl, __fmul2_rn(q, g1));
            if (!(fabsf(t.x) < c2 && fabsf(t.y) < c2)) {
              if (!(fabsf(t.x) < c2)) gg.x = q.x * gL0;
              if (!(fabsf(t.y) < c2)) gg.y = q.y * gL0;
            }
            g[2 * h] = gg.x;
            g[2 * h + 1] = gg.y;
          }
          const int off = static_cast<int>(xs - (lo + vi * EPV));
          if (off >= 0 && off < EPV) {
#pragma unroll
            for (int e = 0; e < EPV; ++e)
              if (e == off) g[e] -= gsT * a.lambda_ce;
          }
          if (!row_ok) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) g[e] = nan;
          }
#pragma unroll
          for (int h = 0; h < EPV / 4; ++h)
            st_stream(out + vi * EPV + 4 * h, g[4 * h], g[4 * h + 1], g[4 * h + 2], g[4 * h + 3]);
        }
    }
  }
  if (tid == 0 && sm.abort && issued_next) mbar_wait_bounded(&sm.mbar[0], 0);  // best effort drain
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
  int64_t CL = (row_bytes + 16383) / 16384;
  if (CL < 1) CL = 1;
  if (CL > kMaxCluster) CL = kMaxCluster;
  int64_t SL = (V + CL - 1) / CL;
  SL = (SL + 7) / 8 * 8;
  p.CL = static_cast<int>(CL);
  p.SL = static_cast<int>(SL);
  p.slice_bytes = static_cast<int>((SL * esize + 127) / 128 * 128);
  const size_t stage = static_cast<size_t>(p.slice_bytes) * 2;
  p.stages = 1;
  p.smem = stage;
  return p;
}

template <int DT, bool BULK, int NT, int STAGES>
cudaError_t launch_opd_t(const OpdArgs &a, const OpdPlan &p, cudaStream_t st) {
  auto kern = opd_kernel<DT, BULK, NT, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(p.smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent clusters: as many as can be co-resident (cached per shape)
  struct Entry {
    int dev;
    const void *fn;
    int CL;
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
    if (cache[q].dev == dev && cache[q].fn == reinterpret_cast<const void *>(kern) && cache[q].CL == p.CL &&
        cache[q].smem == p.smem)
      maxc = cache[q].n;
  if (maxc == 0) {
    cfg.gridDim = dim3(p.CL * 1024, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (maxc <= 0) return cudaErrorInvalidConfiguration;
    if (ncache < 32) cache[ncache++] = Entry{dev, reinterpret_cast<const void *>(kern), p.CL, p.smem, maxc};
  }
  int64_t nclusters = maxc;
  if (nclusters > a.R) nclusters = a.R;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * p.CL), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, a, p.SL, p.slice_bytes);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT, int VPT>
cudaError_t launch_opd_reg(const OpdArgs &a, const OpdPlan &p, cudaStream_t st) {
  auto kern = opd_reg_kernel<DT, 512, VPT>;
  const size_t smem = static_cast<size_t>(p.slice_bytes) * 2;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(512, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int cached[64][9] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int &maxc = cached[dev & 63][p.CL];
  if (maxc == 0) {
    cfg.gridDim = dim3(p.CL * 1024, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (maxc <= 0) return cudaErrorInvalidConfiguration;
  }
  int64_t nclusters = maxc;
  if (nclusters > a.R) nclusters = a.R;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * p.CL), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, a, p.SL, p.slice_bytes);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT, bool BULK>
cudaError_t launch_opd_cfg(const OpdArgs &a, const OpdPlan &p, cudaStream_t st) {
  if (BULK) {
    const int nvec = static_cast<int>(static_cast<int64_t>(p.SL) * Elem<DT>::kSize / 16);
    const int vpt = (nvec + 511) / 512;
    if (vpt <= 1) return launch_opd_reg<DT, 1>(a, p, st);
    if (vpt <= 2) return launch_opd_reg<DT, 2>(a, p, st);
    if (vpt <= 3) return launch_opd_reg<DT, 3>(a, p, st);
    if (vpt <= 5) return launch_opd_reg<DT, 5>(a, p, st);
  }
  return launch_opd_t<DT, BULK, 512, 1>(a, p, st);
}

}  // namespace

bool opd_supported(int64_t V, int esize) { return plan_opd(V, esize).smem <= 200 * 1024; }

cudaError_t launch_opd(const OpdArgs &a, int dtype, bool bulk, cudaStream_t st) {
  const int esize = (dtype == SVW_BF16) ? 2 : 4;
  const OpdPlan p = plan_opd(a.V, esize);
  if (p.smem > 200 * 1024) return cudaErrorInvalidValue;
  if (dtype == SVW_BF16) return bulk ? launch_opd_cfg<1, true>(a, p, st) : launch_opd_cfg<1, false>(a, p, st);
  return bulk ? launch_opd_cfg<0, true>(a, p, st) : launch_opd_cfg<0, false>(a, p, st);
}

}  // namespace svw
