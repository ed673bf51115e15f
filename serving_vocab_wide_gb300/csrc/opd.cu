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
// the target and the draft row (76 KB at V = 151936 bf16, two CTAs of
// different clusters per SM).  Slices arrive by 1-D bulk async copies
// (cp.async.bulk, mbarrier completion): HBM sees each logit byte once.
//
// Fast kernel (16-byte-pitched rows).  Each thread moves its vectors of the
// slices from shared memory into registers as soon as they land, and the
// buffer is handed to the next row's copies at once.  One pass over the
// registers gives, per row, S_y = sum 2^((y - m_y)k), W = sum (2^((z - m_z)k)
// - 2^((y - m_y)k)) (so S_z = S_y + W), the target argmax with the draft
// logit there, and U = sum_v 2^((z_v - m_z)k) ((z_v - y_v)k - (m_z - m_y)k),
// so that without clipping
//   KL(q||p) = ln2 (U/S_z - log2(1 + W/S_y)),  S = sum_v q_v a_v = KL + 1;
// one exchange of partials merges these over the cluster, and a second
// register pass writes the gradient.  Precision: where the draft is close to
// its target (on-policy distillation converges there) log q - log p is small
// and the KL is its second moment, so nothing may be formed as a difference
// of two quantities of magnitude ~20.  The log ratio of an entry is
// (z - y)k - dC (the logit difference is exact for bf16, dC = Cd - Ct comes
// from W with an accurate log1p), never (z k - Cd) - (y k - Ct); W is summed
// term by term, never as S_z - S_y.  What is left is about 1e-7 (absolute)
// of KL from the exp2 unit and rounding; a row whose loss is small enough
// for that to matter (below kFastLossFloor) is flagged for a loss-only
// recomputation by the fix-up.  An entry whose term reaches the clip bound,
// or a non-finite KL (masked entries), flags the row for the full
// recomputation: the flag word is set to the call's tag (never cleared), so
// flags need no ordering and a stale tag at worst sends a row to the exact
// fix-up once more.
// Fix-up.  After the exchange every warp of the fast kernel also leaves its
// share of the exact clamped sum and of S: in closed form from its pass-1
// sums, corrected at the few entries that reach the clip.  Rows that need
// their sums term by term (masked entries, a small loss) leave that to the
// fix-up: one grid sums those rows' entries, a second adds the partials up
// for the rows the fast kernel flagged, writes the loss and rewrites the
// gradient.
// Exact kernel.  Without a workspace (or for rows that are not 16-byte
// pitched) every row is done from shared memory in three passes:
// log-sum-exps; clamped terms, S and the argmax; gradient -- two exchanges.
// The exact kernel and the fix-up sum sum_v [clamp(t_v) - q_v + p_v] (= the
// clamped sum, since both rows are normalised; see psi_series): this form is to
// first order insensitive to the rounding of the row constants, and it keeps
// the small-KL regime precise without the fast kernel's W machinery.
// In log2 units: log2 q = z k - Cd, log2 p = y k - Ct, d2 = (z - y) k - dC,
// t/ln2 = q d2; per-entry arithmetic runs on f32x2 pairs.
// Every wait on a bulk copy is bounded by a clock deadline; on expiry the CTA
// records SVW_DEV_TIMEOUT, stops issuing copies and keeps joining the cluster
// barriers so that no peer can hang.
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <mutex>

#include "opd_common.cuh"
#include "svw_device.cuh"
#include "svw_internal.h"

namespace cg = cooperative_groups;

namespace svw {

namespace {

constexpr int kMaxWarps = 32;
// The fast kernel's KL comes from the row sums s_y, w, u: rounding and the
// SFU's exp2 error leave about 1e-7 (absolute, nats) in it.  A loss smaller
// than this bound (a draft almost equal to its target with a small lambda) is
// summed again exactly by the fix-up grids, so that it keeps its relative
// precision; the gradient does not need it (its scale is that of log q - log p).
constexpr float kFastLossFloor = 4e-3f;
constexpr int kMaxCluster = 8;
static_assert(kMaxCluster <= kBonusParts, "bonus partial stride");

struct OpdSmem {
  unsigned long long mbar;
  float red[kMaxWarps][4];
  int32_t redi[kMaxWarps];
  float partA[8];  // this CTA's mt, st, md, sd, abort
  float partB[4];  // this CTA's rkl (log2 units), S, argmax candidate (bits)
  float rowA[8];   // merged over the cluster: Mt, St, Md, Sd, any abort
  float rowB[4];   // merged over the cluster: rkl, S, argmax (bits)
  int64_t tr;      // target row of the current row (-1: outside its request)
  int32_t abort;
  uint32_t abort_parity;  // phase of the copy that timed out
};

// Exact three-pass kernel (every row; the path without a workspace).
template <int DT, bool BULK>
__global__ void __launch_bounds__(512, 2) opd_exact_kernel(OpdArgs a, OpdGeo geo) {
  constexpr int NT = 512;
  const int32_t SL = geo.SL, slice_bytes = geo.slice_bytes;
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
    mbar_init(&sm.mbar, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  unsigned char *tbuf = dyn;
  unsigned char *dbuf = dyn + slice_bytes;
  const uint32_t tb = smem_u32(tbuf), db = smem_u32(dbuf);
  // thread 0: start the bulk copies of row r's slices (after a timeout the
  // barrier is left alone: its phase never completed)
  auto issue = [&](int64_t r) {
    const int64_t t = target_row_of(a, r);
    sm.tr = t;
    const uint32_t bytes = static_cast<uint32_t>(n) * E::kSize;
    if (sm.abort) return;
    if (t >= 0 && bytes > 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&sm.mbar, 2 * bytes);
      bulk_g2s(tbuf, static_cast<const char *>(a.target) + (t * V + lo) * E::kSize, bytes, &sm.mbar);
      bulk_g2s(dbuf, static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize, bytes, &sm.mbar);
    } else {
      mbar_arrive(&sm.mbar);
    }
  };

  for (int64_t r = cid, it = 0; r < a.R; r += nclusters) {
    const uint32_t parity = static_cast<uint32_t>(it & 1);
    // ---- fill the slices ----
    if (BULK) {
      if (tid == 0) issue(r);
      if (!sm.abort && !mbar_wait_bounded(&sm.mbar, parity)) {
        if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        sm.abort_parity = parity;
        sm.abort = 1;
      }
      __syncthreads();
    } else {
      if (tid == 0) sm.tr = target_row_of(a, r);
      __syncthreads();
      const int64_t t = sm.tr;
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
    const bool valid = (sm.tr >= 0);
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
    // dC = Cd - Ct from the maxima's exact difference and an accurate log2 of
    // the ratio of the sums: log2 q - log2 p = (z - y) k - dC, with no
    // cancellation between two row offsets of magnitude ~20
    const float dC = fmaf(Md - Mt, k, log2f(Sd / St));
    const float Cd = Ct + dC;               // log2 q = z k - Cd
    const float c2 = a.clip_c * kLog2e;     // clip bound in log2 units of t
    float rkl = 0.f, S = 0.f;
    int32_t cand = INT32_MAX;

    // ---------------- pass B: clamped terms, S, argmax ----------------
    // rkl = sum_v [clamp(t_v) - q_v + p_v] (nats), insensitive to first order
    // to the rounding of Ct and dC (see psi_series)
    if (row_ok) {
      const float2 kk = make_float2(k, k), neg1 = make_float2(-1.f, -1.f);
      const float2 nCd = make_float2(-Cd, -Cd), ndC = make_float2(-dC, -dC);
      for (int vi = tid; vi < nvec; vi += kThreads) {
        const Pairs<DT> y(lds128(tb + vi * 16)), z(lds128(db + vi * 16));
#pragma unroll
        for (int h = 0; h < Pairs<DT>::kN; ++h) {
          const float2 A = __ffma2_rn(z.p[h], kk, nCd);                                  // log2 q
          const float2 q = make_float2(ex2(A.x), ex2(A.y));
          const float2 d = __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC);        // log2 q - log2 p
          clamped_term(q.x, d.x, y.p[h].x, k, Ct, c2, a.clip_c, rkl, S);
          clamped_term(q.y, d.y, y.p[h].y, k, Ct, c2, a.clip_c, rkl, S);
        }
      }
      if (!BULK && tid == 0)
        for (int v = nvec * EPV; v < n; ++v) {
          const float y = E::load_plain(tbuf, v), z = E::load_plain(dbuf, v);
          const float q = ex2(fmaf(z, k, -Cd));
          clamped_term(q, fmaf(z - y, k, -dC), y, k, Ct, c2, a.clip_c, rkl, S);
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
    const float RKL = sm.rowB[0], SS = sm.rowB[1];
    const int32_t xs = __float_as_int(sm.rowB[2]);
    if (rank == 0 && tid == 0) {
      float out = __int_as_float(0x7fffffff);
      if (row_ok && xs != INT32_MAX) {
        const float zx = E::load(a.draft, r * V + xs);
        // loss = sum clamp(t) + lambda * (-lq[x*]);  -lq[x*] = ln2 ((Md - z_x*) k + log2 Sd)
        out = fmaf(a.lambda_ce * kLn2, fmaf(Md - zx, k, lg2(Sd)), RKL);
      } else if (a.status && !any_abort) {
        atomicOr(a.status, SVW_DEV_BAD_INPUT);
      }
      a.loss[r] = out;
    }

    // ---------------- pass C: gradient wrt the draft logits ----------------
    // dz = gsT (qa + q (lambda - S)) - gsT lambda [v = x*], qa = t + q when
    // |t| < c else 0; in log2 units dz = t2 gsT ln2 + q gsT (lambda - S + 1).
    // SS holds S - 1.
    if (a.dlogits != nullptr && valid && !any_abort) {
      const float gsT = a.grad_scale * a.invT;
      const float gL0 = gsT * (a.lambda_ce - SS - 1.f);
      const float gL1 = gsT * (a.lambda_ce - SS);
      const float nan = __int_as_float(0x7fffffff);
      float *out = a.dlogits + r * V + lo;
      if (BULK) {
        const float2 kk = make_float2(k, k), neg1 = make_float2(-1.f, -1.f);
        const float2 nCd = make_float2(-Cd, -Cd), ndC = make_float2(-dC, -dC);
        const float2 gl = make_float2(gsT * kLn2, gsT * kLn2), g1 = make_float2(gL1, gL1);
        for (int vi = tid; vi < nvec; vi += kThreads) {
          const Pairs<DT> y(lds128(tb + vi * 16)), z(lds128(db + vi * 16));
          float g[EPV];
#pragma unroll
          for (int h = 0; h < Pairs<DT>::kN; ++h) {
            const float2 A = __ffma2_rn(z.p[h], kk, nCd);
            const float2 q = make_float2(ex2(A.x), ex2(A.y));
            const float2 t = __fmul2_rn(q, __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC));
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
          const float q = ex2(fmaf(z, k, -Cd));
          const float t = q * fmaf(z - y, k, -dC);
          float g = (fabsf(t) < c2) ? fmaf(t, gsT * kLn2, q * gL1) : q * gL0;
          if (lo + v == xs) g -= gsT * a.lambda_ce;
          out[v] = row_ok ? g : nan;
        }
      }
    }
    __syncthreads();  // the slices are fully consumed before the next copy
    ++it;
  }
  // after a timeout no copy is issued; let the one that timed out land if it can
  if (BULK && tid == 0 && sm.abort) mbar_wait_bounded(&sm.mbar, sm.abort_parity);
  cluster.sync();  // peers may still read this CTA's partials
}


struct FastSmem {
  unsigned long long mbar;
  // row exchange: every CTA pushes its partial into slot [rank] of each peer's
  // inbox; xbar[s] completes when all CL partials of the row have landed.
  // Two slots: a peer may send row r+1's partial before this CTA has merged
  // row r's, but never row r+2's.
  unsigned long long xbar[2];
  FastPart inbox[2][kMaxCluster];
  FastPart red[16];  // one partial per warp
  FastPart row;      // merged over the cluster
  // the row's constants, computed once from it (row_ok, any_abort, exact, small in bits)
  struct {
    float Ct, dC, kl, loss;
    int32_t bits;
  } rk;
  // bonus rows (fused verification) are not exchanged: double-buffered warp
  // partials, merged by the last warp and stored per CTA
  FastPart bred[2][16];
  uint32_t nbred[2];  // warps done with bonus rows, by row parity (a warp may be a row ahead)
  int64_t tr;
  uint32_t nread;  // warps done reading the slice buffer (16 per row)
  int32_t abort;
  uint32_t abort_parity;  // phase of the copy that timed out
};


template <int DT, int VPT, int NT>
__global__ void __launch_bounds__(NT, 2) opd_fast_kernel(OpdArgs a, OpdGeo geo) {
  using E = Elem<DT>;
  constexpr int kWarps = NT / 32;
  constexpr int EPV = E::kPerVec;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ FastSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nclusters = gridDim.x / CL;
  const int64_t cid = blockIdx.x / CL;
  const int64_t V = a.V;
  const int64_t lo = static_cast<int64_t>(rank) * geo.SL;
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(geo.SL), V - lo)));
  const int nvec = n / EPV;  // V is a multiple of EPV on this path: no tail
  const int nj = (tid < nvec) ? min(VPT, (nvec - tid + NT - 1) / NT) : 0;
  const float k = a.k;
  unsigned char *tbuf = dyn;
  unsigned char *dbuf = dyn + geo.slice_bytes;
  int32_t *tab = reinterpret_cast<int32_t *>(dyn + 2 * static_cast<size_t>(geo.slice_bytes));
  const uint32_t tb = smem_u32(tbuf), db = smem_u32(dbuf);

  if (tid == 0) {
    mbar_init(&sm.mbar, 1);
    mbar_init(&sm.xbar[0], 1);
    mbar_init(&sm.xbar[1], 1);
    sm.abort = 0;
    sm.nread = 0;
    sm.nbred[0] = sm.nbred[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster.sync();  // every inbox barrier exists before any peer sends
  const int64_t R_all = a.R + a.nbonus;  // draft rows, then bonus rows (fused verification)
  if (a.nbonus > 0) {
    // the fused finalize kernel may be scheduled as this grid drains
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // this CTA's share of the CSR consistency check: cu[0] = 0, cu[N] = R,
    // non-decreasing (the fused finalize kernel ORs the flags)
    int bad = 0;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * NT + tid; j < a.N; j += static_cast<int64_t>(gridDim.x) * NT)
      bad |= (__ldg(a.cu + j) > __ldg(a.cu + j + 1)) ? 1 : 0;
    if (blockIdx.x == 0 && tid == 0)
      bad |= (__ldg(a.cu) != 0 || static_cast<int64_t>(__ldg(a.cu + a.N)) != a.R) ? 1 : 0;
    bad = __syncthreads_or(bad);
    if (tid == 0) a.csr_bad[blockIdx.x] = bad;
  }
  // one thread: start the bulk copies of row r (target row t; draft row r
  // unless r is a bonus row)
  auto issue = [&](int64_t r, int64_t t) {
    sm.tr = t;
    const uint32_t bytes = static_cast<uint32_t>(n) * E::kSize;
    if (sm.abort) return;  // after a timeout the barrier is left alone
    // test-only fault (svw_set_fault): cluster 0 issues nothing, so its first
    // wait runs out with no copy in flight
    if (a.fault == 1 && cid == 0) return;
    if (t >= 0 && bytes > 0) {
      const bool pair = r < a.R;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&sm.mbar, (pair ? 2 : 1) * bytes);
      bulk_g2s(tbuf, static_cast<const char *>(a.target) + (t * V + lo) * E::kSize, bytes, &sm.mbar);
      if (pair) bulk_g2s(dbuf, static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize, bytes, &sm.mbar);
    } else {
      mbar_arrive(&sm.mbar);
    }
  };
  if (tid == 0 && cid < R_all) issue(cid, fast_target_row(a, cid));
  // target rows of this cluster's later rows (verify layout), looked up once
  for (int q = 1 + tid; q < geo.ntab; q += NT) {
    const int64_t r = cid + q * nclusters;
    tab[q] = (r < R_all) ? static_cast<int32_t>(fast_target_row(a, r)) : -1;
  }
  __syncthreads();

  int64_t ib = 0;  // bonus rows done by this CTA
  for (int64_t r = cid, it = 0; r < R_all; r += nclusters, ++it) {
    const bool pair = r < a.R;  // false: a bonus row (target only, statistics only)
    if (!sm.abort && !mbar_wait_bounded(&sm.mbar, static_cast<uint32_t>(it & 1))) {
      if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
      sm.abort_parity = static_cast<uint32_t>(it & 1);
      sm.abort = 1;
    }
    const int64_t sm_tr_row = sm.tr;
    const bool valid = (sm_tr_row >= 0);
    uint4 ty[VPT], tz[VPT];
    const uint32_t ninf = (DT == 1) ? 0xff80ff80u : 0xff800000u;  // -inf in every lane of the vector
#pragma unroll
    for (int j = 0; j < VPT; ++j)
      if (j < nj) {
        ty[j] = lds128(tb + (tid + j * NT) * 16);
        tz[j] = pair ? lds128(db + (tid + j * NT) * 16) : make_uint4(ninf, ninf, ninf, ninf);
      }
    const bool work = valid && !sm.abort;
    // the buffer is free once every warp holds its vectors: the last warp to
    // get there streams the next row in, nobody waits
    if (last_warp_done<kWarps>(&sm.nread, it)) {
      const int64_t rn = r + nclusters;
      if (rn < R_all) {
        const int64_t q = it + 1;
        const int64_t tn = !a.has_bonus ? rn : (q < geo.ntab ? static_cast<int64_t>(tab[q]) : fast_target_row(a, rn));
        issue(rn, tn);
      }
    }

    if (!pair) {
      // ---- bonus row: maximum, exp-sum and first argmax of this CTA's slice,
      // stored for the fused finalize kernel (no exchange, no barrier) ----
      FastPart P = empty_part();
      P.abort = sm.abort;
      if (work) {
        float my;
        if (DT == 1) {
          uint32_t py = 0xff80ff80u;
#pragma unroll
          for (int j = 0; j < VPT; ++j)
            if (j < nj) py = bf16x2_max(py, bf16x2_max(bf16x2_max(ty[j].x, ty[j].y), bf16x2_max(ty[j].z, ty[j].w)));
          const float2 fy = bf16x2_f2(py);
          my = fmaxf(fy.x, fy.y);
        } else {
          my = -INFINITY;
#pragma unroll
          for (int j = 0; j < VPT; ++j)
            if (j < nj) my = vec_max<DT>(ty[j], my);
        }
        float My = my;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) My = fmaxf(My, __shfl_xor_sync(0xffffffffu, My, o));
        int32_t idx = INT32_MAX;
        if (my == My) {
          if (DT == 1) {
            const uint32_t m16 = __float_as_uint(My) >> 16, m2 = m16 | (m16 << 16);
#pragma unroll
            for (int j = 0; j < VPT; ++j)
              if (j < nj && idx == INT32_MAX) {
                const int e = bf16_vec_find(ty[j], m2);
                if (e >= 0) idx = static_cast<int32_t>(lo + (tid + j * NT) * EPV + e);
              }
          } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j)
              if (j < nj && idx == INT32_MAX) {
                float y[EPV];
                E::unpack(ty[j], y);
#pragma unroll
                for (int e = EPV - 1; e >= 0; --e)
                  if (y[e] == My) idx = static_cast<int32_t>(lo + (tid + j * NT) * EPV + e);
              }
          }
        }
        const float nmy = (My == -INFINITY) ? 0.f : -My * k;
        const float2 kk = make_float2(k, k), ny2 = make_float2(nmy, nmy);
        float2 sy = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j < nj) {
            const Pairs<DT> y(ty[j]);
#pragma unroll
            for (int h = 0; h < Pairs<DT>::kN; ++h) {
              const float2 ay = __ffma2_rn(y.p[h], kk, ny2);
              sy = __fadd2_rn(sy, make_float2(ex2(ay.x), ex2(ay.y)));
            }
          }
        float s0 = sy.x + sy.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        P.my = My;
        P.sy = s0;
        P.idx = static_cast<int32_t>(__reduce_min_sync(0xffffffffu, static_cast<uint32_t>(idx)));
      }
      if (lane == 0) sm.bred[ib & 1][warp] = P;
      if (last_warp_all<kWarps>(&sm.nbred[ib & 1], ib >> 1)) {
        const FastPart Pc = merge_lanes<kWarps>(lane < kWarps ? sm.bred[ib & 1][lane] : empty_part(), k);
        if (lane == 0) {
          float4 *dst = reinterpret_cast<float4 *>(a.bpart + ((r - a.R) * kBonusParts + rank));
          dst[0] = make_float4(Pc.my, Pc.sy, __int_as_float(Pc.idx), __int_as_float(valid ? Pc.abort : 2));
        }
      }
      ++ib;
      continue;
    }

    // ---------------- pass 1: row statistics ----------------
    FastPart P = empty_part();
    P.abort = sm.abort;
    if (work) {
      float my, mz;
      if (DT == 1) {
        uint32_t py = 0xff80ff80u, pz = 0xff80ff80u;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j < nj) {
            py = bf16x2_max(py, bf16x2_max(bf16x2_max(ty[j].x, ty[j].y), bf16x2_max(ty[j].z, ty[j].w)));
            pz = bf16x2_max(pz, bf16x2_max(bf16x2_max(tz[j].x, tz[j].y), bf16x2_max(tz[j].z, tz[j].w)));
          }
        const float2 fy = bf16x2_f2(py), fz = bf16x2_f2(pz);
        my = fmaxf(fy.x, fy.y);
        mz = fmaxf(fz.x, fz.y);
      } else {
        my = -INFINITY;
        mz = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j < nj) {
            my = vec_max<DT>(ty[j], my);
            mz = vec_max<DT>(tz[j], mz);
          }
      }
      // warp offsets
      float My = my, Mz = mz;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        My = fmaxf(My, __shfl_xor_sync(0xffffffffu, My, o));
        Mz = fmaxf(Mz, __shfl_xor_sync(0xffffffffu, Mz, o));
      }
      // first index of the warp's target maximum (only its holders look)
      int32_t idx = INT32_MAX;
      float zx = 0.f;
      if (my == My) {
        if (DT == 1) {
          const uint32_t m16 = __float_as_uint(My) >> 16, m2 = m16 | (m16 << 16);  // My is a bf16 value
#pragma unroll
          for (int j = 0; j < VPT; ++j)
            if (j < nj && idx == INT32_MAX) {
              const int e = bf16_vec_find(ty[j], m2);
              if (e >= 0) {
                idx = static_cast<int32_t>(lo + (tid + j * NT) * EPV + e);
                zx = bf16_vec_get(tz[j], e);
              }
            }
        } else {
#pragma unroll
          for (int j = 0; j < VPT; ++j)
            if (j < nj && idx == INT32_MAX) {
              float y[EPV], z[EPV];
              E::unpack(ty[j], y);
              E::unpack(tz[j], z);
#pragma unroll
              for (int e = EPV - 1; e >= 0; --e)
                if (y[e] == My) {
                  idx = static_cast<int32_t>(lo + (tid + j * NT) * EPV + e);
                  zx = z[e];
                }
            }
        }
      }
      const float nmy = (My == -INFINITY) ? 0.f : -My * k;
      const float nmz = (Mz == -INFINITY) ? 0.f : -Mz * k;
      // log-ratio reference (m_z - m_y) k of this warp's partial
      const float ncw = (My == -INFINITY || Mz == -INFINITY) ? 0.f : -(Mz - My) * k;
      const float2 kk = make_float2(k, k), ny2 = make_float2(nmy, nmy), nz2 = make_float2(nmz, nmz);
      const float2 nc2 = make_float2(ncw, ncw), neg1 = make_float2(-1.f, -1.f);
      float2 sy = make_float2(0.f, 0.f), ww = make_float2(0.f, 0.f), uu = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < VPT; ++j)
        if (j < nj) {
          const Pairs<DT> y(ty[j]), z(tz[j]);
#pragma unroll
          for (int h = 0; h < Pairs<DT>::kN; ++h) {
            const float2 ay = __ffma2_rn(y.p[h], kk, ny2);  // (y - m_y) k
            const float2 az = __ffma2_rn(z.p[h], kk, nz2);  // (z - m_z) k
            const float2 ey = make_float2(ex2(ay.x), ex2(ay.y));
            const float2 ez = make_float2(ex2(az.x), ex2(az.y));
            // (z - y) k - (m_z - m_y) k as the difference of the two scaled entries:
            // its rounding (~1e-7 of |az|) is weighted by ez, small where |az| is large
            const float2 xd = __ffma2_rn(ay, neg1, az);
            sy = __fadd2_rn(sy, ey);
            ww = __fadd2_rn(ww, __ffma2_rn(ey, neg1, ez));
            uu = __ffma2_rn(ez, xd, uu);
          }
        }
      float s0 = sy.x + sy.y, s1 = ww.x + ww.y, s2 = uu.x + uu.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      }
      const int32_t best = static_cast<int32_t>(__reduce_min_sync(0xffffffffu, static_cast<uint32_t>(idx)));
      const uint32_t holders = __ballot_sync(0xffffffffu, idx == best);
      P.my = My;
      P.mz = Mz;
      P.sy = s0;
      P.w = s1;
      P.u = s2;
      P.idx = best;
      P.zx = __shfl_sync(0xffffffffu, zx, holders ? __ffs(holders) - 1 : 0);
    }
    if (lane == 0) sm.red[warp] = P;
    if (warp == 0) {
      const int slot = static_cast<int>(it & 1);
      if (lane == 0) mbar_arrive_expect_tx(&sm.xbar[slot], static_cast<uint32_t>(CL) * sizeof(FastPart));
      named_sync(2, NT);  // every warp's partial is in
      const FastPart Pc = merge_lanes<kWarps>(lane < kWarps ? sm.red[lane] : empty_part(), k);
      if (lane < CL) {  // lane q pushes this CTA's partial to CTA q
        const uint4 w0 = make_uint4(__float_as_uint(Pc.my), __float_as_uint(Pc.sy), __float_as_uint(Pc.mz),
                                    __float_as_uint(Pc.w));
        const uint4 w1 = make_uint4(__float_as_uint(Pc.u), static_cast<uint32_t>(Pc.idx), __float_as_uint(Pc.zx),
                                    static_cast<uint32_t>(Pc.abort));
        const uint32_t dst = mapa_shared(smem_u32(&sm.inbox[slot][rank]), lane);
        const uint32_t bar = mapa_shared(smem_u32(&sm.xbar[slot]), lane);
        st_async16(dst, w0, bar);
        st_async16(dst + 16, w1, bar);
      }
      FastPart Pq = empty_part();
      if (mbar_wait_bounded(&sm.xbar[slot], static_cast<uint32_t>((it >> 1) & 1))) {
        if (lane < CL) Pq = sm.inbox[slot][lane];
      } else {
        if (lane == 0 && a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        Pq.abort = 1;
      }
      const FastPart M = merge_lanes<kMaxCluster>(Pq, k);
      if (lane == 0) {
        sm.row = M;
        // the row's constants, once per CTA (the merged row is the same in
        // every CTA of the cluster, so these are too)
        const bool any_abort = M.abort != 0;
        const float Sz = M.sy + M.w;
        const bool row_ok = valid && !any_abort && (M.sy > 0.f && M.sy <= FLT_MAX) && (Sz > 0.f && Sz <= FLT_MAX);
        const float Ct = fmaf(M.my, k, lg2(M.sy));  // log2 p = y k - Ct
        // log2(S_z / S_y) from the termwise difference w (accurate log1p), and
        // dC = Cd - Ct: log2 q - log2 p = (z - y) k - dC
        const float l2r = log1pf(M.w / M.sy) * kLog2e;
        const float dC = fmaf(M.mz - M.my, k, l2r);
        // unclipped KL(q||p) = E_q[(z - y) k - (m_z - m_y) k] - log2(S_z / S_y), in nats
        const float kl = kLn2 * (M.u / Sz - l2r);
        const bool exact = (kl == kl) && fabsf(kl) <= FLT_MAX;
        // loss = KL + lambda (-lq[x*]),  -lq[x*] = ln2 ((m_z - z_x*) k + log2 S_z)
        const float loss_r = fmaf(a.lambda_ce * kLn2, fmaf(M.mz - M.zx, k, lg2(Sz)), kl);
        const bool small = !(fabsf(loss_r) >= kFastLossFloor);
        sm.rk.Ct = Ct;
        sm.rk.dC = dC;
        sm.rk.kl = kl;
        sm.rk.loss = loss_r;
        sm.rk.bits = (row_ok ? 1 : 0) | (any_abort ? 2 : 0) | (exact ? 4 : 0) | (small ? 8 : 0);
      }
    } else {
      named_arrive(2, NT);
    }
    __syncthreads();  // the merged row and its constants are published
    const FastPart Rw = sm.row;
    const int32_t kbits = sm.rk.bits;
    const bool row_ok = (kbits & 1) != 0, any_abort = (kbits & 2) != 0;
    const bool exact = (kbits & 4) != 0, small = (kbits & 8) != 0;
    const float Ct = sm.rk.Ct, dC = sm.rk.dC, kl = sm.rk.kl, loss_r = sm.rk.loss;
    const float Cd = Ct + dC;                     // log2 q = z k - Cd
    const float c2 = a.clip_c * kLog2e;           // clip bound for t / ln 2
    const int32_t xs = Rw.idx;
    if (rank == 0 && tid == 0) {
      float out = __int_as_float(0x7fffffff);
      float4 rc = make_float4(__int_as_float(0x7fffffff), 0.f, 0.f, 0.f);  // NaN: not a row to fix
      if (row_ok && xs != INT32_MAX) {
        out = loss_r;
        if (!exact)
          atomicExch(a.flags + r, a.epoch);  // masked entries: the fix-up redoes this row
        else if (small)
          flag_loss_only(a.flags + r, a.epoch);  // a loss this small: the fix-up sums it exactly
        const int64_t t = sm_tr_row;
        rc = make_float4(Ct, dC, __int_as_float(xs),
                         __int_as_float(t < (int64_t{1} << 31) ? static_cast<int32_t>(t) : -2));
      } else if (a.status && !any_abort) {
        atomicOr(a.status, SVW_DEV_BAD_INPUT);
      }
      a.rowc[r] = rc;
      a.loss[r] = out;
    }

    // ---------------- pass 2: gradient wrt the draft logits ----------------
    // dz = gsT q (d + 1 - S + lambda) - gsT lambda [v = x*] with S = KL + 1,
    // d = ln2 d2:  dz = q (d2 gsT ln2 + gsT (lambda - KL)).
    if (valid && !any_abort && (a.dlogits != nullptr || row_ok)) {
      const float gsT = a.grad_scale * a.invT;
      const float2 kk = make_float2(k, k), neg1 = make_float2(-1.f, -1.f);
      const float2 nCd = make_float2(-Cd, -Cd), ndC = make_float2(-dC, -dC);
      float tmax = 0.f;  // largest |t| / ln2 seen by this thread
      if (a.dlogits != nullptr) {
        const float nan = __int_as_float(0x7fffffff);
        float *out = a.dlogits + r * V + lo;
        const float2 gl = make_float2(gsT * kLn2, gsT * kLn2);
        const float g0 = gsT * (a.lambda_ce - kl);
        const float2 g02 = make_float2(g0, g0);
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j < nj) {
            const int vi = tid + j * NT;
            const Pairs<DT> y(ty[j]), z(tz[j]);
            float g[EPV];
#pragma unroll
            for (int h = 0; h < Pairs<DT>::kN; ++h) {
              const float2 A = __ffma2_rn(z.p[h], kk, nCd);                               // log2 q
              const float2 q = make_float2(ex2(A.x), ex2(A.y));
              const float2 d = __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC);   // log2 q - log2 p
              const float2 t = __fmul2_rn(q, d);                                          // t / ln 2
              tmax = fmaxf(tmax, fmaxf(fabsf(t.x), fabsf(t.y)));
              const float2 gg = __fmul2_rn(q, __ffma2_rn(d, gl, g02));
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
#pragma unroll
        for (int j = 0; j < VPT; ++j)
          if (j < nj) {
            const Pairs<DT> y(ty[j]), z(tz[j]);
#pragma unroll
            for (int h = 0; h < Pairs<DT>::kN; ++h) {
              const float2 A = __ffma2_rn(z.p[h], kk, nCd);
              const float2 q = make_float2(ex2(A.x), ex2(A.y));
              const float2 t = __fmul2_rn(q, __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC));
              tmax = fmaxf(tmax, fmaxf(fabsf(t.x), fabsf(t.y)));
            }
          }
      }
      // some term reached the clip: the fix-up kernel redoes the row (every
      // writer stores the same call tag, so no ordering is needed)
      if (row_ok && !(tmax < c2)) atomicExch(a.flags + r, a.epoch);
      // the fix-up's partial sums over this warp's entries, sum [clamp(t) - q + p]
      // and S - 1 (nats): in closed form from the warp's pass-1 sums as if no
      // term were clipped, sum q d2 = 2^(m_z k - Cd) (u + ((m_z - m_y) k - dC)
      // s_z), plus a correction at the entries that reach the clip.  NaN where
      // the row needs its sums term by term (masked entries, a small loss):
      // the fix-up sums those rows' entries exactly.
      if (row_ok) {
        float rk = 0.f, s1 = 0.f;
        if (!exact || small) {
          rk = s1 = __int_as_float(0x7fffffff);
        } else {
          if (P.my != -INFINITY && P.mz != -INFINITY) {
            const float Szw = P.sy + P.w;
            const float fq = ex2(fmaf(P.mz, k, -Cd)), fp = ex2(fmaf(P.my, k, -Ct));
            const float qd2 = fq * fmaf(fmaf(P.mz - P.my, k, -dC), Szw, P.u);
            s1 = kLn2 * qd2;
            rk = fmaf(fp, P.sy, fmaf(-fq, Szw, s1));
          }
          if (__any_sync(0xffffffffu, !(tmax < c2))) {
            // the warp holds a term at the clip: such an entry contributes
            // +-c - t instead of nothing more to the clamped sum, and -q(1 + d)
            // to S - 1 (t = q d, d = ln2 d2)
            float cr = 0.f, cs = 0.f;
#pragma unroll
            for (int j = 0; j < VPT; ++j)
              if (j < nj) {
                const Pairs<DT> y(ty[j]), z(tz[j]);
#pragma unroll
                for (int h = 0; h < Pairs<DT>::kN; ++h) {
                  const float2 A = __ffma2_rn(z.p[h], kk, nCd);
                  const float2 q = make_float2(ex2(A.x), ex2(A.y));
                  const float2 d = __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC);
                  const float2 t = __fmul2_rn(q, d);
                  if (!(fabsf(t.x) < c2)) {
                    cr += fmaf(-kLn2, t.x, (t.x > 0.f) ? a.clip_c : -a.clip_c);
                    cs -= fmaf(q.x * kLn2, d.x, q.x);
                  }
                  if (!(fabsf(t.y) < c2)) {
                    cr += fmaf(-kLn2, t.y, (t.y > 0.f) ? a.clip_c : -a.clip_c);
                    cs -= fmaf(q.y * kLn2, d.y, q.y);
                  }
                }
              }
            rk += warp_sum(cr);
            s1 += warp_sum(cs);
          }
        }
        if (lane == 0) a.fixp[r * kOpdFixParts + rank * kWarps + warp] = make_float2(rk, s1);
      }
    }
  }
  // after a timeout no copy is issued; let the one that timed out land if it can
  if (tid == 0 && sm.abort) mbar_wait_bounded(&sm.mbar, sm.abort_parity);
  cluster.sync();  // peers may still read this CTA's partials
}

// Fix-up of the rows the fast kernel flagged (a term at the clip bound, or
// masked draft entries; or, loss only, a loss below kFastLossFloor),
// exactly, from the row constants it stored (Ct, dC, x*, target row) and the
// per-warp partial sums sum [clamp(t) - q + p] and S - 1 (nats) it left in
// the workspace (NaN for every warp of a row that needs its sums term by
// term):
//   opd_fix_parts: one warp per row: for a flagged row, each NaN part's
//                  entries summed term by term;
//   opd_fix_grad:  one warp per (flagged row, vocabulary chunk) item,
//                  kOpdFixChunks chunks per row: the row totals (a fixed
//                  order over the partials, identical in every warp), the
//                  loss (chunk 0) and the chunk's gradient (its logits read
//                  again).
// Both walk the flags in batches of kFixBatch rows; a batch's flagged rows
// are listed in row order by every CTA (a block scan), so the item order is
// the same everywhere.  No waits on other CTAs: nothing can hang.
constexpr int kFixBatch = 4096;  // flags scanned per batch
constexpr int32_t kFixFullBit = 1 << 30;  // in a FixList entry: the row's gradient is rewritten
constexpr int kFixNT = 256;
constexpr int kFixU = 5;  // 16-byte vectors of each row in flight per thread

struct FixGeo {
  int32_t CH;   // entries per chunk (a multiple of 8)
  int32_t nch;  // chunks per row (<= kOpdFixChunks)
  // the fast kernel's layout: its clusters left np = CL * fw partial sums
  // per row, part q from warp q % fw of CTA q / fw, whose threads held
  // vectors tid + j fnt (j < vpt) of vocabulary slice [SL (q / fw), SL (q / fw + 1))
  int32_t np, fw, fnt, vpt, SL;
  // opd_fix_grad: 0 = wait for the grid ahead (the parts grid) before reading
  // the partial sums; 1 = read them at once and wait at the end (the grid
  // ahead is the fused finalize, which lets its dependents go only once it
  // has waited for the parts grid, itself complete only after the fast kernel)
  int32_t wait_last;
};

struct FixList {
  int32_t list[kFixBatch];  // flagged rows of the batch (offsets from its base), in order
  int32_t wcnt[kFixNT / 32];
};

// The flagged rows of batch [base, base + kFixBatch) into fl.list, in row
// order (kFixFullBit set for a row flagged for the full recomputation, clear
// for a loss-only one); returns their number (in every thread).  Warp w reads rows
// [w 512, (w + 1) 512) of the batch 32 at a time (coalesced) and keeps one
// ballot per 32.  A flag is this call's tag; a stale tag on a row the fast
// kernel found bad (NaN row constants) is not.
__device__ __forceinline__ int fix_scan(const OpdArgs &a, int64_t base, FixList &fl) {
  constexpr int kWarps = kFixNT / 32;
  constexpr int kPerWarp = kFixBatch / kWarps;
  constexpr int kRounds = kPerWarp / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t wb = base + static_cast<int64_t>(warp) * kPerWarp;
  uint32_t ball[kRounds], full[kRounds];
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < kRounds; ++i) {
    const int64_t r = wb + i * 32 + lane;
    bool f = false, g = false;
    if (r < a.R) {
      const int32_t fv = __ldcg(a.flags + r);
      g = (fv == a.epoch);
      f = g || (fv == (a.epoch ^ kLossOnlyTag));
    }
    if (f) {
      const float ct = __ldcg(&a.rowc[r].x);
      f = (ct == ct);
    }
    ball[i] = __ballot_sync(0xffffffffu, f);
    full[i] = __ballot_sync(0xffffffffu, f && g);
    cnt += __popc(ball[i]);
  }
  if (lane == 0) fl.wcnt[warp] = cnt;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = fl.wcnt[w];
    before += (w < warp) ? c : 0;
    total += c;
  }
  const uint32_t below = (1u << lane) - 1u;
  int g = before;
#pragma unroll
  for (int i = 0; i < kRounds; ++i) {
    if (ball[i] & (1u << lane))
      fl.list[g + __popc(ball[i] & below)] =
          (warp * kPerWarp + i * 32 + lane) | ((full[i] & (1u << lane)) ? kFixFullBit : 0);
    g += __popc(ball[i]);
  }
  __syncthreads();  // the list is complete; every thread has read fl.wcnt
  return total;
}

// target row of flagged row r from its row constants (the fast kernel stores
// it when it fits an int32, else -2)
__device__ __forceinline__ int64_t fix_target_row(const OpdArgs &a, int64_t r, const float4 &rc) {
  const int32_t t32 = __float_as_int(rc.w);
  return (t32 >= 0) ? static_cast<int64_t>(t32) : target_row_of(a, r);
}

// Exact partial sums, term by term, of the warps the fast kernel left NaN (a
// row that needs its sums term by term): one warp per draft row, no block
// barrier.  The warp reads the row's flag; for a
// flagged row lane q checks parts q, q + 32, ... and the warp sums each NaN
// part's entries (the entries that fast-kernel warp held).  Parts already in
// closed form are left alone.
template <int DT>
__global__ void __launch_bounds__(kFixNT, 3) opd_fix_parts(OpdArgs a, FixGeo fg) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int kW = kFixNT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t V = a.V;
  const float k = a.k, c2 = a.clip_c * kLog2e;
  // the grid behind may be scheduled now (the gradient grid scans the flags,
  // then waits for this one; the fused finalize reads its inputs, then
  // waits).  The kernel ahead is the fast kernel, which in the fused call
  // lets this grid start as it begins: wait for its output.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kW + warp; r < a.R; r += static_cast<int64_t>(gridDim.x) * kW) {
    const int32_t fv = __ldcg(a.flags + r);
    if (fv != a.epoch && fv != (a.epoch ^ kLossOnlyTag)) continue;
    const float4 rc = __ldcg(a.rowc + r);
    if (!(rc.x == rc.x)) continue;  // a bad row: not fixed
    const int64_t t = fix_target_row(a, r, rc);
    if (t < 0) continue;
    uint32_t todo = 0;  // bit u: part lane + 32 u is NaN
#pragma unroll
    for (int u = 0; u < kOpdFixParts / 32; ++u)
      if (lane + 32 * u < fg.np) {
        const float x = __ldcg(&a.fixp[r * kOpdFixParts + lane + 32 * u].x);
        if (!(x == x)) todo |= 1u << u;
      }
    const float Ct = rc.x, dC = rc.y, Cd = Ct + dC;
    const float2 kk = make_float2(k, k), neg1 = make_float2(-1.f, -1.f);
    const float2 nCd = make_float2(-Cd, -Cd), ndC = make_float2(-dC, -dC);
#pragma unroll 1
    for (int u = 0; u < kOpdFixParts / 32; ++u) {
      uint32_t ball = __ballot_sync(0xffffffffu, (todo >> u) & 1u);
      while (ball) {
        const int q = 32 * u + __ffs(ball) - 1;
        ball &= ball - 1;
        const int64_t lo = static_cast<int64_t>(q / fg.fw) * fg.SL;
        const int nvec =
            static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(fg.SL), V - lo))) / EPV;
        const char *trow = static_cast<const char *>(a.target) + (t * V + lo) * E::kSize;
        const char *drow = static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize;
        const int v0 = (q % fg.fw) * 32 + lane;
        float rk = 0.f, s1 = 0.f;
        for (int j0 = 0; j0 < fg.vpt; j0 += kFixU) {
          // kFixU vectors of each row in flight before any arithmetic
          uint4 ty[kFixU], tz[kFixU];
#pragma unroll
          for (int w = 0; w < kFixU; ++w) {
            const int v = v0 + (j0 + w) * fg.fnt;
            if (j0 + w < fg.vpt && v < nvec) {
              ty[w] = ld_vec(trow + static_cast<int64_t>(v) * 16);
              tz[w] = ld_vec(drow + static_cast<int64_t>(v) * 16);
            }
          }
#pragma unroll
          for (int w = 0; w < kFixU; ++w) {
            const int v = v0 + (j0 + w) * fg.fnt;
            if (!(j0 + w < fg.vpt && v < nvec)) continue;
            const Pairs<DT> y(ty[w]), z(tz[w]);
#pragma unroll
            for (int h = 0; h < Pairs<DT>::kN; ++h) {
              const float2 A = __ffma2_rn(z.p[h], kk, nCd);                              // log2 q
              const float2 qq = make_float2(ex2(A.x), ex2(A.y));
              const float2 d = __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC);  // log2 q - log2 p
              clamped_term(qq.x, d.x, y.p[h].x, k, Ct, c2, a.clip_c, rk, s1);
              clamped_term(qq.y, d.y, y.p[h].y, k, Ct, c2, a.clip_c, rk, s1);
            }
          }
        }
        rk = warp_sum(rk);
        s1 = warp_sum(s1);
        if (lane == 0) a.fixp[r * kOpdFixParts + q] = make_float2(rk, s1);
      }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kFixNT, 3) opd_fix_grad(OpdArgs a, FixGeo fg) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  __shared__ FixList fl;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t V = a.V;
  const float k = a.k, c2 = a.clip_c * kLog2e;
  const float gsT = a.grad_scale * a.invT;
  // this grid may start while the grid ahead of it runs: it scans the flags
  // (final since the fast kernel ended), then, behind the parts grid, waits
  // for it; behind the fused finalize (fg.wait_last) it works at once, beside
  // the finalize, and waits only at its end
  bool waited = false;
  for (int64_t base = 0; base < a.R; base += kFixBatch) {
    const int m = fix_scan(a, base, fl);
    if (!waited && !fg.wait_last) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    // one warp per (flagged row, chunk) item
    const int64_t items = static_cast<int64_t>(m) * fg.nch;
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (kFixNT / 32) + (tid >> 5); item < items;
         item += static_cast<int64_t>(gridDim.x) * (kFixNT / 32)) {
      const int kq = static_cast<int>(item / fg.nch), c = static_cast<int>(item % fg.nch);
      const int32_t ent = fl.list[kq];
      const int64_t r = base + (ent & ~kFixFullBit);
      const bool full = (ent & kFixFullBit) != 0;
      // the row constants and the fast kernel's partial sums in one round of loads
      const float4 rc = __ldcg(a.rowc + r);
      float2 pv[kOpdFixParts / 32];
#pragma unroll
      for (int q = 0; q < kOpdFixParts / 32; ++q)
        pv[q] = (lane + 32 * q < fg.np) ? __ldcg(a.fixp + r * kOpdFixParts + lane + 32 * q) : make_float2(0.f, 0.f);
      const int64_t t = fix_target_row(a, r, rc);
      if (t < 0) continue;
      const float Ct = rc.x, dC = rc.y, Cd = Ct + dC;
      const int32_t xs = __float_as_int(rc.z);
      // row totals of the partial sums: a fixed order (lane q adds partials
      // q, q + 32, ..., then a butterfly), the same in every warp
      float2 p = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kOpdFixParts / 32; ++q) {
        p.x += pv[q].x;
        p.y += pv[q].y;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        p.x += __shfl_xor_sync(0xffffffffu, p.x, o);
        p.y += __shfl_xor_sync(0xffffffffu, p.y, o);
      }
      const float RKL = p.x, SS = p.y;
      if (c == 0 && lane == 0) {
        const float zx = E::load(a.draft, r * V + xs);
        a.loss[r] = fmaf(a.lambda_ce * kLn2, Cd - zx * k, RKL);  // -lq[x*] = ln2 (Cd - z_x* k)
      }
      // rows flagged only for the size of their loss keep the fast kernel's gradient
      if (a.dlogits == nullptr || !full) continue;
      // gradient: gsT (q a + q (lambda - S)) - gsT lambda [v = x*]  (SS holds S - 1)
      const int64_t lo = static_cast<int64_t>(c) * fg.CH;
      const int nv = static_cast<int>(min(static_cast<int64_t>(fg.CH), V - lo)) / EPV;
      const char *trow = static_cast<const char *>(a.target) + (t * V + lo) * E::kSize;
      const char *drow = static_cast<const char *>(a.draft) + (r * V + lo) * E::kSize;
      float *out = a.dlogits + r * V + lo;
      const float gL0 = gsT * (a.lambda_ce - SS - 1.f);
      const float gL1 = gsT * (a.lambda_ce - SS);
      const float2 kk = make_float2(k, k), neg1 = make_float2(-1.f, -1.f);
      const float2 nCd = make_float2(-Cd, -Cd), ndC = make_float2(-dC, -dC);
      const float2 gl = make_float2(gsT * kLn2, gsT * kLn2), g1 = make_float2(gL1, gL1);
      for (int v0 = lane; v0 < nv; v0 += 32 * kFixU) {
        uint4 ty[kFixU], tz[kFixU];
#pragma unroll
        for (int u = 0; u < kFixU; ++u) {
          const int v = v0 + u * 32;
          if (v < nv) {
            ty[u] = ld_vec(trow + static_cast<int64_t>(v) * 16);
            tz[u] = ld_vec(drow + static_cast<int64_t>(v) * 16);
          }
        }
#pragma unroll
        for (int u = 0; u < kFixU; ++u) {
          const int v = v0 + u * 32;
          if (v < nv) {
            const Pairs<DT> y(ty[u]), z(tz[u]);
            float g[EPV];
#pragma unroll
            for (int h = 0; h < Pairs<DT>::kN; ++h) {
              const float2 A = __ffma2_rn(z.p[h], kk, nCd);
              const float2 q = make_float2(ex2(A.x), ex2(A.y));
              const float2 tt = __fmul2_rn(q, __ffma2_rn(__ffma2_rn(y.p[h], neg1, z.p[h]), kk, ndC));
              float2 gg = __ffma2_rn(tt, gl, __fmul2_rn(q, g1));
              if (!(fabsf(tt.x) < c2)) gg.x = q.x * gL0;
              if (!(fabsf(tt.y) < c2)) gg.y = q.y * gL0;
              g[2 * h] = gg.x;
              g[2 * h + 1] = gg.y;
            }
            const int off = static_cast<int>(xs - (lo + static_cast<int64_t>(v) * EPV));
            if (off >= 0 && off < EPV) {
#pragma unroll
              for (int e = 0; e < EPV; ++e)
                if (e == off) g[e] -= gsT * a.lambda_ce;
            }
#pragma unroll
            for (int h = 0; h < EPV / 4; ++h)
              st_stream(out + static_cast<int64_t>(v) * EPV + 4 * h, g[4 * h], g[4 * h + 1], g[4 * h + 2],
                        g[4 * h + 3]);
          }
        }
      }
    }
    __syncthreads();  // the list is rewritten by the next batch
  }
  if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// chunk geometry of the fix-up grids
FixGeo fix_geo(int64_t V, int CL, int NT, int VPT, int SL) {
  FixGeo g;
  g.fw = NT / 32;
  g.np = CL * g.fw;
  g.fnt = NT;
  g.vpt = VPT;
  g.SL = SL;
  int64_t CH = (V + kOpdFixChunks - 1) / kOpdFixChunks;
  CH = (CH + 7) / 8 * 8;
  g.CH = static_cast<int32_t>(CH);
  g.nch = static_cast<int32_t>((V + CH - 1) / CH);
  return g;
}

// the fix-up grids after the fast kernel (CL CTAs of NT threads, VPT vectors
// per thread, slices of SL entries): which = kFixBoth (parts, then the
// gradient behind it), kFixParts, or kFixGradLast (the gradient grid behind
// the fused finalize, see FixGeo::wait_last)
template <int DT>
cudaError_t launch_fix(const OpdArgs &a, cudaStream_t st, int CL, int NT, int VPT, int SL, int which) {
  static std::atomic<int> nsm_cache[64];  // zero-initialised (static storage)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int nsm = (dev >= 0 && dev < 64) ? nsm_cache[dev].load(std::memory_order_relaxed) : 0;
  if (nsm == 0) {
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) nsm_cache[dev].store(nsm, std::memory_order_relaxed);
  }
  FixGeo fg = fix_geo(a.V, CL, NT, VPT, SL);
  fg.wait_last = (which == kFixGradLast) ? 1 : 0;
  // programmatic launches: each overlaps the tail of the kernel ahead of it
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(3 * nsm), 1, 1);
  cfg.blockDim = dim3(kFixNT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (which != kFixGradLast) {
    void *tm = timer_before("opd_fix_parts", st);
    e = cudaLaunchKernelEx(&cfg, opd_fix_parts<DT>, a, fg);
    timer_after(tm, st);
    if (e != cudaSuccess) return e;
  }
  if (which != kFixParts) {
    void *tm = timer_before("opd_fix_grad", st);
    e = cudaLaunchKernelEx(&cfg, opd_fix_grad<DT>, a, fg);
    timer_after(tm, st);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
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

constexpr int kTab = 1024;  // target-row table entries per cluster (beyond: binary search)

// what follows the two slices in dynamic shared memory
enum SmemTail { kNone, kTable };

// launch a persistent grid of clusters (as many as can be co-resident)
template <typename Kern>
cudaError_t launch_clusters(const char *name, Kern kern, int nt, const OpdArgs &a, const OpdPlan &p, SmemTail tail,
                            cudaStream_t st, int *grid_out = nullptr) {
  const size_t tail_max = (tail == kTable) ? kTab * sizeof(int32_t) : 0;
  const size_t smem_max = p.smem + tail_max;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(nt, 1, 1);
  cfg.dynamicSmemBytes = smem_max;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  struct Entry {
    int dev;
    const void *fn;
    int CL;
    size_t smem;
    int n;
  };
  static Entry cache[64];
  static int ncache = 0;
  static std::mutex mu;  // calls from several host threads share the cache
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int maxc = 0;
  std::unique_lock<std::mutex> lk(mu);
  for (int q = 0; q < ncache; ++q)
    if (cache[q].dev == dev && cache[q].fn == reinterpret_cast<const void *>(kern) && cache[q].CL == p.CL &&
        cache[q].smem == smem_max)
      maxc = cache[q].n;
  if (maxc == 0) {
    cfg.gridDim = dim3(p.CL * 1024, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (maxc <= 0) return cudaErrorInvalidConfiguration;
    if (ncache < 64) cache[ncache++] = Entry{dev, reinterpret_cast<const void *>(kern), p.CL, smem_max, maxc};
  }
  lk.unlock();
  const int64_t rows = (tail == kTable) ? a.R + a.nbonus : a.R;  // rows the kernel walks
  int64_t nclusters = maxc;
  if (nclusters > rows) nclusters = rows;
  OpdGeo geo;
  geo.SL = p.SL;
  geo.slice_bytes = p.slice_bytes;
  geo.ntab = 0;
  // target rows fit the int32 table when the target has fewer than 2^31 rows
  size_t tail_bytes = 0;
  if (tail == kTable && a.has_bonus && a.R + a.N < (int64_t{1} << 31)) {
    geo.ntab = static_cast<int32_t>(std::min<int64_t>((rows + nclusters - 1) / nclusters, kTab));
    tail_bytes = static_cast<size_t>(geo.ntab) * sizeof(int32_t);
  }
  cfg.dynamicSmemBytes = p.smem + tail_bytes;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * p.CL), 1, 1);
  if (grid_out) *grid_out = static_cast<int>(nclusters * p.CL);
  void *tm = timer_before(name, st);
  e = cudaLaunchKernelEx(&cfg, kern, a, geo);
  timer_after(tm, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// fast pass and / or fix-up with NT threads and up to VPT vectors per thread
template <int DT, int VPT, int NT>
cudaError_t launch_fast(const OpdArgs &a, const OpdPlan &p, cudaStream_t st, bool fast, int fix, int *grid) {
  if (fast) {
    const cudaError_t e = launch_clusters("opd_fast_kernel", opd_fast_kernel<DT, VPT, NT>, NT, a, p, kTable, st, grid);
    if (e != cudaSuccess || fix == kFixNone) return e;
  }
  return launch_fix<DT>(a, st, p.CL, NT, VPT, p.SL, fix);
}

// the fast-path variant for this row geometry; false if the row is too wide
template <int DT>
cudaError_t launch_fast_any(const OpdArgs &a, const OpdPlan &p, cudaStream_t st, bool fast, int fix, int *grid,
                            bool *ok) {
  const int nvec = static_cast<int>(static_cast<int64_t>(p.SL) * Elem<DT>::kSize / 16);
  *ok = true;
  if (nvec <= 512 * 1) return launch_fast<DT, 1, 512>(a, p, st, fast, fix, grid);
  if (nvec <= 512 * 2) return launch_fast<DT, 2, 512>(a, p, st, fast, fix, grid);
  if (nvec <= 512 * 3) return launch_fast<DT, 3, 512>(a, p, st, fast, fix, grid);
  if (nvec <= 256 * 10) return launch_fast<DT, 10, 256>(a, p, st, fast, fix, grid);
  *ok = false;
  return cudaErrorInvalidValue;
}

template <int DT, bool BULK>
cudaError_t launch_opd_cfg(const OpdArgs &a, const OpdPlan &p, cudaStream_t st) {
  if (BULK && a.flags != nullptr) {
    bool ok = false;
    const cudaError_t e = launch_fast_any<DT>(a, p, st, true, kFixBoth, nullptr, &ok);
    if (ok) return e;
  }
  return launch_clusters("opd_exact_kernel", opd_exact_kernel<DT, BULK>, 512, a, p, kNone, st);
}

}  // namespace

bool opd_supported(int64_t V, int esize) { return plan_opd(V, esize).smem <= 200 * 1024; }

int opd_cluster_size(int64_t V, int esize) { return plan_opd(V, esize).CL; }

bool opd_fast_supported(int64_t V, int esize) {
  const OpdPlan p = plan_opd(V, esize);
  return p.smem <= 200 * 1024 && static_cast<int64_t>(p.SL) * esize / 16 <= 256 * 10;
}

cudaError_t launch_opd_fused_fast(const OpdArgs &a, int dtype, int *grid, cudaStream_t st) {
  const int esize = (dtype == SVW_BF16) ? 2 : 4;
  const OpdPlan p = plan_opd(a.V, esize);
  bool ok = false;
  const cudaError_t e = (dtype == SVW_BF16) ? launch_fast_any<1>(a, p, st, true, kFixNone, grid, &ok)
                                            : launch_fast_any<0>(a, p, st, true, kFixNone, grid, &ok);
  return ok ? e : cudaErrorInvalidValue;
}

cudaError_t launch_opd_fix(const OpdArgs &a, int dtype, int which, cudaStream_t st) {
  const int esize = (dtype == SVW_BF16) ? 2 : 4;
  const OpdPlan p = plan_opd(a.V, esize);
  bool ok = false;
  const cudaError_t e = (dtype == SVW_BF16) ? launch_fast_any<1>(a, p, st, false, which, nullptr, &ok)
                                            : launch_fast_any<0>(a, p, st, false, which, nullptr, &ok);
  return ok ? e : cudaErrorInvalidValue;
}

cudaError_t launch_opd(const OpdArgs &a, int dtype, bool bulk, cudaStream_t st) {
  const int esize = (dtype == SVW_BF16) ? 2 : 4;
  const OpdPlan p = plan_opd(a.V, esize);
  if (p.smem > 200 * 1024) return cudaErrorInvalidValue;
  if (dtype == SVW_BF16) return bulk ? launch_opd_cfg<1, true>(a, p, st) : launch_opd_cfg<1, false>(a, p, st);
  return bulk ? launch_opd_cfg<0, true>(a, p, st) : launch_opd_cfg<0, false>(a, p, st);
}

}  // namespace svw
