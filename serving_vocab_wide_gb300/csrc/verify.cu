// verify.cu -- batched speculative verification on sm_103a.
//
// Method ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.1, §5.2 eqs. (6)-(8),
// Algorithm 1; "AdaFlash: Taming Variance in Diffusion Speculative Decoding",
// "Speculative Decoding: The Basic Idea" steps 3-4):
//   accept x_j iff u_j < min(1, p_j(x_j)/q_j(x_j)); keep the leftmost-rejection
//   prefix; draw one token from [p - q]_+ at the rejected row or from p at the
//   bonus row.  Greedy (T = 0): accept iff x_j is the target argmax.
//
// GPU design: four stream-ordered kernels, no CTA ever waits for another.
//  1. verify_prologue   validates CSR offsets and tokens, resets the sampler's
//                       arrival counters, writes the -1 defaults.
//  2. verify_stats      the HBM stream.  Each logit row is cut into C chunks
//                       (C <= 32, ~30 KB); a (row, chunk) pair is a work item.
//                       Persistent CTAs take items in a fixed stride.  One
//                       producer warp streams each chunk into a 4-stage
//                       shared-memory ring with 1-D bulk async copies
//                       (cp.async.bulk, full/empty mbarriers); eight consumer
//                       warps reduce their share of the chunk to
//                       (max, sum 2^((x - max) log2e/T)) -- or (max, argmax)
//                       when greedy -- with packed bf16 max and f32x2
//                       arithmetic, and write one Partial per warp.  No block
//                       barrier in the steady state.
//  3. verify_finalize   one CTA per request: merges the partials into row
//                       log-sum-exps (or argmaxes), runs every accept test in
//                       one warp (ballot + ffs = leftmost rejection), writes
//                       accept_len and the sampling row (greedy: next_token).
//  4. verify_sample     (T > 0) inverse-CDF draw over the sampling row (pair),
//                       split into 4096-entry sampler chunks so the whole GPU
//                       takes part; the CTA that completes a request's chunks
//                       (arrival counter) resolves the token.
//
// Inverse-CDF prefix sums.  Weights w_v = [p_v - q_v]_+ (or p_v).  The prefix
// C_v is defined level by level, each level a sequential fp32 sum (from 0, in
// index order) of non-negative terms, so that it is reproducible,
// non-decreasing and equal at every level boundary:
//   group  8 consecutive entries           partial sums part_k, total a_g
//   lane   2 consecutive groups            running R, total T_l
//   warp   32 lanes                        prefix E_l, total W_w
//   chunk  8 warps (4096 entries)          prefix P_w, total Z_c
//   row    chunks                          prefix B_c, total Z
//   C_v = fl(B_c + fl(P_w + fl(E_l + fl(R + part_k))))
// next = smallest v with C_v > w Z; that v always has w_v > 0.  If rounding
// leaves no crossing, the last positive entry is taken.
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace svw {

namespace {

constexpr int kCW = 8;                         // consumer warps of the stats kernel
constexpr int kStatsThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kStages = 3;                     // bulk-copy ring depth (2 CTAs per SM)
constexpr int kThreads = 256;                  // finalize / sample kernels
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 2 * SVW_MAX_LEN + 1;
constexpr int kMaxGroupsPerSpan = 512;  // single-CTA fallback sampler: V <= 256 * 512 * 8

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
// work items of the stats stream
// ---------------------------------------------------------------------------
struct ItemMeta {
  int64_t item;  // < 0: no more work
  int64_t prow;  // partial row index (target rows, then draft rows)
  const char *src;
  int32_t chunk;
  int32_t n;  // elements in this chunk
  int32_t valid;
  int32_t pad;
};

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

// items are numbered request-major: request i owns C * (L_i + 1) (greedy) or
// C * (2 L_i + 1) consecutive items; within a request, target rows 0..L_i come
// first, then draft rows 0..L_i-1.
template <int DT, bool GREEDY>
__device__ __forceinline__ ItemMeta decode_item(const VerifyArgs &a, int64_t item) {
  using E = Elem<DT>;
  ItemMeta m;
  m.item = item;
  const int32_t i = find_request<GREEDY>(a, item);
  const int64_t c_i = __ldg(a.cu + i);
  const int32_t L = __ldg(a.cu + i + 1) - static_cast<int32_t>(c_i);
  const int64_t off = static_cast<int64_t>(a.C) * (GREEDY ? (c_i + i) : (2 * c_i + i));
  const int64_t local = item - off;
  const int32_t rl = static_cast<int32_t>(local / a.C);
  m.chunk = static_cast<int32_t>(local - static_cast<int64_t>(rl) * a.C);
  const int64_t c0 = static_cast<int64_t>(m.chunk) * a.chunk_len;
  m.n = static_cast<int32_t>(min(static_cast<int64_t>(a.chunk_len), a.V - c0));
  const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
  m.valid = (a.req_ok[i] != 0 && rl < nrows) ? 1 : 0;
  const char *row;
  if (GREEDY || rl <= L) {
    m.prow = c_i + i + rl;
    row = static_cast<const char *>(a.target) + m.prow * a.V * E::kSize;
  } else {
    const int64_t dr = c_i + (rl - L - 1);
    m.prow = a.rows_t + dr;
    row = static_cast<const char *>(a.draft) + dr * a.V * E::kSize;
  }
  m.src = row + c0 * E::kSize;
  return m;
}

// ---------------------------------------------------------------------------
// consumer-warp reductions over one chunk held in shared memory (16-byte
// vectors vi = wid*32 + lane + j*256 of the chunk)
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void warp_lse_smem(uint32_t base, int nvec, int wid, int lane, float k,
                                              float &m, float &s) {
  const int v0 = wid * 32 + lane;
  float mx = -INFINITY;
  if (DT == 1) {
    uint32_t mw = 0xff80ff80u;  // (-inf, -inf)
    for (int vi = v0; vi < nvec; vi += kCW * 32) {
      const uint4 q = lds128(base + vi * 16);
      mw = bf16x2_max(mw, bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w)));
    }
    const float2 f = bf16x2_f2(mw);
    mx = fmaxf(f.x, f.y);
  } else {
    for (int vi = v0; vi < nvec; vi += kCW * 32) {
      const uint4 q = lds128(base + vi * 16);
      mx = fmaxf(fmaxf(mx, fmaxf(__uint_as_float(q.x), __uint_as_float(q.y))),
                 fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
  }
  // one reference for the whole warp, so the lane sums add directly
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  const float2 nm = make_float2(-mref, -mref), kk = make_float2(k, k);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
  for (int vi = v0; vi < nvec; vi += kCW * 32) {
    const uint4 q = lds128(base + vi * 16);
    if (DT == 1) {
      const float2 d0 = __fmul2_rn(__fadd2_rn(bf16x2_f2(q.x), nm), kk);  // (x - max) exact, then * log2e/T
      const float2 d1 = __fmul2_rn(__fadd2_rn(bf16x2_f2(q.y), nm), kk);
      const float2 d2 = __fmul2_rn(__fadd2_rn(bf16x2_f2(q.z), nm), kk);
      const float2 d3 = __fmul2_rn(__fadd2_rn(bf16x2_f2(q.w), nm), kk);
      acc0 = __fadd2_rn(acc0, __fadd2_rn(make_float2(ex2(d0.x), ex2(d0.y)), make_float2(ex2(d1.x), ex2(d1.y))));
      acc1 = __fadd2_rn(acc1, __fadd2_rn(make_float2(ex2(d2.x), ex2(d2.y)), make_float2(ex2(d3.x), ex2(d3.y))));
    } else {
      const float2 d0 = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(q.x), __uint_as_float(q.y)), nm), kk);
      const float2 d1 = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(q.z), __uint_as_float(q.w)), nm), kk);
      acc0 = __fadd2_rn(acc0, make_float2(ex2(d0.x), ex2(d0.y)));
      acc1 = __fadd2_rn(acc1, make_float2(ex2(d1.x), ex2(d1.y)));
    }
  }
  const float2 acc = __fadd2_rn(acc0, acc1);
  s = warp_sum(__fadd_rn(acc.x, acc.y));
  m = mx;
  if (!(mx == mx)) s = mx;  // all-NaN warp: keep the NaN visible
}

template <int DT>
__device__ __forceinline__ void warp_amax_smem(uint32_t base, int nvec, int32_t c0, int wid, int lane,
                                               float &best, int32_t &idx, int32_t &nan) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  const int v0 = wid * 32 + lane;
  float mx = -INFINITY;
  uint32_t nanw = 0;
  if (DT == 1) {
    uint32_t mw = 0xff80ff80u;  // NaN-propagating max: a NaN anywhere survives
    for (int vi = v0; vi < nvec; vi += kCW * 32) {
      const uint4 q = lds128(base + vi * 16);
      mw = bf16x2_max_nan(mw, bf16x2_max_nan(bf16x2_max_nan(q.x, q.y), bf16x2_max_nan(q.z, q.w)));
    }
    nanw = bf16x2_nan(mw);
    const float2 f = bf16x2_f2(mw);
    mx = fmaxf(f.x, f.y);
  } else {
    for (int vi = v0; vi < nvec; vi += kCW * 32) {
      const uint4 q = lds128(base + vi * 16);
      const float x[4] = {__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z),
                          __uint_as_float(q.w)};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        nanw |= (x[e] != x[e]);
        mx = fmaxf(mx, x[e]);
      }
    }
  }
  float wmx = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wmx = fmaxf(wmx, __shfl_xor_sync(0xffffffffu, wmx, o));
  // only lanes holding the warp maximum look for its first index
  // (each lane's vectors are in index order, lanes interleave by vector)
  idx = INT32_MAX;
  if (mx == wmx && nvec > 0) {
    for (int vi = v0; vi < nvec && idx == INT32_MAX; vi += kCW * 32) {
      float x[EPV];
      E::unpack(lds128(base + vi * 16), x);
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        if (idx == INT32_MAX && x[e] == wmx) idx = c0 + vi * EPV + e;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
  best = wmx;
  nan = __any_sync(0xffffffffu, nanw != 0) ? 1 : 0;
}

// plain-load variants for rows that are not 16-byte pitched (whole warp,
// elements v = wid*32 + lane + j*256 of the chunk)
template <int DT>
__device__ __forceinline__ void warp_lse_global(const char *p0, int n, int wid, int lane, float k, float &m,
                                                float &s) {
  using E = Elem<DT>;
  float mx = -INFINITY;
  for (int v = wid * 32 + lane; v < n; v += kCW * 32) mx = fmaxf(mx, E::load(p0, v));
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  float acc = 0.f;
  for (int v = wid * 32 + lane; v < n; v += kCW * 32)
    acc = __fadd_rn(acc, ex2(__fmul_rn(__fsub_rn(E::load(p0, v), mref), k)));
  m = -INFINITY;
  s = 0.f;
  lse_combine(m, s, mx, acc, k);
  warp_lse(m, s, k);
}

template <int DT>
__device__ __forceinline__ void warp_amax_global(const char *p0, int n, int32_t c0, int wid, int lane,
                                                 float &best, int32_t &idx, int32_t &nan) {
  using E = Elem<DT>;
  best = -INFINITY;
  idx = INT32_MAX;
  nan = 0;
  for (int v = wid * 32 + lane; v < n; v += kCW * 32) {
    const float x = E::load(p0, v);
    nan |= (x != x);
    if (x > best || (idx == INT32_MAX && x == x)) {
      best = x;
      idx = c0 + v;
    }
  }
  warp_amax(best, idx);
  nan = __any_sync(0xffffffffu, nan);
}

// ---------------------------------------------------------------------------
// kernel 2: stats stream
// ---------------------------------------------------------------------------
template <int DT, bool BULK, bool GREEDY>
__global__ void __launch_bounds__(kStatsThreads, 2) verify_stats(VerifyArgs a, int stage_bytes) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ unsigned long long full[kStages], empty[kStages];
  __shared__ ItemMeta meta[kStages];
  if (*a.global_ok == 0) return;  // inconsistent CSR offsets: nothing may be read
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;

  if (!BULK) {
    // plain loads: every warp walks the CTA's items itself (no producer)
    if (wid == kCW) return;
    for (int64_t item = blockIdx.x; item < a.total_items; item += G) {
      const ItemMeta m = decode_item<DT, GREEDY>(a, item);
      if (!m.valid) continue;
      Partial res;
      if (GREEDY) {
        warp_amax_global<DT>(m.src, m.n, m.chunk * a.chunk_len, wid, lane, res.m, res.idx, res.nan);
        res.s = 0.f;
      } else {
        warp_lse_global<DT>(m.src, m.n, wid, lane, a.k, res.m, res.s);
        res.idx = 0;
        res.nan = 0;
      }
      if (lane == 0) a.part[(m.prow * a.C + m.chunk) * kCW + wid] = res;
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (wid == kCW) {
    // ---------------- producer warp (one lane) ----------------
    if (lane != 0) return;
    int k = 0;
    for (int64_t item = blockIdx.x;; item += G, ++k) {
      const int s = k % kStages;
      if (k >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((k / kStages) - 1) & 1))) {
        // consumers stopped releasing stages: report, hand them an end marker
        if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        return;
      }
      if (item >= a.total_items) {
        meta[s].item = -1;
        mbar_arrive(&full[s]);
        return;
      }
      const ItemMeta m = decode_item<DT, GREEDY>(a, item);
      meta[s] = m;
      if (!m.valid) {
        mbar_arrive(&full[s]);
        continue;
      }
      const uint32_t bytes = static_cast<uint32_t>(m.n) * Elem<DT>::kSize;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&full[s], bytes);
      bulk_g2s(ring + static_cast<size_t>(s) * stage_bytes, m.src, bytes, &full[s]);
    }
  }

  // ---------------- consumer warps ----------------
  for (int k = 0;; ++k) {
    const int s = k % kStages;
    if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((k / kStages) & 1))) {
      if (lane == 0 && a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
      return;
    }
    const ItemMeta m = meta[s];
    if (m.item < 0) return;  // every later stage would be empty too
    if (m.valid) {
      const uint32_t base = smem_u32(ring + static_cast<size_t>(s) * stage_bytes);
      const int nvec = m.n / Elem<DT>::kPerVec;
      Partial res;
      if (GREEDY) {
        warp_amax_smem<DT>(base, nvec, m.chunk * a.chunk_len, wid, lane, res.m, res.idx, res.nan);
        res.s = 0.f;
      } else {
        warp_lse_smem<DT>(base, nvec, wid, lane, a.k, res.m, res.s);
        res.idx = 0;
        res.nan = 0;
      }
      if (lane == 0) a.part[(m.prow * a.C + m.chunk) * kCW + wid] = res;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// ---------------------------------------------------------------------------
// kernel 3: per-request merge + accept tests
// ---------------------------------------------------------------------------
template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads) verify_finalize(VerifyArgs a) {
  using E = Elem<DT>;
  __shared__ float row_m[kMaxRows];
  __shared__ float row_l[kMaxRows];
  __shared__ int32_t row_idx[kMaxRows];
  __shared__ int32_t row_bad[kMaxRows];
  if (*a.global_ok == 0) return;
  const int32_t i = blockIdx.x;
  if (!a.req_ok[i]) return;  // outputs keep the -1 defaults
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c_i = __ldg(a.cu + i);
  const int32_t L = __ldg(a.cu + i + 1) - static_cast<int32_t>(c_i);
  const int64_t t0 = c_i + i, d0 = c_i;
  const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
  const int np = a.C * kCW;  // partials per row
  for (int r = warp; r < nrows; r += kWarps) {
    const int64_t prow = (r <= L) ? (t0 + r) : (a.rows_t + d0 + (r - L - 1));
    const Partial *pp = a.part + prow * np;
    if (GREEDY) {
      float v = -INFINITY;
      int32_t idx = INT32_MAX, nan = 0;
      for (int p = lane; p < np; p += 32) {
        const Partial q = ldcg_partial(pp + p);
        amax_combine(v, idx, q.m, q.idx);
        nan |= q.nan;
      }
      warp_amax(v, idx);
      nan = __any_sync(0xffffffffu, nan);
      if (lane == 0) {
        row_idx[r] = idx;
        row_bad[r] = nan;
      }
    } else {
      float mm = -INFINITY, s = 0.f;
      for (int p = lane; p < np; p += 32) {
        const Partial q = ldcg_partial(pp + p);
        lse_combine(mm, s, q.m, q.s, a.k);
      }
      warp_lse(mm, s, a.k);
      if (lane == 0) {
        row_m[r] = mm;
        row_l[r] = lg2(s);
        row_bad[r] = !(s > 0.f && s <= FLT_MAX);
      }
    }
  }
  __syncthreads();
  if (warp != 0) return;
  int bad = 0;
  for (int r = lane; r < nrows; r += 32) bad |= row_bad[r];
  bad = __any_sync(0xffffffffu, bad);
  bool acc = true;
  if (lane < L) {
    const int32_t x = __ldg(a.tokens + d0 + lane);
    if (GREEDY) {
      acc = (x == row_idx[lane]);
    } else {
      // log2(p(x)/q(x)) from raw logits and row log-sum-exps
      const float yx = E::load(a.target, (t0 + lane) * a.V + x);
      const float zx = E::load(a.draft, (d0 + lane) * a.V + x);
      float thr;
      if (zx == -INFINITY) {
        thr = 1.f;  // q(x) = 0: accept
      } else {
        const float dl = __fsub_rn(
            __fmul_rn(__fsub_rn(__fsub_rn(yx, row_m[lane]), __fsub_rn(zx, row_m[L + 1 + lane])), a.k),
            __fsub_rn(row_l[lane], row_l[L + 1 + lane]));
        thr = (dl >= 0.f) ? 1.f : ex2(dl);
      }
      const float u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(lane), 0u);
      acc = (u < thr);
    }
  }
  const unsigned rej = __ballot_sync(0xffffffffu, !acc);
  const int32_t js = rej ? (__ffs(rej) - 1) : L;
  if (lane != 0) return;
  if (bad) {
    if (a.status) atomicOr(a.status, SVW_DEV_BAD_INPUT);
    return;
  }
  a.accept_len[i] = js;
  if (GREEDY) {
    a.next_token[i] = row_idx[js];
  } else {
    SampleInfo si;
    si.js = js;
    si.resid = (js < L) ? 1 : 0;
    si.valid = 1;
    si.w = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(js), 1u);
    si.Mt = row_m[js];
    si.lt = row_l[js];
    si.Md = (js < L) ? row_m[L + 1 + js] : 0.f;
    si.ld = (js < L) ? row_l[L + 1 + js] : 0.f;
    a.sinfo[i] = si;
  }
}

// ---------------------------------------------------------------------------
// sampling weights
// ---------------------------------------------------------------------------
struct RowConst {
  float Mt, lt, Md, ld, k;
};

// [p - q]_+ (resid) or p, from raw logits and the row constants
__device__ __forceinline__ float weight(float y, float z, bool resid, const RowConst &c) {
  const float lp = __fsub_rn(__fmul_rn(__fsub_rn(y, c.Mt), c.k), c.lt);  // log2 p
  if (!resid) return ex2(lp);
  const float lq = __fsub_rn(__fmul_rn(__fsub_rn(z, c.Md), c.k), c.ld);  // log2 q
  if (!(lq < lp)) return 0.f;
  return fmaxf(__fsub_rn(ex2(lp), ex2(lq)), 0.f);
}

// raw logits of group g (entries 8g .. 8g+7, -inf at v >= V)
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

// the 8 weights of group g and their sequential sum a_g
template <int DT, bool VEC>
__device__ __forceinline__ float group_weights(const char *trow, const char *drow, bool resid, int64_t g,
                                               int64_t V, const RowConst &c, float (&w)[8]) {
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

struct SampleSmem {
  float lane_tot[kThreads];
  float E[kThreads + 1];
  int32_t lastv[kThreads];
  float grp[kMaxGroupsPerSpan];
  float chunk_tot[1024];
  float warp_tot[kWarps];
  int32_t is_last;
  int32_t cstar;
  int32_t result;
  int32_t degenerate;
  float t;
  float Bc;
  float Pw;
  float El;
  int32_t wstar;
  int32_t lstar;
};

// Single-CTA inverse CDF over a whole row of p.  Used only when a rejected
// row has no residual mass after rounding; its prefix is defined with 256
// thread spans (sequential within and across spans).
template <int DT, bool VEC>
__device__ __noinline__ int32_t sample_whole_row_p(const char *trow, int64_t V, const RowConst &c, float wu,
                                                   SampleSmem &sm) {
  const int tid = threadIdx.x;
  const int64_t NG = (V + 7) / 8;
  const int64_t GPT = (NG + kThreads - 1) / kThreads;
  const int64_t g0 = min(NG, static_cast<int64_t>(tid) * GPT), g1 = min(NG, g0 + GPT);
  float R = 0.f;
  int32_t last = -1;
  for (int64_t g = g0; g < g1; ++g) {
    float w[8];
    R = __fadd_rn(R, group_weights<DT, VEC>(trow, nullptr, false, g, V, c, w));
    for (int e = 0; e < 8; ++e)
      if (w[e] > 0.f) last = static_cast<int32_t>(g * 8 + e);
  }
  sm.lane_tot[tid] = R;
  sm.lastv[tid] = last;
  __syncthreads();
  if (tid == 0) {
    float E = 0.f;
    sm.E[0] = 0.f;
    for (int s = 0; s < kThreads; ++s) {
      E = __fadd_rn(E, sm.lane_tot[s]);
      sm.E[s + 1] = E;
    }
    sm.t = __fmul_rn(wu, E);
    sm.lstar = INT32_MAX;
  }
  __syncthreads();
  const float t = sm.t;
  if (sm.E[tid + 1] > t) atomicMin(&sm.lstar, tid);
  __syncthreads();
  const int32_t ts = sm.lstar;
  if (ts == INT32_MAX) {
    if (tid == 0) {
      int32_t lv = -1;
      for (int s = 0; s < kThreads; ++s) lv = max(lv, sm.lastv[s]);
      sm.result = lv;
    }
    __syncthreads();
    return sm.result;
  }
  const int64_t h0 = min(NG, static_cast<int64_t>(ts) * GPT), h1 = min(NG, h0 + GPT);
  for (int64_t g = h0 + tid; g < h1; g += kThreads) {
    float w[8];
    sm.grp[g - h0] = group_weights<DT, VEC>(trow, nullptr, false, g, V, c, w);
  }
  __syncthreads();
  if (tid == 0) {
    const float Es = sm.E[ts];
    float Rr = 0.f;
    int32_t pick = -1;
    for (int64_t g = h0; g < h1 && pick < 0; ++g) {
      const float R2 = __fadd_rn(Rr, sm.grp[g - h0]);
      if (__fadd_rn(Es, R2) > t) {
        float w[8];
        group_weights<DT, VEC>(trow, nullptr, false, g, V, c, w);
        float part = 0.f;
        for (int e = 0; e < 8; ++e) {
          part = __fadd_rn(part, w[e]);
          if (__fadd_rn(Es, __fadd_rn(Rr, part)) > t) {
            pick = static_cast<int32_t>(g * 8 + e);
            break;
          }
        }
      }
      Rr = R2;
    }
    sm.result = (pick < 0) ? sm.lastv[ts] : pick;
  }
  __syncthreads();
  return sm.result;
}

// ---------------------------------------------------------------------------
// kernel 4: inverse-CDF sampling over (request, sampler chunk) items
// ---------------------------------------------------------------------------
constexpr int kGPL = 2;                               // groups per lane
constexpr int kSChunk = kThreads * kGPL * 8;          // 4096 entries per sampler chunk

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) verify_sample(VerifyArgs a) {
  using E = Elem<DT>;
  __shared__ SampleSmem sm;
  if (*a.global_ok == 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t Cs = a.Cs;
  // last requests first: their rows were streamed most recently
  const int64_t item = static_cast<int64_t>(a.N) * Cs - 1 - blockIdx.x;
  const int32_t i = static_cast<int32_t>(item / Cs);
  const int32_t c = static_cast<int32_t>(item - static_cast<int64_t>(i) * Cs);
  const SampleInfo si = a.sinfo[i];
  if (!si.valid) return;
  const int64_t ci = __ldg(a.cu + i);
  const char *trow = static_cast<const char *>(a.target) + (ci + i + si.js) * a.V * E::kSize;
  const bool resid = si.resid != 0;
  const char *drow = resid ? static_cast<const char *>(a.draft) + (ci + si.js) * a.V * E::kSize : nullptr;
  RowConst rc;
  rc.Mt = si.Mt;
  rc.lt = si.lt;
  rc.Md = si.Md;
  rc.ld = si.ld;
  rc.k = a.k;
  const int64_t NG = (a.V + 7) / 8;

  // ---- this chunk: lane totals, warp totals, chunk total ----
  const int64_t g0 = static_cast<int64_t>(c) * (kSChunk / 8) + static_cast<int64_t>(tid) * kGPL;
  float a_g[kGPL];
  int32_t last = -1;
  {
    float w[kGPL][8];
#pragma unroll
    for (int u = 0; u < kGPL; ++u)
      a_g[u] = (g0 + u < NG) ? group_weights<DT, VEC>(trow, drow, resid, g0 + u, a.V, rc, w[u]) : 0.f;
#pragma unroll
    for (int u = 0; u < kGPL; ++u)
      if (g0 + u < NG) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (w[u][e] > 0.f) last = static_cast<int32_t>((g0 + u) * 8 + e);
      }
  }
  float T = 0.f;
#pragma unroll
  for (int u = 0; u < kGPL; ++u) T = __fadd_rn(T, a_g[u]);
  const int64_t slot = static_cast<int64_t>(i) * Cs + c;
  a.span_tot[slot * kThreads + tid] = T;
  // warp total: sequential over lanes 0..31
  float W = 0.f;
  for (int l = 0; l < 32; ++l) W = __fadd_rn(W, __shfl_sync(0xffffffffu, T, l));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0) {
    sm.warp_tot[warp] = W;
    sm.lastv[warp] = last;
  }
  __syncthreads();
  if (tid == 0) {
    float Z = 0.f;
    int32_t lv = -1;
    for (int w = 0; w < kWarps; ++w) {
      Z = __fadd_rn(Z, sm.warp_tot[w]);
      lv = max(lv, sm.lastv[w]);
    }
    a.chunk_tot[slot] = Z;
    a.chunk_last[slot] = lv;
    __threadfence();
    const int32_t prev = atomicAdd(a.sample_counters + i, 1);
    sm.is_last = (prev == Cs - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.is_last) return;
  __threadfence();

  // ---- resolve (the CTA that completed request i) ----
  for (int q = tid; q < Cs; q += kThreads) sm.chunk_tot[q] = __ldcg(a.chunk_tot + static_cast<int64_t>(i) * Cs + q);
  __syncthreads();
  if (tid == 0) {
    float B = 0.f;
    for (int q = 0; q < Cs; ++q) B = __fadd_rn(B, sm.chunk_tot[q]);
    const float t = __fmul_rn(si.w, B);
    sm.t = t;
    sm.degenerate = (resid && !(B > 0.f)) ? 1 : 0;
    int32_t cs = -1;
    float Bc = 0.f, Bp = 0.f;
    for (int q = 0; q < Cs && cs < 0; ++q) {
      Bp = Bc;
      Bc = __fadd_rn(Bc, sm.chunk_tot[q]);
      if (Bc > t) cs = q;
    }
    sm.cstar = cs;
    sm.Bc = Bp;  // prefix before the crossing chunk
  }
  __syncthreads();
  int32_t tok;
  if (sm.degenerate) {
    // no residual mass after rounding: draw from p at that row instead
    tok = sample_whole_row_p<DT, VEC>(trow, a.V, rc, si.w, sm);
  } else if (sm.cstar < 0) {
    // w Z rounded up to Z: the last entry with positive weight
    if (tid == 0) {
      int32_t lv = -1;
      for (int q = 0; q < Cs; ++q) lv = max(lv, __ldcg(a.chunk_last + static_cast<int64_t>(i) * Cs + q));
      sm.result = lv;
    }
    __syncthreads();
    tok = sm.result;
  } else {
    const int32_t cs = sm.cstar;
    sm.lane_tot[tid] = __ldcg(a.span_tot + (static_cast<int64_t>(i) * Cs + cs) * kThreads + tid);
    __syncthreads();
    if (tid == 0) {
      const float t = sm.t, B = sm.Bc;
      // warp level
      float P = 0.f;
      int32_t ws = -1;
      float Pw = 0.f;
      for (int w = 0; w < kWarps && ws < 0; ++w) {
        float Ww = 0.f;
        for (int l = 0; l < 32; ++l) Ww = __fadd_rn(Ww, sm.lane_tot[w * 32 + l]);
        const float P2 = __fadd_rn(P, Ww);
        if (__fadd_rn(B, P2) > t) {
          ws = w;
          Pw = P;
        }
        P = P2;
      }
      // lane level
      int32_t ls = -1;
      float El = 0.f;
      if (ws >= 0) {
        float Ecur = 0.f;
        for (int l = 0; l < 32 && ls < 0; ++l) {
          const float E2 = __fadd_rn(Ecur, sm.lane_tot[ws * 32 + l]);
          if (__fadd_rn(B, __fadd_rn(Pw, E2)) > t) {
            ls = l;
            El = Ecur;
          }
          Ecur = E2;
        }
      }
      // group and entry level
      int32_t pick = -1;
      if (ls >= 0) {
        const int64_t gg0 = static_cast<int64_t>(cs) * (kSChunk / 8) + static_cast<int64_t>(ws * 32 + ls) * kGPL;
        float R = 0.f;
        for (int u = 0; u < kGPL && pick < 0; ++u) {
          if (gg0 + u >= NG) break;
          float w[8];
          const float ag = group_weights<DT, VEC>(trow, drow, resid, gg0 + u, a.V, rc, w);
          const float R2 = __fadd_rn(R, ag);
          if (__fadd_rn(B, __fadd_rn(Pw, __fadd_rn(El, R2))) > t) {
            float part = 0.f;
            for (int e = 0; e < 8; ++e) {
              part = __fadd_rn(part, w[e]);
              if (__fadd_rn(B, __fadd_rn(Pw, __fadd_rn(El, __fadd_rn(R, part)))) > t) {
                pick = static_cast<int32_t>((gg0 + u) * 8 + e);
                break;
              }
            }
          }
          R = R2;
        }
      }
      if (pick < 0) pick = __ldcg(a.chunk_last + static_cast<int64_t>(i) * Cs + cs);  // unreachable
      sm.result = pick;
    }
    __syncthreads();
    tok = sm.result;
  }
  if (tid == 0) a.next_token[i] = tok;
}

// ---------------------------------------------------------------------------
// kernel 1: prologue
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) verify_prologue(VerifyArgs a) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int bad = 0;
  if (threadIdx.x == 0 && (__ldg(a.cu) != 0 || static_cast<int64_t>(__ldg(a.cu + a.N)) != a.total_rows))
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
    a.sample_counters[i] = 0;
    a.sinfo[i].valid = 0;
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

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
struct GridCache {
  int dev;
  const void *fn;
  int smem;
  int blocks;
};

int cached_grid(const void *fn, int threads, int smem, cudaError_t &e) {
  static GridCache cache[64];
  static int n = 0;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return 0;
  for (int q = 0; q < n; ++q)
    if (cache[q].dev == dev && cache[q].fn == fn && cache[q].smem == smem) return cache[q].blocks;
  int nsm = 0, occ = 0;
  e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem);
  if (e != cudaSuccess) return 0;
  const int blocks = nsm * (occ > 0 ? occ : 1);
  if (n < 64) cache[n++] = GridCache{dev, fn, smem, blocks};
  return blocks;
}

template <int DT, bool VEC, bool GREEDY>
cudaError_t launch_all_t(const VerifyArgs &a, cudaStream_t st) {
  using E = Elem<DT>;
  const int stage_bytes = VEC ? (a.chunk_len * E::kSize + 127) / 128 * 128 : 0;
  const int smem = VEC ? kStages * stage_bytes : 0;
  auto fn = verify_stats<DT, VEC, GREEDY>;
  cudaError_t e = cudaSuccess;
  if (VEC) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  int grid = cached_grid(reinterpret_cast<const void *>(fn), kStatsThreads, smem, e);
  if (e != cudaSuccess) return e;
  if (grid > a.total_items) grid = static_cast<int>(a.total_items);
  fn<<<grid, kStatsThreads, smem, st>>>(a, stage_bytes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  verify_finalize<DT, GREEDY><<<a.N, kThreads, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || GREEDY) return e;
  verify_sample<DT, VEC><<<static_cast<unsigned>(static_cast<int64_t>(a.N) * a.Cs), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int DT, bool VEC>
cudaError_t launch_all(const VerifyArgs &a, bool greedy, cudaStream_t st) {
  return greedy ? launch_all_t<DT, VEC, true>(a, st) : launch_all_t<DT, VEC, false>(a, st);
}

}  // namespace

int32_t sampler_chunks(int64_t V) { return static_cast<int32_t>((V + kSChunk - 1) / kSChunk); }

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
  const size_t Cs = static_cast<size_t>(sampler_chunks(V));
  VerifyLayout l;
  const size_t rows = static_cast<size_t>(total_rows + N) + static_cast<size_t>(total_rows);
  const size_t ns = static_cast<size_t>(N) * Cs;
  size_t off = 0;
  l.part_off = off;
  off += align256(rows * static_cast<size_t>(p.C) * kCW * sizeof(Partial));
  l.sample_counters_off = off;
  off += align256(static_cast<size_t>(N) * 4);
  l.req_ok_off = off;
  off += align256(static_cast<size_t>(N) * 4);
  l.sinfo_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(SampleInfo));
  l.span_off = off;
  off += align256(ns * kThreads * sizeof(float));
  l.chunk_tot_off = off;
  off += align256(ns * sizeof(float));
  l.chunk_last_off = off;
  off += align256(ns * sizeof(int32_t));
  l.global_ok_off = off;
  off += 256;
  l.total = off;
  return l;
}

cudaError_t launch_verify(const VerifyArgs &a, int dtype, bool vec, bool greedy, cudaStream_t st) {
  verify_prologue<<<1, 1024, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dtype == SVW_BF16) return vec ? launch_all<1, true>(a, greedy, st) : launch_all<1, false>(a, greedy, st);
  return vec ? launch_all<0, true>(a, greedy, st) : launch_all<0, false>(a, greedy, st);
}

}  // namespace svw
