// verify.cu -- batched speculative verification on sm_103a.
//
// Method ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.1, §5.2 eqs. (6)-(8),
// Algorithm 1; "AdaFlash: Taming Variance in Diffusion Speculative Decoding",
// "Speculative Decoding: The Basic Idea" steps 3-4):
//   accept x_j iff u_j < min(1, p_j(x_j)/q_j(x_j)); keep the leftmost-rejection
//   prefix; draw one token from [p - q]_+ at the rejected row or from p at the
//   bonus row.  Greedy (T = 0): accept iff x_j is the target argmax.
//
// GPU design: two stream-ordered kernels; no CTA ever waits for another.
//  1. verify_stats      the HBM stream.  Each logit row is cut into C chunks
//                       (C <= 32, ~30 KB); a (row, chunk) pair is a work item.
//                       Persistent CTAs take items in a fixed stride.  One
//                       producer warp streams each chunk into a 3-stage
//                       shared-memory ring with 1-D bulk async copies
//                       (cp.async.bulk, full/empty mbarriers); 8 consumer (16
//                       when greedy) warps reduce their share of the chunk to
//                       (max, sum 2^((x - max) log2e/T)) -- or (max, argmax)
//                       when greedy -- with packed bf16 max and f32x2
//                       arithmetic, and write one Partial per warp.  No block
//                       barrier in the steady state.  Each CTA also checks a
//                       share of the CSR offsets.
//  2. verify_finalize   one CTA per request (two per SM, so every request of
//                       a large batch is in flight at once): validates the
//                       request, merges the partials into row log-sum-exps
//                       (or argmaxes), runs every accept test in one warp
//                       (ballot + ffs = leftmost rejection), writes
//                       accept_len, then (T > 0) the whole CTA draws the next
//                       token by inverse CDF over the residual row pair or the
//                       bonus row (svw_sample.cuh), in one coalesced pass.
// The finalize kernel is launched as a programmatic dependent of the stats
// kernel: it is scheduled while the stream drains and reads the draft tokens
// and their logits before waiting (griddepcontrol.wait) for the partials.
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"
#include "svw_sample.cuh"

namespace svw {

namespace {

// consumer warps of the stats kernel: the argmax reduction is cheap per entry
// and latency-bound, so greedy mode takes twice the warps
constexpr int kCWMax = 16;
template <bool GREEDY>
struct StatsShape {
  static constexpr int kCW = GREEDY ? 16 : 8;
  static constexpr int kThreads = (kCW + 1) * 32;  // + one producer warp
};
constexpr int kStages = 3;                     // bulk-copy ring depth (2 CTAs per SM)
constexpr int kFinThreads = 512;               // finalize (and sampling) kernel, two CTAs per SM
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kMaxRows = 2 * SVW_MAX_LEN + 1;

// programmatic dependent launch: let the next kernel be scheduled / wait for
// the previous kernel's results
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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
  const int64_t c_e = __ldg(a.cu + i + 1);
  // requests the finalize kernel will reject are not read (this also keeps
  // every address in range when the offsets are inconsistent)
  const bool req_ok = (c_e - c_i >= 1 && c_e - c_i <= a.max_len && c_i >= 0 && c_e <= a.total_rows);
  const int32_t L = req_ok ? static_cast<int32_t>(c_e - c_i) : 0;
  const int64_t off = static_cast<int64_t>(a.C) * (GREEDY ? (c_i + i) : (2 * c_i + i));
  const int64_t local = item - off;
  const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
  m.valid = (req_ok && local >= 0 && local < static_cast<int64_t>(nrows) * a.C) ? 1 : 0;
  if (!m.valid) {
    m.prow = 0;
    m.src = nullptr;
    m.chunk = 0;
    m.n = 0;
    return m;
  }
  const int32_t rl = static_cast<int32_t>(local / a.C);
  m.chunk = static_cast<int32_t>(local - static_cast<int64_t>(rl) * a.C);
  const int64_t c0 = static_cast<int64_t>(m.chunk) * a.chunk_len;
  m.n = static_cast<int32_t>(min(static_cast<int64_t>(a.chunk_len), a.V - c0));
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
template <int DT, int CW>
__device__ __forceinline__ void warp_lse_smem(uint32_t base, int nvec, int wid, int lane, float k,
                                              float &m, float &s) {
  const int v0 = wid * 32 + lane;
  float mx = -INFINITY;
  if (DT == 1) {
    uint32_t mw = 0xff80ff80u;  // (-inf, -inf)
    for (int vi = v0; vi < nvec; vi += CW * 32) {
      const uint4 q = lds128(base + vi * 16);
      mw = bf16x2_max(mw, bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w)));
    }
    const float2 f = bf16x2_f2(mw);
    mx = fmaxf(f.x, f.y);
  } else {
    for (int vi = v0; vi < nvec; vi += CW * 32) {
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
  for (int vi = v0; vi < nvec; vi += CW * 32) {
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

template <int DT, int CW>
__device__ __forceinline__ void warp_amax_smem(uint32_t base, int nvec, int32_t c0, int wid, int lane,
                                               float &best, int32_t &idx, int32_t &nan) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  const int v0 = wid * 32 + lane;
  float mx = -INFINITY;
  int bvi = (v0 < nvec) ? v0 : -1;  // this lane's first vector holding its maximum (-inf rows: the first)
  uint32_t nanw = 0;
  if (DT == 1) {
    for (int vi = v0; vi < nvec; vi += CW * 32) {
      const uint4 q = lds128(base + vi * 16);
      // NaN-propagating max of the vector: a NaN anywhere survives
      const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(q.x, q.y), bf16x2_max_nan(q.z, q.w));
      nanw |= bf16x2_nan(m2);
      const float2 f = bf16x2_f2(m2);
      const float vm = fmaxf(f.x, f.y);
      if (vm > mx) {
        mx = vm;
        bvi = vi;
      }
    }
  } else {
    for (int vi = v0; vi < nvec; vi += CW * 32) {
      const uint4 q = lds128(base + vi * 16);
      const float x[4] = {__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z),
                          __uint_as_float(q.w)};
      float vm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        nanw |= (x[e] != x[e]);
        vm = fmaxf(vm, x[e]);
      }
      if (vm > mx) {
        mx = vm;
        bvi = vi;
      }
    }
  }
  float wmx = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wmx = fmaxf(wmx, __shfl_xor_sync(0xffffffffu, wmx, o));
  // only lanes holding the warp maximum look for its first index, in the
  // one vector where their maximum first appeared (each lane's vectors are in
  // index order, lanes interleave by vector)
  idx = INT32_MAX;
  if (mx == wmx && bvi >= 0) {
    float x[EPV];
    E::unpack(lds128(base + bvi * 16), x);
#pragma unroll
    for (int e = EPV - 1; e >= 0; --e)
      if (x[e] == wmx) idx = c0 + bvi * EPV + e;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
  best = wmx;
  nan = __any_sync(0xffffffffu, nanw != 0) ? 1 : 0;
}

template <int DT, int CW>
__device__ __forceinline__ void warp_lse_global(const char *p0, int n, int wid, int lane, float k, float &m,
                                                float &s) {
  using E = Elem<DT>;
  float mx = -INFINITY;
  for (int v = wid * 32 + lane; v < n; v += CW * 32) mx = fmaxf(mx, E::load(p0, v));
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  float acc = 0.f;
  for (int v = wid * 32 + lane; v < n; v += CW * 32)
    acc = __fadd_rn(acc, ex2(__fmul_rn(__fsub_rn(E::load(p0, v), mref), k)));
  m = -INFINITY;
  s = 0.f;
  lse_combine(m, s, mx, acc, k);
  warp_lse(m, s, k);
}

template <int DT, int CW>
__device__ __forceinline__ void warp_amax_global(const char *p0, int n, int32_t c0, int wid, int lane,
                                                 float &best, int32_t &idx, int32_t &nan) {
  using E = Elem<DT>;
  best = -INFINITY;
  idx = INT32_MAX;
  nan = 0;
  for (int v = wid * 32 + lane; v < n; v += CW * 32) {
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
__global__ void __launch_bounds__(StatsShape<GREEDY>::kThreads, 2) verify_stats(VerifyArgs a, int stage_bytes) {
  constexpr int kCW = StatsShape<GREEDY>::kCW;
  constexpr int kStatsThreads = StatsShape<GREEDY>::kThreads;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ unsigned long long full[kStages], empty[kStages];
  __shared__ ItemMeta meta[kStages];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  pdl_launch_dependents();  // the finalize grid may be scheduled now
  {
    // this CTA's share of the CSR consistency check: cu[0] = 0,
    // cu[N] = total rows, non-decreasing (the finalize kernel ORs the flags)
    int bad = 0;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kStatsThreads + threadIdx.x; j < a.N;
         j += G * kStatsThreads)
      bad |= (__ldg(a.cu + j) > __ldg(a.cu + j + 1)) ? 1 : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0)
      bad |= (__ldg(a.cu) != 0 || static_cast<int64_t>(__ldg(a.cu + a.N)) != a.total_rows) ? 1 : 0;
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) a.csr_bad[blockIdx.x] = bad;
  }

  if (!BULK) {
    // plain loads: every warp walks the CTA's items itself (no producer)
    if (wid == kCW) return;
    for (int64_t item = blockIdx.x; item < a.total_items; item += G) {
      const ItemMeta m = decode_item<DT, GREEDY>(a, item);
      if (!m.valid) continue;
      Partial res;
      if (GREEDY) {
        warp_amax_global<DT, kCW>(m.src, m.n, m.chunk * a.chunk_len, wid, lane, res.m, res.idx, res.nan);
        res.s = 0.f;
      } else {
        warp_lse_global<DT, kCW>(m.src, m.n, wid, lane, a.k, res.m, res.s);
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
        warp_amax_smem<DT, kCW>(base, nvec, m.chunk * a.chunk_len, wid, lane, res.m, res.idx, res.nan);
        res.s = 0.f;
      } else {
        warp_lse_smem<DT, kCW>(base, nvec, wid, lane, a.k, res.m, res.s);
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
// kernel 2: per-request validation, merge, accept tests
// ---------------------------------------------------------------------------
template <int DT, bool GREEDY, bool VEC>
__global__ void __launch_bounds__(kFinThreads) verify_finalize(VerifyArgs a) {
  using E = Elem<DT>;
  __shared__ float row_m[kMaxRows];
  __shared__ float row_l[kMaxRows];
  __shared__ int32_t row_idx[kMaxRows];
  __shared__ int32_t row_bad[kMaxRows];
  __shared__ int32_t s_ok, s_js;
  __shared__ SampleSmem<kFinThreads> ssm;
  const int32_t i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();

  // ---- inputs only: this part overlaps the end of the stats kernel ----
  const int64_t c_i = __ldg(a.cu + i), c_e = __ldg(a.cu + i + 1);
  const bool len_ok = (c_e - c_i >= 1 && c_e - c_i <= a.max_len && c_i >= 0 && c_e <= a.total_rows);
  const int32_t L = len_ok ? static_cast<int32_t>(c_e - c_i) : 0;
  const int64_t t0 = c_i + i, d0 = c_i;
  int32_t x = 0;
  float yx = 0.f, zx = 0.f, u = 0.f;
  if (warp == 0) {
    bool tok_ok = true;
    if (lane < L) {
      x = __ldg(a.tokens + d0 + lane);
      tok_ok = (x >= 0 && static_cast<int64_t>(x) < a.V);
      if (tok_ok && !GREEDY) {
        yx = E::load(a.target, (t0 + lane) * a.V + x);
        zx = E::load(a.draft, (d0 + lane) * a.V + x);
        u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(lane), 0u);
      }
    }
    const bool ok = len_ok && __all_sync(0xffffffffu, tok_ok);
    if (lane == 0) s_ok = ok ? 1 : 0;
  }
  pdl_wait();  // the stats kernel's partials and CSR flags are complete

  int csr_bad = 0;
  for (int b = tid; b < a.stats_grid; b += kFinThreads) csr_bad |= __ldcg(a.csr_bad + b);
  csr_bad = __syncthreads_or(csr_bad);
  auto reject = [&]() {  // one thread: a bad request
    a.accept_len[i] = -1;
    a.next_token[i] = -1;
    if (a.status) atomicOr(a.status, SVW_DEV_BAD_INPUT);
  };
  if (!s_ok || csr_bad) {
    if (tid == 0) reject();
    return;
  }
  const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
  const int np = a.C * StatsShape<GREEDY>::kCW;  // partials per row
  for (int r = warp; r < nrows; r += kFinWarps) {
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
  if (warp == 0) {
    int bad = 0;
    for (int r = lane; r < nrows; r += 32) bad |= row_bad[r];
    bad = __any_sync(0xffffffffu, bad);
    bool acc = true;
    if (lane < L) {
      if (GREEDY) {
        acc = (x == row_idx[lane]);
      } else {
        // log2(p(x)/q(x)) from raw logits and row log-sum-exps
        float thr;
        if (zx == -INFINITY) {
          thr = 1.f;  // q(x) = 0: accept
        } else {
          const float dl = __fsub_rn(
              __fmul_rn(__fsub_rn(__fsub_rn(yx, row_m[lane]), __fsub_rn(zx, row_m[L + 1 + lane])), a.k),
              __fsub_rn(row_l[lane], row_l[L + 1 + lane]));
          thr = (dl >= 0.f) ? 1.f : ex2(dl);
        }
        acc = (u < thr);
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !acc);
    const int32_t js = rej ? (__ffs(rej) - 1) : L;
    if (lane == 0) {
      if (bad) {
        reject();
        s_js = -1;
      } else {
        a.accept_len[i] = js;
        if (GREEDY) a.next_token[i] = row_idx[js];
        s_js = js;
      }
    }
  }
  if (GREEDY) return;
  __syncthreads();
  const int32_t js = s_js;
  if (js < 0) return;
  // ---- the next token: inverse CDF over [p - q]_+ at row js, or p at the bonus row ----
  RowConst rc;
  rc.k = a.k;
  rc.resid = js < L;
  rc.nT = -__fmaf_rn(row_m[js], a.k, row_l[js]);
  rc.nD = rc.resid ? -__fmaf_rn(row_m[L + 1 + js], a.k, row_l[L + 1 + js]) : 0.f;
  const char *trow = static_cast<const char *>(a.target) + (t0 + js) * a.V * E::kSize;
  const char *drow = rc.resid ? static_cast<const char *>(a.draft) + (d0 + js) * a.V * E::kSize : nullptr;
  const float w = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(js), 1u);
  const int32_t tok = cta_sample<DT, VEC, kFinThreads>(trow, drow, a.V, rc, w, ssm);
  if (tid == 0) a.next_token[i] = tok;
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

// launch as a programmatic dependent of the previous kernel in the stream
template <typename Kern>
cudaError_t launch_dependent(const char *name, Kern kern, unsigned grid, unsigned block, const VerifyArgs &a,
                             cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *tm = timer_before(name, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  timer_after(tm, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DT, bool VEC, bool GREEDY>
cudaError_t launch_all_t(const VerifyArgs &args, cudaStream_t st) {
  using E = Elem<DT>;
  const int stage_bytes = VEC ? (args.chunk_len * E::kSize + 127) / 128 * 128 : 0;
  const int smem = VEC ? kStages * stage_bytes : 0;
  auto fn = verify_stats<DT, VEC, GREEDY>;
  cudaError_t e = cudaSuccess;
  if (VEC) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  constexpr int kStatsThreads = StatsShape<GREEDY>::kThreads;
  int grid = cached_grid(reinterpret_cast<const void *>(fn), kStatsThreads, smem, e);
  if (e != cudaSuccess) return e;
  if (grid > args.total_items) grid = static_cast<int>(args.total_items);
  if (grid > kMaxStatsGrid) grid = kMaxStatsGrid;
  if (grid < 1) grid = 1;
  VerifyArgs a = args;
  a.stats_grid = grid;
  // the first kernel is an ordinary launch: it waits for all earlier work in
  // the stream (a previous call's sampler may still read this workspace)
  void *tm = timer_before("verify_stats", st);
  fn<<<grid, kStatsThreads, smem, st>>>(a, stage_bytes);
  timer_after(tm, st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_dependent("verify_finalize", verify_finalize<DT, GREEDY, VEC>, static_cast<unsigned>(a.N), kFinThreads,
                          a, st);
}

template <int DT, bool VEC>
cudaError_t launch_all(const VerifyArgs &a, bool greedy, cudaStream_t st) {
  return greedy ? launch_all_t<DT, VEC, true>(a, st) : launch_all_t<DT, VEC, false>(a, st);
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
  size_t off = 0;
  l.part_off = off;
  off += align256(rows * static_cast<size_t>(p.C) * kCWMax * sizeof(Partial));
  l.csr_bad_off = off;
  off += align256(kMaxStatsGrid * sizeof(int32_t));
  l.total = off;
  return l;
}

FusedLayout fused_layout(int32_t N, int64_t total_rows, int64_t V) {
  (void)V;
  const size_t R = static_cast<size_t>(total_rows);
  FusedLayout l;
  size_t off = 0;
  l.flags_off = off;
  off += align256(R * 4);
  l.rowc_off = off;
  off += align256(R * 16);
  l.bpart_off = off;
  off += align256(static_cast<size_t>(N) * 8 * 16);
  l.csr_bad_off = off;
  off += align256(kMaxStatsGrid * sizeof(int32_t));
  l.total = off;
  return l;
}

cudaError_t launch_verify(const VerifyArgs &a, int dtype, bool vec, bool greedy, cudaStream_t st) {
  if (dtype == SVW_BF16) return vec ? launch_all<1, true>(a, greedy, st) : launch_all<1, false>(a, greedy, st);
  return vec ? launch_all<0, true>(a, greedy, st) : launch_all<0, false>(a, greedy, st);
}

}  // namespace svw
