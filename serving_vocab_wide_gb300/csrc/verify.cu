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
//  2. verify_finalize   one CTA per request (at T > 0 a cluster of CTAs per
//                       request, as many as fill the GPU once): CTA 0
//                       validates the request, merges the partials into row
//                       log-sum-exps (or argmaxes), runs every accept test in
//                       one warp (ballot + ffs = leftmost rejection), writes
//                       accept_len, then (T > 0) the cluster draws the next
//                       token by inverse CDF over the residual row pair or the
//                       bonus row (svw_sample.cuh), one slice of the row
//                       per CTA.
// The finalize kernel is launched as a programmatic dependent of the stats
// kernel: it is scheduled while the stream drains and reads the draft tokens
// and their logits before waiting (griddepcontrol.wait) for the partials.
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>
#include <mutex>

#include "svw_device.cuh"
#include "svw_internal.h"
#include "svw_sample.cuh"

namespace svw {

namespace {

// consumer warps of the stats kernel.  Each warp ends a ring stage with a
// reduction and a partial, so fewer warps with more vectors each waste less;
// the argmax needs no exponentials, so greedy mode keeps up with half the
// warps (4 and 8 measured best at V = 151936 bf16)
constexpr int kCWMax = 16;
template <bool GREEDY, bool EARLY = false>
struct StatsShape {
  static constexpr int kCW = GREEDY ? 4 : 8;
  // + one producer warp (+ one accounting warp with early exit)
  static constexpr int kThreads = (kCW + (EARLY ? 2 : 1)) * 32;
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
  int32_t test;  // early exit: the accept test (kq * max_len + j) this item feeds, -1 if none
  int64_t c_i;   // early exit: the request's first draft row
  int32_t req;   // early exit: the request
  int32_t pos;   // early exit: the position j
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
  m.test = -1;
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

// Early exit: items are numbered position-major.  Wave j holds position j of
// every request that has it, requests in the order of the plan's permutation
// (longest first): the first A_j requests (L_i > j) contribute target row j
// and draft row j (greedy: target row j only), C chunks each; the next B_j
// (L_i = j) contribute their bonus row.  W[j] is the first item of wave j.
// An item whose request already stopped (a rejection or a bad row at a
// position before j) is skipped: no copy, no partial.
//
// The producer locates an item (shared-memory arithmetic only) and starts the
// two loads it depends on -- the request record and the stop word, both kept
// in permutation order -- before it waits for a free stage, and finishes the
// decode after the wait.
struct EarlyPre {
  int64_t item;
  int32_t j, kq, kind, chunk;
  int4 info;     // {request, first draft row, L, 0}
  int32_t stop;  // first position known to stop the request
};

template <bool GREEDY>
__device__ __forceinline__ EarlyPre early_locate(const VerifyArgs &a, int64_t item, int64_t total, const int64_t *W,
                                                 const int32_t *A) {
  EarlyPre e;
  e.item = item;
  e.j = 0;
  e.kq = 0;
  e.kind = 0;
  e.chunk = 0;
  e.info = make_int4(0, 0, 0, 0);
  e.stop = -1;
  if (item >= total) return e;
  int32_t j = 0;
  while (j < a.max_len && W[j + 1] <= item) ++j;
  const int64_t local = item - W[j];
  const int64_t C = a.C;
  int64_t kq;
  if (!GREEDY && local < 2 * C * A[j]) {
    kq = local / (2 * C);
    const int64_t rem = local - kq * 2 * C;
    e.kind = rem >= C ? 1 : 0;
    e.chunk = static_cast<int32_t>(rem - e.kind * C);
  } else {
    const int64_t l2 = GREEDY ? local : local - 2 * C * A[j];
    const int64_t q = l2 / C;
    kq = (GREEDY ? 0 : A[j]) + q;
    e.chunk = static_cast<int32_t>(l2 - q * C);
  }
  e.j = j;
  e.kq = static_cast<int32_t>(kq);
  e.info = __ldcg(a.pinfo + kq);
  e.stop = __ldcg(a.stop + kq);
  return e;
}

template <int DT>
__device__ __forceinline__ ItemMeta early_finish(const VerifyArgs &a, const EarlyPre &e) {
  using E = Elem<DT>;
  ItemMeta m;
  m.item = e.item;
  m.valid = 0;
  m.test = -1;
  m.prow = 0;
  m.src = nullptr;
  m.chunk = e.chunk;
  m.n = 0;
  const int32_t i = e.info.x, L = e.info.z, j = e.j;
  const int64_t c_i = e.info.y;
  m.c_i = c_i;
  m.req = i;
  m.pos = j;
  if (e.stop < j) return m;  // the request stopped before j
  const int64_t c0 = static_cast<int64_t>(m.chunk) * a.chunk_len;
  m.n = static_cast<int32_t>(min(static_cast<int64_t>(a.chunk_len), a.V - c0));
  const char *row;
  if (e.kind == 0) {
    m.prow = c_i + i + j;
    row = static_cast<const char *>(a.target) + m.prow * a.V * E::kSize;
  } else {
    m.prow = a.rows_t + c_i + j;
    row = static_cast<const char *>(a.draft) + (c_i + j) * a.V * E::kSize;
  }
  m.src = row + c0 * E::kSize;
  m.test = (j < L) ? e.kq * a.max_len + j : -1;
  m.valid = 1;
  return m;
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
// one row's statistics merged from its np partials by one warp, in a fixed
// order (lane-strided, then a butterfly), so that every caller -- the
// finalize kernels and the early-exit tests -- gets the same bits
// ---------------------------------------------------------------------------
__device__ __forceinline__ void merge_row_lse(const Partial *pp, int np, float k, int lane, float &m, float &l,
                                              int32_t &bad) {
  float mm = -INFINITY, s = 0.f;
  for (int p = lane; p < np; p += 32) {
    const Partial q = ldcg_partial(pp + p);
    lse_combine(mm, s, q.m, q.s, k);
  }
  warp_lse(mm, s, k);
  m = mm;
  l = lg2(s);
  bad = (s > 0.f && s <= FLT_MAX) ? 0 : 1;
}

__device__ __forceinline__ void merge_row_amax(const Partial *pp, int np, int lane, int32_t &idx, int32_t &bad) {
  float v = -INFINITY;
  int32_t id = INT32_MAX, nan = 0;
  for (int p = lane; p < np; p += 32) {
    const Partial q = ldcg_partial(pp + p);
    amax_combine(v, id, q.m, q.idx);
    nan |= q.nan;
  }
  warp_amax(v, id);
  idx = id;
  bad = __any_sync(0xffffffffu, nan != 0) ? 1 : 0;
}

// Two rows merged as merge_row_lse merges each (same order per row, same
// bits), with both rows' loads in flight together.
__device__ __forceinline__ void merge_two_rows_lse(const Partial *pa, const Partial *pb, int np, float k, int lane,
                                                   float &ma, float &la, int32_t &bada, float &mb, float &lb,
                                                   int32_t &badb) {
  float m0 = -INFINITY, s0 = 0.f, m1 = -INFINITY, s1 = 0.f;
#pragma unroll 4
  for (int p = lane; p < np; p += 32) {
    const Partial qa = ldcg_partial(pa + p);
    const Partial qb = ldcg_partial(pb + p);
    lse_combine(m0, s0, qa.m, qa.s, k);
    lse_combine(m1, s1, qb.m, qb.s, k);
  }
  warp_lse(m0, s0, k);
  warp_lse(m1, s1, k);
  ma = m0;
  la = lg2(s0);
  bada = (s0 > 0.f && s0 <= FLT_MAX) ? 0 : 1;
  mb = m1;
  lb = lg2(s1);
  badb = (s1 > 0.f && s1 <= FLT_MAX) ? 0 : 1;
}

// Early exit: the accept test of position j of request i, run by the warp
// that delivered the last partial of its rows.  A rejection or a bad row
// (non-finite statistics, token out of range) lowers the request's stop word
// (so later positions are no longer read) and its first rejected / bad
// position (for the finalize kernel).
template <int DT, bool GREEDY, int CW>
__device__ __noinline__ void early_test(const VerifyArgs &a, int32_t kq, int32_t i, int64_t c_i, int32_t j,
                                        int lane) {
  using E = Elem<DT>;
  const int64_t trow = c_i + i + j, drow = c_i + j;
  const int np = a.C * CW;
  const int32_t x = __ldg(a.tokens + drow);
  int32_t bad = (x < 0 || static_cast<int64_t>(x) >= a.V) ? 1 : 0;
  bool acc = false;
  if (GREEDY) {
    int32_t idx = INT32_MAX, nan = 0;
    merge_row_amax(a.part + trow * np, np, lane, idx, nan);
    bad |= nan;
    acc = (x == idx);
  } else {
    // the logits at x and the uniform do not depend on the partials
    const float yx = bad ? 0.f : E::load(a.target, trow * a.V + x);
    const float zx = bad ? 0.f : E::load(a.draft, drow * a.V + x);
    const float u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(j), 0u);
    float mT, lT, mD, lD;
    int32_t bT, bD;
    merge_two_rows_lse(a.part + trow * np, a.part + (a.rows_t + drow) * np, np, a.k, lane, mT, lT, bT, mD, lD,
                       bD);
    bad |= bT | bD;
    acc = !bad && accept_token(u, yx, zx, mT, lT, mD, lD, a.k);
  }
  if (lane == 0) {
    if (bad) {
      atomicMin(a.stop + kq, j);
      atomicMin(a.badpos + i, j);
    } else if (!acc) {
      atomicMin(a.stop + kq, j);
      atomicMin(a.rej + i, j);
    }
  }
}

// Early exit: count inc consumer-warp partials towards their accept test; the
// warp that completes the count (2 rows x C chunks x CW warps; greedy: the
// target row only) runs the test.  Store -> (CTA sync) -> release on every
// side, acquire -> loads on the last.
template <int DT, bool GREEDY, int CW>
__device__ __forceinline__ void early_arrive(const VerifyArgs &a, const ItemMeta &m, int lane, int inc) {
  int last = 0;
  if (lane == 0) {
    const int need = (GREEDY ? 1 : 2) * a.C * CW;
    int old;
    // release: the partials written before it (by this thread, or by the
    // consumer warps whose mbarrier arrivals this thread observed) are
    // visible before the count; acquire: the last counter sees all of them
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(a.cnt + m.test), "r"(inc)
                 : "memory");
    last = (old == need - inc) ? 1 : 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();  // lane 0's acquire orders the whole warp's loads below
  if (last) early_test<DT, GREEDY, CW>(a, m.test / a.max_len, m.req, m.c_i, m.pos, lane);
}

// Early exit, ahead of the stats stream (one CTA): per-request checks, the
// position-major wave layout (W[j], A_j = requests longer than j), the valid
// requests' records {request, first draft row, L} in permutation order by
// length (longest first; the order within a length is arbitrary and does not
// affect any result), the CSR flag, and this call's state reset: test
// counters, stop words, first rejected / bad positions, byte counter.
template <bool GREEDY>
__global__ void __launch_bounds__(1024) early_plan(VerifyArgs a) {
  __shared__ int32_t hist[SVW_MAX_LEN + 1];
  __shared__ int32_t cur[SVW_MAX_LEN + 1];
  pdl_launch_dependents();  // the stats grid may be scheduled now
  const int tid = threadIdx.x;
  if (tid <= SVW_MAX_LEN) hist[tid] = 0;
  __syncthreads();
  auto length_of = [&](int32_t i, int64_t &c_i) -> int32_t {
    c_i = __ldg(a.cu + i);
    const int64_t c_e = __ldg(a.cu + i + 1);
    const int64_t L = c_e - c_i;
    return (L >= 1 && L <= a.max_len && c_i >= 0 && c_e <= a.total_rows) ? static_cast<int32_t>(L) : 0;
  };
  int bad = 0;
  for (int32_t i = tid; i < a.N; i += 1024) {
    int64_t c_i;
    const int32_t L = length_of(i, c_i);
    bad |= (c_i > static_cast<int64_t>(__ldg(a.cu + i + 1))) ? 1 : 0;
    if (L > 0) atomicAdd(&hist[L], 1);
    a.rej[i] = INT32_MAX;
    a.badpos[i] = INT32_MAX;
    a.stop[i] = INT32_MAX;  // indexed by permutation slot; N slots at most
    if (a.eres) a.eres[i] = make_int4(-1, 1, 0, 0);  // a request no cluster finished is bad
  }
  if (tid == 0) bad |= (__ldg(a.cu) != 0 || static_cast<int64_t>(__ldg(a.cu + a.N)) != a.total_rows) ? 1 : 0;
  const int64_t ncnt = static_cast<int64_t>(a.N) * a.max_len;
  for (int64_t q = tid; q < ncnt; q += 1024) a.cnt[q] = 0;
  bad = __syncthreads_or(bad);
  if (tid == 0) {
    a.csr_bad[0] = bad;
    if (a.bytes_read) *a.bytes_read = 0ull;
    int32_t above = 0;  // valid requests longer than Lq
    for (int32_t Lq = a.max_len; Lq >= 1; --Lq) {
      cur[Lq] = above;
      above += hist[Lq];
    }
    int32_t Aj = above;  // every valid request has position 0
    int64_t w = 0;
    for (int32_t j = 0; j <= a.max_len; ++j) {
      const int32_t Bj = (j >= 1) ? hist[j] : 0;  // bonus rows at position j
      if (j >= 1) Aj -= hist[j];
      a.waveA[j] = Aj;
      a.W[j] = w;
      w += static_cast<int64_t>(a.C) * (GREEDY ? (Aj + Bj) : (2 * static_cast<int64_t>(Aj) + Bj));
    }
    a.W[a.max_len + 1] = w;
    *a.nvalid = above;
    *a.qnext = 0;
  }
  __syncthreads();
  for (int32_t i = tid; i < a.N; i += 1024) {
    int64_t c_i;
    const int32_t L = length_of(i, c_i);
    if (L > 0) a.pinfo[atomicAdd(&cur[L], 1)] = make_int4(i, static_cast<int32_t>(c_i), L, 0);
  }
}

// ---------------------------------------------------------------------------
// kernel 2: stats stream
// ---------------------------------------------------------------------------
template <int DT, bool BULK, bool GREEDY, bool EARLY>
__global__ void __launch_bounds__(StatsShape<GREEDY, EARLY>::kThreads, 2)
    verify_stats(VerifyArgs a, int stage_bytes) {
  constexpr int kCW = StatsShape<GREEDY>::kCW;
  constexpr int kStatsThreads = StatsShape<GREEDY, EARLY>::kThreads;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ unsigned long long full[kStages], empty[kStages];
  __shared__ unsigned long long done[kStages];  // early exit: the consumers' partials of a stage are written
  __shared__ ItemMeta meta[kStages];
  __shared__ int64_t waveW[SVW_MAX_LEN + 2];  // early exit: first item of each wave
  __shared__ int32_t waveA[SVW_MAX_LEN + 1];  // early exit: requests longer than j
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  pdl_launch_dependents();  // the finalize grid may be scheduled now
  int64_t total_items = a.total_items;
  if (EARLY) {
    // the plan kernel's layout and reset state (the CSR check is its job too)
    pdl_wait();
    for (int q = threadIdx.x; q <= a.max_len + 1; q += kStatsThreads) {
      waveW[q] = __ldcg(a.W + q);
      if (q <= a.max_len) waveA[q] = __ldcg(a.waveA + q);
    }
    __syncthreads();
    total_items = waveW[a.max_len + 1];
  } else {
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
  auto decode = [&](int64_t item) {
    return EARLY ? early_finish<DT>(a, early_locate<GREEDY>(a, item, total_items, waveW, waveA))
                 : decode_item<DT, GREEDY>(a, item);
  };

  if (!BULK) {
    // plain loads: every warp walks the CTA's items itself (no producer)
    if (wid >= kCW) return;
    unsigned long long nbytes = 0;
    for (int64_t item = blockIdx.x; item < total_items; item += G) {
      const ItemMeta m = decode(item);
      if (!m.valid) continue;
      nbytes += static_cast<unsigned long long>(m.n) * Elem<DT>::kSize;
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
      if (EARLY && m.test >= 0) early_arrive<DT, GREEDY, kCW>(a, m, lane, 1);
    }
    if (EARLY && a.bytes_read && wid == 0 && lane == 0) atomicAdd(a.bytes_read, nbytes);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], EARLY ? 1 : kCW);  // early exit: released by the accounting warp
      mbar_init(&done[s], kCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (wid == kCW) {
    // ---------------- producer warp (one lane) ----------------
    if (lane != 0) return;
    unsigned long long nbytes = 0;
    auto add_bytes = [&]() {
      if (EARLY && a.bytes_read) atomicAdd(a.bytes_read, nbytes);
    };
    int k = 0;
    // test-only fault (svw_set_fault): CTA 0 issues nothing, so its consumers'
    // first wait runs out with no copy in flight
    if (a.fault == 1 && blockIdx.x == 0) return;
    // early exit: the next item's two loads are in flight while this lane
    // waits for its stage
    EarlyPre pre;
    if (EARLY) pre = early_locate<GREEDY>(a, blockIdx.x, total_items, waveW, waveA);
    for (int64_t item = blockIdx.x;; item += G, ++k) {
      const int s = k % kStages;
      if (k >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((k / kStages) - 1) & 1))) {
        // consumers stopped releasing stages: report, hand them an end marker
        if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        add_bytes();
        return;
      }
      if (item >= total_items) {
        meta[s].item = -1;
        mbar_arrive(&full[s]);
        add_bytes();
        return;
      }
      const ItemMeta m = EARLY ? early_finish<DT>(a, pre) : decode_item<DT, GREEDY>(a, item);
      meta[s] = m;
      if (m.valid) {
        const uint32_t bytes = static_cast<uint32_t>(m.n) * Elem<DT>::kSize;
        nbytes += bytes;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(ring + static_cast<size_t>(s) * stage_bytes, m.src, bytes, &full[s]);
      } else {
        mbar_arrive(&full[s]);
      }
      if (EARLY) pre = early_locate<GREEDY>(a, item + G, total_items, waveW, waveA);
    }
  }

  if (EARLY && wid == kCW + 1) {
    // ---------------- accounting warp (early exit) ----------------
    // Follows the ring one stage behind the consumers: once a stage's
    // partials are written it frees the stage, then counts them towards their
    // accept test with one fenced atomic, and runs the test if they complete
    // it -- all off the consumers' path.
    for (int k = 0;; ++k) {
      const int s = k % kStages;
      const uint32_t par = static_cast<uint32_t>((k / kStages) & 1);
      if (!mbar_wait_bounded(&full[s], par)) {
        if (lane == 0 && a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        return;
      }
      const ItemMeta m = meta[s];
      if (m.item < 0) return;
      if (!mbar_wait_bounded(&done[s], par)) {
        if (lane == 0 && a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        return;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (m.valid && m.test >= 0) early_arrive<DT, GREEDY, kCW>(a, m, lane, kCW);
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
    if (lane == 0) mbar_arrive(EARLY ? &done[s] : &empty[s]);
  }
}

// ---------------------------------------------------------------------------
// kernel 2: per-request validation, merge, accept tests
// ---------------------------------------------------------------------------
// MODE 0: spec_verify (merge every row's partials, run every test);
// MODE 1: early exit by the chunk stream (the tests ran in the stats kernel);
// MODE 2: early exit by clusters (stop position and statistics recorded).
template <int DT, bool GREEDY, bool VEC, int MODE>
__global__ void __launch_bounds__(kFinThreads) verify_finalize(VerifyArgs a) {
  using E = Elem<DT>;
  __shared__ float row_m[kMaxRows];
  __shared__ float row_l[kMaxRows];
  __shared__ int32_t row_idx[kMaxRows];
  __shared__ int32_t row_bad[kMaxRows];
  __shared__ int32_t s_ok, s_js;
  __shared__ uint32_t s_draw[4];  // the draw's inputs from CTA 0 of the cluster: js, nT, nD, resid
  __shared__ SampleSmem<kFinThreads> ssm;
  extern __shared__ float sample_w[];  // T > 0: the draw's warp totals
  // at T > 0 a cluster of CL CTAs serves request i: CTA 0 merges and tests,
  // then all of them draw the next token (one slice of the row each)
  const int CL = GREEDY ? 1 : static_cast<int>(cluster_size());
  const int rank = GREEDY ? 0 : static_cast<int>(cluster_rank());
  const int32_t i = blockIdx.x / CL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  if (rank == 0) {
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
        if (tok_ok && !GREEDY && MODE == 0) {
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
    const int np = a.C * StatsShape<GREEDY>::kCW;  // partials per row
    if (!s_ok || csr_bad) {
      if (tid == 0) {
        reject();
        s_js = -1;
      }
    } else if (MODE == 2) {
      if (warp == 0) {
        const int4 r = __ldcg(a.eres + i);
        const float4 f = __ldcg(a.erow + i);
        const int32_t js = r.x;
        if (lane == 0) {
          if (r.y != 0 || js < 0 || js > L) {
            reject();
            s_js = -1;
          } else {
            a.accept_len[i] = js;
            if (GREEDY) a.next_token[i] = r.z;
            row_m[js] = f.x;
            row_l[js] = f.y;
            if (js < L) {
              row_m[L + 1 + js] = f.z;
              row_l[L + 1 + js] = f.w;
            }
            s_js = js;
          }
        }
      }
    } else if (MODE == 1) {
      // the stats stream ran the accept tests in position order and stopped
      // reading a request at its first rejection (or bad row): only the rows
      // at that position are merged here
      if (warp == 0) {
        const int32_t r = min(__ldcg(a.rej + i), L);
        int32_t bad = (__ldcg(a.badpos + i) <= r) ? 1 : 0;
        int32_t idx = INT32_MAX, b = 0;
        if (GREEDY) {
          merge_row_amax(a.part + (t0 + r) * np, np, lane, idx, b);
          bad |= b;
        } else {
          float m, l;
          merge_row_lse(a.part + (t0 + r) * np, np, a.k, lane, m, l, b);
          bad |= b;
          if (lane == 0) {
            row_m[r] = m;
            row_l[r] = l;
          }
          if (r < L) {
            merge_row_lse(a.part + (a.rows_t + d0 + r) * np, np, a.k, lane, m, l, b);
            bad |= b;
            if (lane == 0) {
              row_m[L + 1 + r] = m;
              row_l[L + 1 + r] = l;
            }
          }
        }
        if (lane == 0) {
          if (bad) {
            reject();
            s_js = -1;
          } else {
            a.accept_len[i] = r;
            if (GREEDY) a.next_token[i] = idx;
            s_js = r;
          }
        }
      }
    } else {
      const int32_t nrows = GREEDY ? L + 1 : 2 * L + 1;
      for (int r = warp; r < nrows; r += kFinWarps) {
        const int64_t prow = (r <= L) ? (t0 + r) : (a.rows_t + d0 + (r - L - 1));
        const Partial *pp = a.part + prow * np;
        int32_t b;
        if (GREEDY) {
          int32_t idx;
          merge_row_amax(pp, np, lane, idx, b);
          if (lane == 0) row_idx[r] = idx;
        } else {
          float m, l;
          merge_row_lse(pp, np, a.k, lane, m, l, b);
          if (lane == 0) {
            row_m[r] = m;
            row_l[r] = l;
          }
        }
        if (lane == 0) row_bad[r] = b;
      }
      __syncthreads();
      if (warp == 0) {
        int bad = 0;
        for (int r = lane; r < nrows; r += 32) bad |= row_bad[r];
        bad = __any_sync(0xffffffffu, bad);
        bool acc = true;
        if (lane < L)
          acc = GREEDY ? (x == row_idx[lane])
                       : accept_token(u, yx, zx, row_m[lane], row_l[lane], row_m[L + 1 + lane],
                                      row_l[L + 1 + lane], a.k);
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
    }
    if (GREEDY) return;
    __syncthreads();
    // the draw's inputs to every CTA of the cluster
    if (tid < CL) {
      const int32_t js = s_js;
      const bool resid = js >= 0 && js < L;
      const float nT = (js >= 0) ? -__fmaf_rn(row_m[js], a.k, row_l[js]) : 0.f;
      const float nD = resid ? -__fmaf_rn(row_m[L + 1 + js], a.k, row_l[L + 1 + js]) : 0.f;
      const uint32_t v[4] = {static_cast<uint32_t>(js), __float_as_uint(nT), __float_as_uint(nD), resid ? 1u : 0u};
#pragma unroll
      for (int q = 0; q < 4; ++q) st_cluster_b32(mapa_shared(smem_u32(&s_draw[q]), tid), v[q]);
    }
  }  // CTA 0
  if (GREEDY) return;
  cluster_barrier();
  const int32_t js = static_cast<int32_t>(s_draw[0]);
  if (js < 0) return;  // the same in every CTA of the cluster
  // ---- the next token: inverse CDF over [p - q]_+ at row js, or p at the bonus row ----
  const int64_t c_i = __ldg(a.cu + i);
  RowConst rc;
  rc.k = a.k;
  rc.resid = s_draw[3] != 0;
  rc.nT = __uint_as_float(s_draw[1]);
  rc.nD = __uint_as_float(s_draw[2]);
  const char *trow = static_cast<const char *>(a.target) + (c_i + i + js) * a.V * E::kSize;
  const char *drow = rc.resid ? static_cast<const char *>(a.draft) + (c_i + js) * a.V * E::kSize : nullptr;
  const float w = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(js), 1u);
  const int32_t tok =
      cluster_sample<DT, VEC, kFinThreads>(trow, drow, a.V, rc, w, ssm, sample_w, CL, rank);
  if (tid == 0 && tok >= 0) a.next_token[i] = tok;
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
  static std::mutex mu;  // calls from several host threads share the cache
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
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
template <typename Kern, typename... Args>
cudaError_t launch_dependent(const char *name, Kern kern, unsigned grid, unsigned block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *tm = timer_before(name, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  timer_after(tm, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The finalize grid: one CTA per request, or at T > 0 a cluster of CL CTAs
// per request that draws the next token together.
template <bool GREEDY, bool VEC, typename Kern>
cudaError_t launch_finalize(const char *name, Kern kern, int N, int threads, cudaStream_t st, const VerifyArgs &a) {
  int cl = 1;
  size_t smem = 0;  // the draw's warp totals
  if (!GREEDY) {
    cl = draw_cluster(N);
    smem = sample_dyn_bytes(a.V, cl, threads);
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
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
  cfg.gridDim = dim3(static_cast<unsigned>(N) * static_cast<unsigned>(cl), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = GREEDY ? 1 : 2;
  void *tm = timer_before(name, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  timer_after(tm, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DT, bool VEC, bool GREEDY, bool EARLY>
cudaError_t launch_all_t(const VerifyArgs &args, cudaStream_t st) {
  using E = Elem<DT>;
  if (EARLY && VEC) {
    // the cluster path when the rows fit it: plan, clusters, finalize
    const EarlyClusterPlan cp = early_cluster_plan(args.V, E::kSize, GREEDY);
    if (cp.CL > 0) {
      VerifyArgs a = args;
      a.stats_grid = 1;  // the plan kernel writes the one CSR flag
      void *tm = timer_before("early_plan", st);
      early_plan<GREEDY><<<1, 1024, 0, st>>>(a);
      timer_after(tm, st);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      e = launch_early_cluster(a, DT == 1 ? SVW_BF16 : SVW_F32, GREEDY, cp, st);
      if (e != cudaSuccess) return e;
      return launch_finalize<GREEDY, VEC>("verify_finalize", verify_finalize<DT, GREEDY, VEC, 2>, a.N, kFinThreads, st,
                                     a);
    }
  }
  const int stage_bytes = VEC ? (args.chunk_len * E::kSize + 127) / 128 * 128 : 0;
  const int smem = VEC ? kStages * stage_bytes : 0;
  auto fn = verify_stats<DT, VEC, GREEDY, EARLY>;
  cudaError_t e = cudaSuccess;
  if (VEC) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  constexpr int kStatsThreads = StatsShape<GREEDY, EARLY>::kThreads;
  int grid = cached_grid(reinterpret_cast<const void *>(fn), kStatsThreads, smem, e);
  if (e != cudaSuccess) return e;
  if (grid > args.total_items) grid = static_cast<int>(args.total_items);
  if (grid > kMaxStatsGrid) grid = kMaxStatsGrid;
  if (grid < 1) grid = 1;
  VerifyArgs a = args;
  a.stats_grid = EARLY ? 1 : grid;  // early exit: the plan kernel writes the one CSR flag
  if (EARLY) {
    // the plan is an ordinary launch: it waits for all earlier work in the
    // stream (a previous call's kernels may still read this workspace); the
    // stats stream and the finalize kernel follow as programmatic dependents
    void *tm = timer_before("early_plan", st);
    early_plan<GREEDY><<<1, 1024, 0, st>>>(a);
    timer_after(tm, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_dependent("verify_stats", fn, static_cast<unsigned>(grid), kStatsThreads, smem, st, a, stage_bytes);
  } else {
    // the first kernel is an ordinary launch (see above)
    void *tm = timer_before("verify_stats", st);
    fn<<<grid, kStatsThreads, smem, st>>>(a, stage_bytes);
    timer_after(tm, st);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  return launch_finalize<GREEDY, VEC>("verify_finalize", verify_finalize<DT, GREEDY, VEC, EARLY ? 1 : 0>, a.N,
                                 kFinThreads, st, a);
}

template <int DT, bool VEC, bool EARLY>
cudaError_t launch_all(const VerifyArgs &a, bool greedy, cudaStream_t st) {
  return greedy ? launch_all_t<DT, VEC, true, EARLY>(a, st) : launch_all_t<DT, VEC, false, EARLY>(a, st);
}

}  // namespace

// CTAs per request of a finalize grid that draws at T > 0 (1, 2, 4 or 8): the
// largest cluster with which the whole grid is resident at once, two CTAs
// per SM.  Every CTA waits for its request's accept tests before it draws, so
// a grid in several waves would pay that wait once per wave: a small batch
// gets its rows split over the GPU, a large one keeps one CTA per request.
int draw_cluster(int N) {
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    nsm = 1;
  int cl = 1;
  while (cl < kMaxSampleCluster && static_cast<int64_t>(N) * cl * 2 <= 2 * static_cast<int64_t>(nsm)) cl *= 2;
  return cl;
}


ChunkPlan plan_chunks(int64_t V, int esize) {
  // at most 36 KB per chunk: three ring stages of two CTAs fit an SM
  const int64_t target = (esize == 2) ? 18432 : 9216;
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
  off += align256(static_cast<size_t>(N) * kBonusParts * 16);
  l.fixp_off = off;
  off += align256(R * kOpdFixParts * sizeof(float2));
  l.csr_bad_off = off;
  off += align256(kMaxStatsGrid * sizeof(int32_t));
  l.total = off;
  return l;
}

cudaError_t launch_verify(const VerifyArgs &a, int dtype, bool vec, bool greedy, cudaStream_t st) {
  if (dtype == SVW_BF16)
    return vec ? launch_all<1, true, false>(a, greedy, st) : launch_all<1, false, false>(a, greedy, st);
  return vec ? launch_all<0, true, false>(a, greedy, st) : launch_all<0, false, false>(a, greedy, st);
}

EarlyLayout early_layout(int32_t N, int64_t total_rows, int64_t V, int esize) {
  const VerifyLayout v = verify_layout(N, total_rows, V, esize);
  EarlyLayout l;
  size_t off = v.total;
  l.part_off = v.part_off;
  l.csr_bad_off = v.csr_bad_off;
  l.cnt_off = off;
  off += align256(static_cast<size_t>(N) * SVW_MAX_LEN * sizeof(int32_t));
  l.rej_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(int32_t));
  l.badpos_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(int32_t));
  l.stop_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(int32_t));
  l.pinfo_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(int4));
  l.wave_off = off;
  // W[max_len + 2] (int64), A_j[max_len + 1], valid-request count, queue head
  off += align256((SVW_MAX_LEN + 2) * sizeof(int64_t) + (SVW_MAX_LEN + 3) * sizeof(int32_t));
  l.eres_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(int4));
  l.erow_off = off;
  off += align256(static_cast<size_t>(N) * sizeof(float4));
  l.total = off;
  return l;
}

cudaError_t launch_verify_early(const VerifyArgs &a, int dtype, bool vec, bool greedy, cudaStream_t st) {
  if (dtype == SVW_BF16)
    return vec ? launch_all<1, true, true>(a, greedy, st) : launch_all<1, false, true>(a, greedy, st);
  return vec ? launch_all<0, true, true>(a, greedy, st) : launch_all<0, false, true>(a, greedy, st);
}

}  // namespace svw
