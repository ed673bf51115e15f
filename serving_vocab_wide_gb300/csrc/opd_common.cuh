// opd_common.cuh -- pieces shared by the OPD loss kernels: row geometry,
// the target row of a draft row, 16-byte vector helpers, and the partial row
// statistics (with their lane merge) that the one-pass kernels exchange
// across a thread-block cluster.
#pragma once
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace svw {
namespace {


// per-launch geometry: slice length and bytes per CTA, entries of the fast
// kernel's target-row table (verify layout)
struct OpdGeo {
  int32_t SL;
  int32_t slice_bytes;
  int32_t ntab;
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

// target row of fast-kernel row r: draft row r < R pairs with its target row;
// r = R + i is request i's bonus row cu[i+1] + i (-1 if the offset is out of range)
__device__ __forceinline__ int64_t fast_target_row(const OpdArgs &a, int64_t r) {
  if (r < a.R) return target_row_of(a, r);
  const int64_t i = r - a.R;
  const int64_t c1 = __ldg(a.cu + i + 1);
  return (c1 >= 0 && c1 <= a.R) ? c1 + i : -1;
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


// Partial row statistics of the fast kernel over some vocabulary entries,
// relative to offsets m_y, m_z (their maxima):
//   s_y = sum 2^((y - m_y)k),  s_z = sum 2^((z - m_z)k),
//   u   = sum 2^((z - m_z)k) ((z - m_z)k - (y - m_y)k),
// and the first index holding the target maximum with the draft logit there.
struct __align__(16) FastPart {
  float my, sy, mz, sz, u;
  int32_t idx;
  float zx;
  int32_t abort;
};

__device__ __forceinline__ FastPart empty_part() {
  FastPart p;
  p.my = -INFINITY;
  p.mz = -INFINITY;
  p.sy = 0.f;
  p.sz = 0.f;
  p.u = 0.f;
  p.idx = INT32_MAX;
  p.zx = 0.f;
  p.abort = 0;
  return p;
}

// Merge the partials held by lanes [0, SPAN) of a warp (SPAN a power of two;
// lanes beyond the data hold empty partials).  Each lane rescales its own
// partial to the merged offsets (one exp2 per sum, all lanes at once), then
// the sums are added by a fixed butterfly, so every warp that merges the same
// partials gets bit-identical results.  A NaN sum (a NaN or +Inf logit)
// stays NaN; a non-finite u only makes the KL non-finite.
template <int SPAN>
__device__ __forceinline__ FastPart merge_lanes(const FastPart &p, float k) {
  float My = p.my, Mz = p.mz;
#pragma unroll
  for (int o = SPAN / 2; o > 0; o >>= 1) {
    My = fmaxf(My, __shfl_xor_sync(0xffffffffu, My, o));
    Mz = fmaxf(Mz, __shfl_xor_sync(0xffffffffu, Mz, o));
  }
  const bool hy = p.my != -INFINITY, hz = p.mz != -INFINITY;
  const float dy = hy ? (p.my - My) * k : 0.f;
  const float dz = hz ? (p.mz - Mz) * k : 0.f;
  float sy = p.sy * (hy ? ex2(dy) : 0.f);
  const float fz = hz ? ex2(dz) : 0.f;
  float sz = p.sz * fz;
  float u = hz ? fz * (p.u + p.sz * (dz - dy)) : (p.u != p.u ? p.u : 0.f);
#pragma unroll
  for (int o = SPAN / 2; o > 0; o >>= 1) {
    sy += __shfl_xor_sync(0xffffffffu, sy, o);
    sz += __shfl_xor_sync(0xffffffffu, sz, o);
    u += __shfl_xor_sync(0xffffffffu, u, o);
  }
  const int32_t cand = (p.my == My) ? p.idx : INT32_MAX;
  const int32_t best = static_cast<int32_t>(__reduce_min_sync(0xffffffffu, static_cast<uint32_t>(cand)));
  const uint32_t holders = __ballot_sync(0xffffffffu, cand == best);
  const float zx = __shfl_sync(0xffffffffu, p.zx, holders ? __ffs(holders) - 1 : 0);
  FastPart r;
  r.my = My;
  r.mz = Mz;
  r.sy = sy;
  r.sz = sz;
  r.u = u;
  r.idx = best;
  r.zx = zx;
  r.abort = __any_sync(0xffffffffu, p.abort != 0) ? 1 : 0;
  return r;
}

// Called by every thread after its reads of the slice buffer for the it-th
// row.  True in exactly one thread (lane 0 of the last warp to finish): that
// thread may overwrite the buffer.  The acq_rel counter orders every warp's
// reads before the overwrite; the async proxy is fenced by the copy issue.
template <int kWarps>
__device__ __forceinline__ bool last_warp_done(uint32_t *cnt, int64_t it) {
  __syncwarp();
  bool last = false;
  if ((threadIdx.x & 31) == 0) {
    uint32_t prev;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(prev) : "r"(smem_u32(cnt)) : "memory");
    last = (prev == static_cast<uint32_t>(kWarps * it + kWarps - 1));
  }
  return last;
}

// Warp-uniform variant: true in every lane of the last warp to get here for
// the it-th time; that warp then sees every other warp's earlier writes.
template <int kWarps>
__device__ __forceinline__ bool last_warp_all(uint32_t *cnt, int64_t it) {
  __syncwarp();
  uint32_t prev = 0;
  if ((threadIdx.x & 31) == 0)
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(prev) : "r"(smem_u32(cnt)) : "memory");
  prev = __shfl_sync(0xffffffffu, prev, 0);
  const bool last = (prev == static_cast<uint32_t>(kWarps * it + kWarps - 1));
  if (last) __threadfence_block();
  return last;
}


}  // namespace
}  // namespace svw
