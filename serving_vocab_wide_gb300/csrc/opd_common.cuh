// opd_common.cuh -- pieces shared by the OPD loss kernels: row geometry,
// the target row of a draft row, 16-byte vector helpers, and the partial row
// statistics (with their lane merge) that the one-pass kernels exchange
// across a thread-block cluster.
#pragma once
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>
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

// The first entry of a 16-byte vector of bf16 values equal to the bf16 value
// whose bits are m16 in both halves of m2 (float equality: -0 == +0, NaN
// equals nothing), or -1: four packed compares instead of eight unpacked ones.
__device__ __forceinline__ int bf16_vec_find(const uint4 &w, uint32_t m2) {
  const __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162 *>(&m2);
  const uint32_t e0 = __heq2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w.x), m);
  const uint32_t e1 = __heq2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w.y), m);
  const uint32_t e2 = __heq2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w.z), m);
  const uint32_t e3 = __heq2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w.w), m);
  if (!(e0 | e1 | e2 | e3)) return -1;
  const uint32_t f = e0 ? e0 : (e1 ? e1 : (e2 ? e2 : e3));  // the first word with a match
  const int base = e0 ? 0 : (e1 ? 2 : (e2 ? 4 : 6));
  return base + ((f & 0xffffu) ? 0 : 1);  // low half: the even entry
}

// entry e of a 16-byte vector of bf16 values, as a float
__device__ __forceinline__ float bf16_vec_get(const uint4 &w, int e) {
  const uint32_t v = (e < 4) ? ((e < 2) ? w.x : w.y) : ((e < 6) ? w.z : w.w);
  return __uint_as_float((e & 1) ? (v & 0xffff0000u) : (v << 16));
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
//   s_y = sum 2^((y - m_y)k),
//   w   = sum (2^((z - m_z)k) - 2^((y - m_y)k))   (so s_z = s_y + w),
//   u   = sum 2^((z - m_z)k) ((z - y)k - (m_z - m_y)k),
// and the first index holding the target maximum with the draft logit there.
// w is summed term by term rather than as the difference of two sums: where
// the draft is close to the target, s_z / s_y - 1 = w / s_y is small, and a
// difference of two rounded sums would carry the sums' rounding (~1e-7 of
// s_y) into log(s_z / s_y) and from there into the KL.  Likewise the
// log-ratio reference (z - y)k - (m_z - m_y)k is formed from the exact logit
// difference, not from two row offsets of magnitude ~20.
struct __align__(16) FastPart {
  float my, sy, mz, w, u;
  int32_t idx;
  float zx;
  int32_t abort;
};

__device__ __forceinline__ FastPart empty_part() {
  FastPart p;
  p.my = -INFINITY;
  p.mz = -INFINITY;
  p.sy = 0.f;
  p.w = 0.f;
  p.u = 0.f;
  p.idx = INT32_MAX;
  p.zx = 0.f;
  p.abort = 0;
  return p;
}

// e^x - 1 without cancellation: the series to x^7 for |x| < 1/8 (remainder
// below 2e-10 relative), the library's expm1f beyond.
__device__ __forceinline__ float expm1_nat(float x) {
  if (fabsf(x) < 0.125f) {
    float c = 1.f / 5040.f;
    c = fmaf(c, x, 1.f / 720.f);
    c = fmaf(c, x, 1.f / 120.f);
    c = fmaf(c, x, 1.f / 24.f);
    c = fmaf(c, x, 1.f / 6.f);
    c = fmaf(c, x, 0.5f);
    c = fmaf(c, x, 1.f);
    return x * c;
  }
  return expm1f(x);
}

// Merge the partials held by lanes [0, SPAN) of a warp (SPAN a power of two;
// lanes beyond the data hold empty partials).  Each lane rescales its own
// partial to the merged offsets (one exp2 per sum, all lanes at once), then
// the sums are added by a fixed butterfly, so every warp that merges the same
// partials gets bit-identical results.  A lane's w moves to the merged
// offsets as w fz + s_y fy (2^sh - 1), sh = ((m_z - m_y) - (M_z - M_y)) k the
// change of log-ratio reference, with an accurate expm1 (no cancellation when
// sh is small).  A NaN sum (a NaN or +Inf logit) stays NaN; a non-finite u
// only makes the KL non-finite.
template <int SPAN>
__device__ __forceinline__ FastPart merge_lanes(const FastPart &p, float k) {
  float My = p.my, Mz = p.mz;
#pragma unroll
  for (int o = SPAN / 2; o > 0; o >>= 1) {
    My = fmaxf(My, __shfl_xor_sync(0xffffffffu, My, o));
    Mz = fmaxf(Mz, __shfl_xor_sync(0xffffffffu, Mz, o));
  }
  const bool hy = p.my != -INFINITY, hz = p.mz != -INFINITY;
  const float fy = hy ? ex2((p.my - My) * k) : 0.f;
  const float fz = hz ? ex2((p.mz - Mz) * k) : 0.f;
  float sy = p.sy * fy;
  // change of the log-ratio reference from (m_z - m_y) to (M_z - M_y)
  const float sh = (hy && hz) ? ((p.mz - p.my) - (Mz - My)) * k : 0.f;
  float u = hz ? fz * fmaf(p.sy + p.w, sh, p.u) : (p.u != p.u ? p.u : 0.f);
  float w;
  if (!hz)
    w = -sy;  // no draft mass here: s_z = 0
  else if (!hy)
    w = p.w * fz;  // no target mass here: w = s_z
  else
    w = fmaf(p.w, fz, sy * expm1_nat(sh * kLn2));
#pragma unroll
  for (int o = SPAN / 2; o > 0; o >>= 1) {
    sy += __shfl_xor_sync(0xffffffffu, sy, o);
    w += __shfl_xor_sync(0xffffffffu, w, o);
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
  r.w = w;
  r.u = u;
  r.idx = best;
  r.zx = zx;
  r.abort = __any_sync(0xffffffffu, p.abort != 0) ? 1 : 0;
  return r;
}

// psi(d) = d - 1 + e^-d = sum_{n >= 2} (-d)^n / n!, d in nats.  With d the
// log ratio log q - log p of one vocabulary entry, q psi(d) = t - q + p, so
// sum_v q psi(d_v) = KL(q||p) - sum q + sum p: the same value as the KL when
// both rows are normalised, but to first order insensitive to an error in
// the row normalisers (a constant error e in d moves the sum by
// e sum q (1 - e^-d) = e (sum q - sum p) = 0).  For |d| < 1/8 the series,
// summed to d^7 (remainder below 2e-10 relative), gives q psi(d) without the
// cancellation of t - q + p; beyond, t - q + p (q, p from the exp2 unit) is
// within ~3e-5 of q psi(d) per entry, and such entries carry a KL of their
// own well above that.
__device__ __forceinline__ float psi_series(float d) {
  float c = -1.f / 5040.f;
  c = fmaf(c, d, 1.f / 720.f);
  c = fmaf(c, d, -1.f / 120.f);
  c = fmaf(c, d, 1.f / 24.f);
  c = fmaf(c, d, -1.f / 6.f);
  c = fmaf(c, d, 0.5f);
  return d * d * c;
}

// One entry's share of the clamped reverse KL in the form
//   sum_v [clamp(t_v, -c, c) - q_v + p_v]   (= sum_v clamp(t_v, -c, c), since
//   both rows sum to one), and of S - 1 = sum_v q_v a_v - sum_v q_v, in nats:
//   q d for an unclipped entry, -q for a clipped one.  Accumulating S - 1
//   rather than S keeps the normaliser's rounding (sum q = 1 + eta) out of
//   the gradient's q (a - S) term, whose scale is only that of log q - log p.
//   q = 2^(log2 q), d2 = log2 q - log2 p, log2 p = y k - Ct;  t / ln2 = q d2,
//   compared with c2 = c / ln2 as in the gradient passes.
// An entry with q = 0 has t = 0 (it contributes p); an entry whose term
// reaches the clip contributes +-c - q + p.  Branch-free but for the clip.
__device__ __forceinline__ void clamped_term(float q, float d2, float y, float k, float Ct, float c2, float c,
                                             float &rkl, float &Sm1) {
  const float p = ex2(fmaf(y, k, -Ct));
  if (q == 0.f) {
    rkl += p;
    return;
  }
  const float t2 = q * d2;
  const float d = d2 * kLn2;
  if (fabsf(t2) < c2) {
    const float near = q * psi_series(d);
    const float far = fmaf(q, d, p) - q;
    rkl += (fabsf(d) < 0.125f) ? near : far;
    Sm1 = fmaf(q, d, Sm1);
  } else {
    rkl += ((t2 > 0.f) ? c : -c) - q + p;
    Sm1 -= q;
  }
}

// Flag a row for the fix-up's loss-only recomputation (tag epoch ^
// kLossOnlyTag) unless it is already flagged for the full recomputation
// (tag epoch, stored by atomicExch from any CTA at any time): a
// compare-and-swap that gives up as soon as it sees the full tag.  Bounded:
// only a full-tag store can make it retry.
constexpr int32_t kLossOnlyTag = 0x40000000;
__device__ __forceinline__ void flag_loss_only(int32_t *f, int32_t epoch) {
  int32_t old = atomicAdd(f, 0);
  for (int it = 0; it < 4 && old != epoch; ++it) {
    const int32_t prev = atomicCAS(f, old, epoch ^ kLossOnlyTag);
    if (prev == old) return;
    old = prev;
  }
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
