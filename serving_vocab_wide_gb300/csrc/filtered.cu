// filtered.cu -- top-k / top-p filtered speculative verification (sm_103a).
//
// The pages verify with the full temperature softmax ("DFlash 阅读笔记：并行
// 起草、目标特征与精确验证" §5.2 eqs. (6)-(8), Algorithm 1).  Serving stacks
// usually filter both distributions first; this variant is not on the pages
// and follows this reading: both rows are filtered with the same (T, top_k,
// top_p) -- entries ordered by raw logit descending, smaller index first among
// equal logits; the first top_k kept; of those, the shortest prefix whose
// probability reaches top_p of their total kept; renormalised -- and the
// accept test, the residual and the bonus draw run on the filtered p' and q'.
// A drafted token outside the target's kept set has p'(x) = 0 and is
// rejected.  At T = 0 filtering keeps the argmax: greedy is unchanged.
//
// GPU design.  Two kernels.
//  1. filter_rows     one CTA of 1024 threads per logit row at a time
//                     (persistent).  One pass over the row (16-byte vectors)
//                     records each group of 8 entries' largest key in shared
//                     memory.  The K-th largest of those group maxima, tau, is
//                     a lower bound on the row's K-th largest entry, found by a
//                     radix select in shared memory (8-bit digits,
//                     warp-aggregated histogram atomics).  A second pass,
//                     which touches only the groups whose maximum reaches tau
//                     (mostly L2 hits), gathers every entry above tau (fewer
//                     than 8K of them) and, if needed, the entries equal to
//                     tau in index order (a block-wide scan).  The candidates
//                     are sorted in shared memory (bitonic, by logit then
//                     index), the first K kept, their probabilities summed in
//                     that order for the top-p cut (a fixed-order block scan),
//                     renormalised, and stored sorted by index.
//  2. filtered_finalize  one warp per request: validation, the accept tests
//                     (binary search of the drafted token in both lists),
//                     leftmost rejection, and the inverse-CDF draw over the
//                     rejected row's [p' - q']_+ (or the bonus row's p') in
//                     vocabulary order, over the stored lists only.
#include <cfloat>
#include <climits>
#include <cuda_runtime.h>
#include <type_traits>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace svw {

namespace {

constexpr int kFT = 256;  // threads of filter_rows (several CTAs per SM: some stream while others sort)
constexpr int kPer = kFilterMaxK / kFT;  // kept entries per thread in the top-p prefix
constexpr int kRankMax = 256;  // rank sorts (quadratic, no barriers) up to this many entries; bitonic above
constexpr int kFW = kFT / 32;
constexpr int kUnroll = 8;  // vectors per thread whose loads are in flight together

// order-preserving keys: a larger logit has a larger key; -0 is keyed as +0
__device__ __forceinline__ uint32_t key_of_bits16(uint32_t b) {
  if (b == 0x8000u) b = 0u;
  return ((b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u)) << 16;
}
__device__ __forceinline__ uint32_t key_of_f32(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// the logit of a key (bf16 keys hold the 16 bits in the upper half)
template <int DT>
__device__ __forceinline__ float value_of_key(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  if (DT == 1) b &= 0xffff0000u;
  return __uint_as_float(b);
}

template <int DT>
__device__ __forceinline__ uint32_t key_at(const char *row, int64_t v) {
  if (DT == 1) return key_of_bits16(__ldg(reinterpret_cast<const unsigned short *>(row) + v));
  return key_of_f32(__ldg(reinterpret_cast<const float *>(row) + v));
}

// the 8 keys of group g (entries 8g .. 8g+7; entries past V get key 0,
// below every real key) and whether any of them is NaN
template <int DT, bool VEC>
__device__ __forceinline__ void group_keys(const char *row, int64_t g, int64_t V, uint32_t (&k)[8], bool &nan,
                                           float &gmax) {
  const int64_t v0 = g * 8;
  nan = false;
  gmax = -INFINITY;
  float x[8];
  if (VEC && v0 + 8 <= V) {
    if (DT == 1) {
      const uint4 w = ld_vec(row + v0 * 2);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[2 * h] = __uint_as_float(ww[h] << 16);
        x[2 * h + 1] = __uint_as_float(ww[h] & 0xffff0000u);
      }
    } else {
      const uint4 w0 = ld_vec(row + v0 * 4), w1 = ld_vec(row + v0 * 4 + 16);
      const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(ww[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) k[e] = (DT == 1) ? key_of_bits16(__float_as_uint(x[e]) >> 16) : key_of_f32(x[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (v0 + e < V) {
        k[e] = key_at<DT>(row, v0 + e);
        x[e] = Elem<DT>::load(row, v0 + e);
      } else {
        k[e] = 0u;
        x[e] = -INFINITY;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    nan |= (x[e] != x[e]);
    gmax = fmaxf(gmax, x[e]);
  }
}

struct FSmem {
  uint32_t hist[256];
  float wf[kFW];
  uint32_t wu[kFW];
  int32_t ncand;
  int32_t ngl;
  int32_t bad;
  float mx;
  uint32_t tau;
  uint32_t need;
  uint32_t prefix;
  float zk, zf;
  int32_t np;
};

// block-wide inclusive scan of one value per thread (fixed order); the total
// is returned in *total
__device__ __forceinline__ uint32_t block_scan_u32(uint32_t v, FSmem &sm, uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.wu[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = (lane < kFW) ? sm.wu[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kFW) sm.wu[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t r = x + (warp ? sm.wu[warp - 1] : 0u);
  *total = sm.wu[kFW - 1];
  __syncthreads();
  return r;
}

// the same for floats (fixed order of additions), also giving the exclusive
// prefix: the inclusive value of the thread before (0 for thread 0)
__device__ __forceinline__ float block_scan_f32(float v, FSmem &sm, float *total, float *excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, y);
  }
  const float xe = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 31) sm.wf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    float w = (lane < kFW) ? sm.wf[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = __fadd_rn(w, y);
    }
    if (lane < kFW) sm.wf[lane] = w;
  }
  __syncthreads();
  const float base = warp ? sm.wf[warp - 1] : 0.f;
  const float r = warp ? __fadd_rn(base, x) : x;
  *excl = (lane == 0) ? base : (warp ? __fadd_rn(base, xe) : xe);
  *total = sm.wf[kFW - 1];
  __syncthreads();
  return r;
}

// histogram bin increment, aggregated over the lanes that share a bin
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(hist + bin, __popc(peers));
}

// bitonic sort of P (a power of two) entries (key, idx, val) in shared memory:
// DESC: key descending then idx ascending; otherwise idx ascending
template <bool DESC>
__device__ void bitonic(uint32_t *key, int32_t *idx, float *val, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P; i += kFT) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;  // this pair ends in the wanted order
          bool after;                       // entry i belongs after entry j
          if (DESC) after = (key[i] < key[j]) || (key[i] == key[j] && idx[i] > idx[j]);
          else after = idx[i] > idx[j];
          if (after == up) {
            const uint32_t tk = key[i];
            key[i] = key[j];
            key[j] = tk;
            const int32_t ti = idx[i];
            idx[i] = idx[j];
            idx[j] = ti;
            if (val) {
              const float tv = val[i];
              val[i] = val[j];
              val[j] = tv;
            }
          }
        }
      }
      __syncthreads();
    }
  }
}

// the largest of the 8 entries of vector q (entries 8q .. 8q+7; entries past
// V count as -inf) and whether any of them is NaN
template <int DT, bool VEC>
__device__ __forceinline__ void vector_max(const char *row, int64_t q, int64_t V, float &mx, bool &nan) {
  const int64_t v0 = q * 8;
  if (VEC && v0 + 8 <= V) {
    if (DT == 1) {
      const uint4 w = ld_vec(row + v0 * 2);
      const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w));
      nan = bf16x2_nan(m2) != 0;
      const float2 f = bf16x2_f2(m2);
      mx = fmaxf(f.x, f.y);
    } else {
      const uint4 w0 = ld_vec(row + v0 * 4), w1 = ld_vec(row + v0 * 4 + 16);
      const float x[8] = {__uint_as_float(w0.x), __uint_as_float(w0.y), __uint_as_float(w0.z),
                          __uint_as_float(w0.w), __uint_as_float(w1.x), __uint_as_float(w1.y),
                          __uint_as_float(w1.z), __uint_as_float(w1.w)};
      mx = -INFINITY;
      nan = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        nan |= (x[e] != x[e]);
        mx = fmaxf(mx, x[e]);
      }
    }
  } else {
    mx = -INFINITY;
    nan = false;
    for (int e = 0; e < 8; ++e)
      if (v0 + e < V) {
        const float x = Elem<DT>::load(row, v0 + e);
        nan |= (x != x);
        mx = fmaxf(mx, x);
      }
  }
}

// the rank of candidate t among the C in (key descending, index ascending)
// order: how many candidates come before it
__device__ __forceinline__ int rank_desc(const uint32_t *key, const int32_t *idx, int C, int t) {
  const uint32_t kt = key[t];
  const int32_t it = idx[t];
  int r = 0;
  for (int j = 0; j < C; ++j) {
    const uint32_t kj = key[j];
    r += (kj > kt || (kj == kt && idx[j] < it)) ? 1 : 0;
  }
  return r;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kFT, 4) filter_rows(FilterArgs a) {
  using KeyT = typename std::conditional<DT == 1, unsigned short, uint32_t>::type;
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ FSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;
  const int gv = a.gs / 8;                  // 16-byte (8-entry) vectors per group, a power of two <= 16
  const int64_t NVec = (V + 7) / 8;         // 8-entry vectors of the row
  const int64_t NG = (NVec + gv - 1) / gv;  // groups
  const int kCand = a.cand;                 // gs x (top_k rounded up to a power of two)
  uint32_t *ckey = reinterpret_cast<uint32_t *>(dyn);
  int32_t *cidx = reinterpret_cast<int32_t *>(ckey + kCand);
  uint32_t *skey = reinterpret_cast<uint32_t *>(cidx + kCand);  // [kFilterMaxK] in logit order
  int32_t *sidx = reinterpret_cast<int32_t *>(skey + kFilterMaxK);
  float *spv = reinterpret_cast<float *>(sidx + kFilterMaxK);  // their probabilities (unnormalised)
  KeyT *gkey = reinterpret_cast<KeyT *>(spv + kFilterMaxK);
  const int64_t nrows = a.rows_t + a.R;
  const uint32_t K = static_cast<uint32_t>(min(static_cast<int64_t>(a.top_k), V));

  for (int64_t r = blockIdx.x; r < nrows; r += gridDim.x) {
    const char *row = (r < a.rows_t) ? static_cast<const char *>(a.target) + r * V * Elem<DT>::kSize
                                     : static_cast<const char *>(a.draft) + (r - a.rows_t) * V * Elem<DT>::kSize;
    // ---- pass 1: each group's largest entry (as a key), the row maximum, NaN ----
    // thread t of a round holds vector t; a group is gv consecutive lanes
    float mx = -INFINITY;
    bool nan = false;
    for (int64_t q0 = 0; q0 < NVec; q0 += static_cast<int64_t>(kUnroll) * kFT) {
      float vm[kUnroll];
      bool vn[kUnroll];
      if (VEC && DT == 1 && q0 + static_cast<int64_t>(kUnroll) * kFT <= V / 8) {
        // a whole round of full vectors: every load in flight before any arithmetic
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) w[u] = ld_vec(row + (q0 + static_cast<int64_t>(u) * kFT + tid) * 16);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(w[u].x, w[u].y), bf16x2_max_nan(w[u].z, w[u].w));
          vn[u] = bf16x2_nan(m2) != 0;
          const float2 f = bf16x2_f2(m2);
          vm[u] = fmaxf(f.x, f.y);
        }
      } else {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t q = q0 + static_cast<int64_t>(u) * kFT + tid;
          vm[u] = -INFINITY;
          vn[u] = false;
          if (q < NVec) vector_max<DT, VEC>(row, q, V, vm[u], vn[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t q = q0 + static_cast<int64_t>(u) * kFT + tid;
        nan |= vn[u];
        mx = fmaxf(mx, vm[u]);
        float gm = vm[u];
        for (int o = 1; o < gv; o <<= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
        if ((lane & (gv - 1)) == 0 && q < NVec) {
          const uint32_t kk = (DT == 1) ? key_of_bits16(__float_as_uint(gm) >> 16) : key_of_f32(gm);
          gkey[q / gv] = static_cast<KeyT>(DT == 1 ? (kk >> 16) : kk);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int anynan = __syncthreads_or(nan ? 1 : 0);
    if (lane == 0) sm.wf[warp] = mx;
    if (tid == 0) sm.ncand = 0;
    __syncthreads();
    if (warp == 0) {
      float w = (lane < kFW) ? sm.wf[lane] : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
      if (lane == 0) {
        sm.mx = w;
        sm.bad = (anynan || !(w > -INFINITY && w <= FLT_MAX)) ? 1 : 0;
      }
    }
    __syncthreads();
    if (sm.bad) {
      if (tid == 0) a.cnt[r] = -1;
      __syncthreads();
      continue;
    }
    const float m = sm.mx;

    // ---- tau: the K-th largest group maximum (radix select, 8-bit digits) ----
    constexpr int kBits = (DT == 1) ? 16 : 32;
    uint32_t prefix = 0, pmask = 0, need = K;
    if (static_cast<int64_t>(K) < NG) {
      for (int shift = kBits - 8; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kFT) sm.hist[b] = 0;
        __syncthreads();
        for (int64_t g0 = 0; g0 < NG; g0 += kFT) {
          const int64_t g = g0 + tid;
          const uint32_t kg = (g < NG) ? static_cast<uint32_t>(gkey[g]) : 0u;
          hist_add(sm.hist, (kg >> shift) & 255u, g < NG && (kg & pmask) == prefix);
        }
        __syncthreads();
        if (warp == 0) {
          // bins from the top: the first whose cumulative count reaches need
          uint32_t above = 0, sel = 0, sel_above = 0;
          bool found = false;
          for (int c = 0; c < 8 && !found; ++c) {
            const uint32_t h = sm.hist[255 - (c * 32 + lane)];
            uint32_t x = h;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
              if (lane >= o) x += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, above + x >= need);
            if (hit) {
              const int l = __ffs(hit) - 1;
              sel = 255u - static_cast<uint32_t>(c * 32 + l);
              sel_above = above + __shfl_sync(0xffffffffu, x - h, l);
              found = true;
            } else {
              above += __shfl_sync(0xffffffffu, x, 31);
            }
          }
          if (lane == 0) {
            sm.prefix = prefix | (sel << shift);
            sm.need = need - sel_above;
          }
        }
        __syncthreads();
        prefix = sm.prefix;
        need = sm.need;
        pmask |= 255u << shift;
        __syncthreads();
      }
    }
    // as a full 32-bit key; when every group qualifies, 0 (below every real key)
    const uint32_t tau = (static_cast<int64_t>(K) < NG) ? ((DT == 1) ? (prefix << 16) : prefix) : 1u;

    // ---- gather every entry at or above tau, from the vectors of the groups that reach it ----
    const int lgv = __ffs(gv) - 1;
    auto gkey32 = [&](int64_t g) -> uint32_t {
      return (DT == 1) ? (static_cast<uint32_t>(gkey[g]) << 16) : static_cast<uint32_t>(gkey[g]);
    };
    auto take = [&](int64_t q) {  // the entries of vector q at or above tau
      uint32_t k[8];
      bool gn;
      float gm;
      group_keys<DT, VEC>(row, q, V, k, gn, gm);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (k[e] >= tau) {
          const int p = atomicAdd(&sm.ncand, 1);
          if (p < kCand) {
            ckey[p] = k[e];
            cidx[p] = static_cast<int32_t>(q * 8 + e);
          }
        }
    };
    // the groups that reach tau (about top_k of them), listed in sidx first
    if (tid == 0) sm.ngl = 0;
    __syncthreads();
    for (int64_t g = tid; g < NG; g += kFT)
      if (gkey32(g) >= tau) {
        const int p = atomicAdd(&sm.ngl, 1);
        if (p < kFilterMaxK) sidx[p] = static_cast<int32_t>(g);
      }
    __syncthreads();
    const int ngl = sm.ngl;
    if (ngl <= kFilterMaxK) {
      for (int j = tid; j < ngl * gv; j += kFT) {
        const int64_t q = static_cast<int64_t>(sidx[j >> lgv]) * gv + (j & (gv - 1));
        if (q < NVec) take(q);
      }
    } else {
      for (int64_t q = tid; q < NVec; q += kFT)
        if (gkey32(q >> lgv) >= tau) take(q);
    }
    __syncthreads();
    if (sm.ncand > kCand) {
      // many entries equal to tau: every entry above tau (fewer than gs K),
      // then those equal to tau in index order while fewer than K
      __syncthreads();
      if (tid == 0) sm.ncand = 0;
      __syncthreads();
      for (int64_t q = tid; q < NVec; q += kFT) {
        if (gkey32(q >> lgv) > tau) {
          uint32_t k[8];
          bool gn;
          float gm;
          group_keys<DT, VEC>(row, q, V, k, gn, gm);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (k[e] > tau) {
              const int p = atomicAdd(&sm.ncand, 1);
              if (p < kCand) {
                ckey[p] = k[e];
                cidx[p] = static_cast<int32_t>(q * 8 + e);
              }
            }
        }
      }
      __syncthreads();
      const uint32_t above = static_cast<uint32_t>(sm.ncand);
      const uint32_t want = (above < K) ? K - above : 0u;
      uint32_t base = 0;
      for (int64_t q0 = 0; q0 < NVec && base < want; q0 += kFT) {
        const int64_t q = q0 + tid;
        uint32_t k[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint32_t c = 0;
        if (q < NVec) {
          if (gkey32(q >> lgv) >= tau) {
            bool gn;
            float gm;
            group_keys<DT, VEC>(row, q, V, k, gn, gm);
#pragma unroll
            for (int e = 0; e < 8; ++e) c += (k[e] == tau) ? 1u : 0u;
          }
        }
        uint32_t tot;
        const uint32_t incl = block_scan_u32(c, sm, &tot);
        uint32_t rank = base + incl - c;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c && k[e] == tau) {
            if (rank < want) {
              ckey[above + rank] = k[e];
              cidx[above + rank] = static_cast<int32_t>(q * 8 + e);
            }
            ++rank;
          }
        base += tot;
      }
      __syncthreads();
      if (tid == 0) sm.ncand = static_cast<int32_t>(above + min(base, want));
      __syncthreads();
    }
    const int C = min(sm.ncand, kCand);
    const int Kc = min(static_cast<int>(K), C);
    // ---- the first K candidates in (logit descending, index ascending) order ----
    if (C <= kRankMax) {
      // rank sort: every candidate counts those before it
      for (int t = tid; t < C; t += kFT) {
        const int rk = rank_desc(ckey, cidx, C, t);
        if (rk < Kc) {
          skey[rk] = ckey[t];
          sidx[rk] = cidx[t];
        }
      }
      __syncthreads();
    } else {
      int P = 1;
      while (P < C) P <<= 1;
      for (int i = C + tid; i < P; i += kFT) {
        ckey[i] = 0u;
        cidx[i] = INT32_MAX;
      }
      __syncthreads();
      bitonic<true>(ckey, cidx, nullptr, P);
      for (int t = tid; t < Kc; t += kFT) {
        skey[t] = ckey[t];
        sidx[t] = cidx[t];
      }
      __syncthreads();
    }
    // ---- probabilities in that order; the top-p cut; renormalised ----
    // thread t holds entries kPer t .. kPer t + kPer - 1; the prefix is fixed-order
    for (int t = tid; t < Kc; t += kFT) spv[t] = ex2(__fmul_rn(__fsub_rn(value_of_key<DT>(skey[t]), m), a.k));
    __syncthreads();
    const int e0 = kPer * tid;
    float loc[kPer];
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      run = __fadd_rn(run, (e0 + e < Kc) ? spv[e0 + e] : 0.f);
      loc[e] = run;
    }
    float zk, excl;
    block_scan_f32(run, sm, &zk, &excl);
    float cum[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) cum[e] = __fadd_rn(excl, loc[e]);
    int np = Kc;
    if (a.top_p < 1.f) {
      const float thr = __fmul_rn(a.top_p, zk);
      uint32_t below = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) below += (e0 + e < Kc && cum[e] < thr) ? 1u : 0u;
      uint32_t nb;
      block_scan_u32(below, sm, &nb);
      np = min(Kc, static_cast<int>(nb) + 1);
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (e0 + e == np - 1) sm.zf = cum[e];
    __syncthreads();
    const float zf = sm.zf;
    // ---- stored sorted by index, p' = p / kept mass ----
    if (np <= kRankMax) {
      for (int t = tid; t < np; t += kFT) {
        const int32_t it = sidx[t];
        int rk = 0;
        for (int j = 0; j < np; ++j) rk += (sidx[j] < it) ? 1 : 0;
        a.lidx[r * kFilterMaxK + rk] = it;
        a.lp[r * kFilterMaxK + rk] = __fdiv_rn(spv[t], zf);
      }
    } else {
      int Q = 1;
      while (Q < np) Q <<= 1;
      for (int t = np + tid; t < Q; t += kFT) sidx[t] = INT32_MAX;
      __syncthreads();
      bitonic<false>(skey, sidx, spv, Q);
      for (int t = tid; t < np; t += kFT) {
        a.lidx[r * kFilterMaxK + t] = sidx[t];
        a.lp[r * kFilterMaxK + t] = __fdiv_rn(spv[t], zf);
      }
    }
    if (tid == 0) a.cnt[r] = np;
    __syncthreads();
  }
}

// p' of entry v in a stored list (0 if v is not kept): binary search
__device__ __forceinline__ float list_prob(const int32_t *li, const float *lp, int n, int32_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldcg(li + mid) < v) lo = mid + 1;
    else hi = mid;
  }
  return (lo < n && __ldcg(li + lo) == v) ? __ldcg(lp + lo) : 0.f;
}

constexpr int kFinReqPerCta = 4;  // one warp per request

__global__ void __launch_bounds__(32 * kFinReqPerCta) filtered_finalize(FilterArgs a) {
  const int lane = threadIdx.x & 31;
  const int32_t i = blockIdx.x * kFinReqPerCta + (threadIdx.x >> 5);
  if (i >= a.N) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t c_i = __ldg(a.cu + i), c_e = __ldg(a.cu + i + 1);
  const bool csr_ok = (__ldg(a.cu) == 0) && (static_cast<int64_t>(__ldg(a.cu + a.N)) == a.R);
  const bool len_ok = csr_ok && (c_e - c_i >= 1 && c_e - c_i <= a.max_len && c_i >= 0 && c_e <= a.R);
  const int32_t L = len_ok ? static_cast<int32_t>(c_e - c_i) : 0;
  const int64_t t0 = c_i + i, d0 = a.rows_t + c_i;  // stored-list rows
  auto reject = [&]() {
    if (lane == 0) {
      a.accept_len[i] = -1;
      a.next_token[i] = -1;
      if (a.status) atomicOr(a.status, SVW_DEV_BAD_INPUT);
    }
  };
  if (!len_ok) {
    reject();
    return;
  }
  // every row of the request must have been filtered (finite logits)
  int bad = 0;
  for (int q = lane; q <= 2 * L; q += 32) {
    const int64_t rr = (q <= L) ? (t0 + q) : (d0 + q - L - 1);
    bad |= (__ldcg(a.cnt + rr) < 0) ? 1 : 0;
  }
  int32_t x = 0;
  if (lane < L) {
    x = __ldg(a.tokens + c_i + lane);
    bad |= (x < 0 || static_cast<int64_t>(x) >= a.V) ? 1 : 0;
  }
  if (__any_sync(0xffffffffu, bad)) {
    reject();
    return;
  }
  // ---- accept tests on the filtered distributions ----
  bool acc = true;
  if (lane < L) {
    const int64_t tr = t0 + lane, dr = d0 + lane;
    const float p = list_prob(a.lidx + tr * kFilterMaxK, a.lp + tr * kFilterMaxK, __ldcg(a.cnt + tr), x);
    const float q = list_prob(a.lidx + dr * kFilterMaxK, a.lp + dr * kFilterMaxK, __ldcg(a.cnt + dr), x);
    const float thr = (p == 0.f) ? 0.f : ((q > 0.f) ? fminf(1.f, __fdiv_rn(p, q)) : 1.f);
    const float u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(lane), 0u);
    acc = u < thr;
  }
  const unsigned rej = __ballot_sync(0xffffffffu, !acc);
  const int32_t js = rej ? (__ffs(rej) - 1) : L;
  // ---- the next token: [p' - q']_+ at the rejected row, or p' of the bonus row ----
  const int64_t tr = t0 + js;
  const int32_t *ti = a.lidx + tr * kFilterMaxK;
  const float *tp = a.lp + tr * kFilterMaxK;
  const int n = __ldcg(a.cnt + tr);
  const int64_t dr = d0 + js;
  const bool resid = js < L;
  const int nd = resid ? __ldcg(a.cnt + dr) : 0;
  const int32_t *di = a.lidx + dr * kFilterMaxK;
  const float *dp = a.lp + dr * kFilterMaxK;
  const float w = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(js), 1u);
  // the draft row's list in shared memory: every q' lookup of the draw is a
  // binary search there rather than a chain of global loads
  __shared__ int32_t sdi[kFinReqPerCta][kFilterMaxK];
  __shared__ float sdp[kFinReqPerCta][kFilterMaxK];
  const int wq = threadIdx.x >> 5;
  for (int t = lane; t < nd; t += 32) {
    sdi[wq][t] = __ldcg(di + t);
    sdp[wq][t] = __ldcg(dp + t);
  }
  __syncwarp();
  auto weight = [&](int t, bool use_q) -> float {  // entry t of the target row's list
    const float p = __ldcg(tp + t);
    if (!use_q) return p;
    const int32_t v = __ldcg(ti + t);
    int lo = 0, hi = nd;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sdi[wq][mid] < v) lo = mid + 1;
      else hi = mid;
    }
    const float q = (lo < nd && sdi[wq][lo] == v) ? sdp[wq][lo] : 0.f;
    return fmaxf(__fsub_rn(p, q), 0.f);
  };
  int32_t tok = -1;
  for (int attempt = 0; attempt < 2 && tok < 0; ++attempt) {
    const bool use_q = resid && attempt == 0;
    // total in a fixed order: 32-entry chunks, lanes by a butterfly-free
    // inclusive scan, chunks sequentially
    float Z = 0.f;
    for (int c0 = 0; c0 < n; c0 += 32) {
      float x2 = (c0 + lane < n) ? weight(c0 + lane, use_q) : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x2, o);
        if (lane >= o) x2 = __fadd_rn(x2, y);
      }
      Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, x2, 31));
    }
    if (use_q && !(Z > 0.f)) continue;  // no residual mass after rounding: draw from p'
    const float t = __fmul_rn(w, Z);
    float base = 0.f;
    int32_t last = -1;
    for (int c0 = 0; c0 < n && tok < 0; c0 += 32) {
      const float wt = (c0 + lane < n) ? weight(c0 + lane, use_q) : 0.f;
      float x2 = wt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x2, o);
        if (lane >= o) x2 = __fadd_rn(x2, y);
      }
      const unsigned pos = __ballot_sync(0xffffffffu, wt > 0.f);
      if (pos) last = __ldcg(ti + c0 + 31 - __clz(pos));
      const unsigned hit = __ballot_sync(0xffffffffu, wt > 0.f && __fadd_rn(base, x2) > t);
      if (hit) tok = __ldcg(ti + c0 + __ffs(hit) - 1);
      base = __fadd_rn(base, __shfl_sync(0xffffffffu, x2, 31));
    }
    if (tok < 0) tok = last;  // no crossing after rounding: the last entry with weight
  }
  if (lane == 0) {
    a.accept_len[i] = js;
    a.next_token[i] = tok;
  }
}

}  // namespace

// top_k rounded up to a power of two
static int pow2_at_least(int32_t k) {
  int P = 1;
  while (P < k) P <<= 1;
  return P;
}

// entries per group: as large as the candidate space allows (every entry above
// tau lies in one of fewer than top_k groups), between 8 and 128
int filter_group(int32_t top_k) {
  int gs = 2048 / pow2_at_least(top_k);
  if (gs < 8) gs = 8;
  if (gs > 128) gs = 128;
  return gs;
}

int filter_candidates(int32_t top_k) { return filter_group(top_k) * pow2_at_least(top_k); }

size_t filter_smem_bytes(int64_t V, int esize, int32_t top_k) {
  const int64_t gv = filter_group(top_k) / 8;
  const int64_t NG = ((V + 7) / 8 + gv - 1) / gv;
  return static_cast<size_t>(filter_candidates(top_k)) * 8 + static_cast<size_t>(kFilterMaxK) * 12 +
         static_cast<size_t>(NG) * (esize == 2 ? 2 : 4);
}

cudaError_t launch_filtered(const FilterArgs &a, int dtype, bool vec, cudaStream_t st) {
  const int esize = (dtype == SVW_BF16) ? 2 : 4;
  const size_t smem = filter_smem_bytes(a.V, esize, a.top_k);
  auto pick = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kFT, smem)) != cudaSuccess) return e;
    int64_t grid = static_cast<int64_t>(nsm) * (occ > 0 ? occ : 1);
    const int64_t rows = a.rows_t + a.R;
    if (grid > rows) grid = rows;
    if (grid < 1) grid = 1;
    void *tm = timer_before("filter_rows", st);
    kern<<<static_cast<unsigned>(grid), kFT, smem, st>>>(a);
    timer_after(tm, st);
    return cudaGetLastError();
  };
  cudaError_t e;
  if (dtype == SVW_BF16) e = vec ? pick(filter_rows<1, true>) : pick(filter_rows<1, false>);
  else e = vec ? pick(filter_rows<0, true>) : pick(filter_rows<0, false>);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>((a.N + kFinReqPerCta - 1) / kFinReqPerCta), 1, 1);
  cfg.blockDim = dim3(32 * kFinReqPerCta, 1, 1);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *tm = timer_before("filtered_finalize", st);
  e = cudaLaunchKernelEx(&cfg, filtered_finalize, a);
  timer_after(tm, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace svw
