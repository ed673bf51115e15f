// svw_device.cuh -- device helpers shared by the verification and OPD kernels:
// element loads, special-function-unit exp2/log2, warp reductions, Philox.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace svw {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// special-function unit (PTX ISA instructions, flush-to-zero)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// element access.  DT = 1: bf16 stored as uint16 bits; DT = 0: fp32.
// ---------------------------------------------------------------------------
template <int DT>
struct Elem;

template <>
struct Elem<1> {
  static constexpr int kSize = 2;
  static constexpr int kPerVec = 8;  // elements per 16-byte vector
  __device__ __forceinline__ static float load(const void *base, int64_t idx) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(base) + idx);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  // plain load (any state space, e.g. shared memory)
  __device__ __forceinline__ static float load_plain(const void *base, int64_t idx) {
    const unsigned short b = reinterpret_cast<const unsigned short *>(base)[idx];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  // unpack one 16-byte vector into 8 floats, in index order
  __device__ __forceinline__ static void unpack(const uint4 &w, float *o) {
    o[0] = __uint_as_float(w.x << 16);
    o[1] = __uint_as_float(w.x & 0xffff0000u);
    o[2] = __uint_as_float(w.y << 16);
    o[3] = __uint_as_float(w.y & 0xffff0000u);
    o[4] = __uint_as_float(w.z << 16);
    o[5] = __uint_as_float(w.z & 0xffff0000u);
    o[6] = __uint_as_float(w.w << 16);
    o[7] = __uint_as_float(w.w & 0xffff0000u);
  }
};

template <>
struct Elem<0> {
  static constexpr int kSize = 4;
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static float load(const void *base, int64_t idx) {
    return __ldg(reinterpret_cast<const float *>(base) + idx);
  }
  __device__ __forceinline__ static float load_plain(const void *base, int64_t idx) {
    return reinterpret_cast<const float *>(base)[idx];
  }
  __device__ __forceinline__ static void unpack(const uint4 &w, float *o) {
    o[0] = __uint_as_float(w.x);
    o[1] = __uint_as_float(w.y);
    o[2] = __uint_as_float(w.z);
    o[3] = __uint_as_float(w.w);
  }
};

// the two bf16 values of a 32-bit word as floats (low half first)
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// elementwise bf16 max of two packed words (a NaN half yields the other)
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r =
      __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&a), *reinterpret_cast<const __nv_bfloat162 *>(&b));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// elementwise bf16 max that propagates NaN
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                       *reinterpret_cast<const __nv_bfloat162 *>(&b));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// nonzero if either bf16 half of w is a NaN
__device__ __forceinline__ uint32_t bf16x2_nan(uint32_t w) {
  return ((w & 0x7fff7fffu) + 0x007f007fu) & 0x80008000u;
}

// shared-memory / mbarrier / bulk-copy primitives
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait on an mbarrier phase: false if the clock deadline passed first
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
// The deadline in force: each translation unit has its own copy, and every
// copy registers its setter at load time (register_wait_limit, api.cu), so
// that svw_set_wait_limit reaches all of them.  The registry is a weak
// reference: a program built from this header alone keeps the default.
static __constant__ long long c_wait_limit = kWaitCycles;
__attribute__((weak)) cudaError_t register_wait_limit(cudaError_t (*set)(long long));
static cudaError_t set_wait_limit_here(long long v) { return cudaMemcpyToSymbol(c_wait_limit, &v, sizeof(v)); }
[[maybe_unused]] static const cudaError_t wait_limit_registered =
    register_wait_limit ? register_wait_limit(&set_wait_limit_here) : cudaSuccess;
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, uint32_t parity) {
  const long long t0 = clock64();
  const long long limit = c_wait_limit;
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}
// the accept test u < min(1, p(x)/q(x)) of speculative verification from the
// raw logits at x and the row statistics (m: maximum, l = log2 of the sum of
// 2^((x - m) k)): log2 p(x) = (y_x - m_T) k - l_T, log2 q(x) = (z_x - m_D) k - l_D
__device__ __forceinline__ bool accept_token(float u, float yx, float zx, float mT, float lT, float mD, float lD,
                                             float k) {
  float thr;
  if (zx == -INFINITY) {
    thr = 1.f;  // q(x) = 0: accept
  } else {
    const float dl = __fsub_rn(__fmul_rn(__fsub_rn(__fsub_rn(yx, mT), __fsub_rn(zx, mD)), k), __fsub_rn(lT, lD));
    thr = (dl >= 0.f) ? 1.f : ex2(dl);
  }
  return u < thr;
}

// ---------------------------------------------------------------------------
// thread-block clusters: named barriers, peer shared memory, async stores
// ---------------------------------------------------------------------------
// named barriers: some warps arrive, others wait
__device__ __forceinline__ void named_arrive(int id, int nt) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nt) : "memory"); }
__device__ __forceinline__ void named_sync(int id, int nt) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nt) : "memory"); }
// shared::cluster address of the same shared variable in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 32-bit store into a peer's shared memory (ordered by the next cluster barrier)
__device__ __forceinline__ void st_cluster_b32(uint32_t dst, uint32_t v) {
  asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(dst), "r"(v) : "memory");
}
// every thread of every CTA of the cluster (release / acquire)
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// 16-byte store into a peer's shared memory that completes 16 bytes of the
// transaction count of the peer's mbarrier (no fence, no cluster barrier)
__device__ __forceinline__ void st_async16(uint32_t dst, const uint4 &v, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(dst),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(mbar)
               : "memory");
}
// the same for one 32-bit word (4 bytes of the transaction count)
__device__ __forceinline__ void st_async4(uint32_t dst, uint32_t v, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst), "r"(v),
               "r"(mbar)
               : "memory");
}

// 1-D bulk asynchronous copy global -> this CTA's shared memory, completion
// counted (in bytes) on the mbarrier
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         unsigned long long *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// streaming 16-byte load: read-only path, no L1 allocation
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// plain 16-byte load through L1/L2 (data likely resident in L2)
__device__ __forceinline__ uint4 ld_vec(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

// streaming 16-byte store (evict-first)
__device__ __forceinline__ void st_stream(float *p, float a, float b, float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// ---------------------------------------------------------------------------
// (max, sum-of-exp2) pairs: s = sum_i 2^((x_i - m) * k).  Combining is
// commutative bit-for-bit (IEEE addition and max are), so butterfly
// reductions give every lane the same value.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void lse_combine(float &m, float &s, float m2, float s2, float k) {
  if (!(s == s) || !(s2 == s2) || !(m == m) || !(m2 == m2)) {  // NaN anywhere poisons the pair
    m = __int_as_float(0x7fffffff);
    s = __int_as_float(0x7fffffff);
    return;
  }
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {  // both empty / all -inf
    m = M;
    s = 0.f;
    return;
  }
  const float a = (m == -INFINITY) ? 0.f : __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, M), k)));
  const float b = (m2 == -INFINITY) ? 0.f : __fmul_rn(s2, ex2(__fmul_rn(__fsub_rn(m2, M), k)));
  m = M;
  s = __fadd_rn(a, b);
}

__device__ __forceinline__ void warp_lse(float &m, float &s, float k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2, k);
  }
}

// argmax with "smallest index wins"; idx == INT32_MAX means "nothing seen"
__device__ __forceinline__ void amax_combine(float &v, int32_t &i, float v2, int32_t i2) {
  if (i2 == INT32_MAX) return;
  if (i == INT32_MAX || v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_amax(float &v, int32_t &i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int32_t i2 = __shfl_xor_sync(0xffffffffu, i, o);
    amax_combine(v, i, v2, i2);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of two 32x32
// multiplies; the key advances by the Weyl constants between rounds.
// Returns output word 0 for counter {c0, c1, c2, 0}.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(uint64_t seed, uint32_t c0, uint32_t c1,
                                                 uint32_t c2) {
  uint32_t x0 = c0, x1 = c1, x2 = c2, x3 = 0u;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi_a = __umulhi(0xD2511F53u, x0), lo_a = 0xD2511F53u * x0;
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, x2), lo_b = 0xCD9E8D57u * x2;
    const uint32_t y0 = hi_b ^ x1 ^ k0;
    const uint32_t y2 = hi_a ^ x3 ^ k1;
    x0 = y0;
    x1 = lo_b;
    x2 = y2;
    x3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return x0;
}

// 24-bit uniform in [0, 1), exact in fp32
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t i, uint32_t j,
                                                uint32_t stream) {
  return static_cast<float>(philox_word0(seed, i, j, stream) >> 8) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// warp reductions over a span of 16-byte vectors held in shared memory (warp
// wid of CW reads vectors vi = wid*32 + lane + q*CW*32)
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

}  // namespace svw
