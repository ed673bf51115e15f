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
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
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

}  // namespace svw
