// lengthhead.cu -- the adaptive length head: forward and label.
//
// "AdaFlash: Taming Variance in Diffusion Speculative Decoding", "Algorithm
// 3: Adaptive Length Head, Forward Pass" ("AdaFlash：基于在策略蒸馏扩散草稿器的
// 自适应投机解码" §2.2), per request i with drafter hidden states h_i (k x H):
//   h'_p = SiLU(W1 h_i[p] + b1)   (W1: H' x H)    -- a dense contraction
//   hbar = mean_p h'_p
//   a_hat = sigmoid(w2 . hbar + b2),  k_hat = clamp(floor(gamma a_hat k), 1, k)
// and "Online Update of the Length Head, Derived": a* = accept_len / L,
// loss = (a_hat - a*)^2.
//
// GPU design.  The projection of all M = N k positions, Y = X W1^T with X the
// [M, H] hidden states, is the one dense contraction of the head and runs on
// the tensor cores: tcgen05.mma (kind::f16, bf16 operands, fp32 accumulator
// in tensor memory), both operands K-major, staged by TMA (cp.async.bulk.tensor
// with the 128-byte swizzle).  A CTA owns a 128-row tile of X and a 256-column
// tile of W1 (H' <= 256: all of it) over one quarter of K = H, so that 128
// CTAs share the work at the benchmark's shape; a thread-block cluster holds
// four row tiles with the same K quarter, which load one quarter each of
// their common W1 tile and multicast it to all four (W1 is re-read by every
// row tile: without this it is two thirds of the traffic into the SMs).  X tiles come from DRAM through a seven-stage ring,
// W1 tiles through a three-stage ring, each fed by its own producer thread;
// one thread issues the MMAs.  The fp32 partial tile leaves tensor memory
// through shared memory (a transpose for coalesced stores) into the caller's
// workspace.  A second kernel, one CTA per request and a programmatic
// dependent of the first, sums the four K partials of each of the request's
// positions in a fixed order and finishes the head: bias, SiLU, the mean
// over positions, the dot with w2, sigmoid, gamma, floor and clamp.
//
// Every mbarrier wait is bounded by a clock deadline; a CTA that gives up
// stops issuing work, lets the copies it started land (again bounded), writes
// NaN for its rows, still joins every cluster barrier and frees its tensor
// memory.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace cg = cooperative_groups;

namespace svw {

namespace {

constexpr int kTM = 128;          // rows of X per CTA (the MMA's M)
constexpr int kTN = 256;          // columns of W1 rows per CTA (the MMA's N at most)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int kStagesA = 7;       // X tiles come from DRAM: the deeper ring
constexpr int kStagesB = 3;       // W1 tiles mostly hit L2
constexpr int kKSplit = 4;        // K quarters
constexpr int kMGroup = 4;        // row tiles per cluster, sharing their W1 tiles
constexpr int kCluster = kMGroup;
constexpr int kMmaThreads = 128;  // four warps: TMEM lanes 0-127
constexpr int kStageA = kTM * kBK * 2;  // 16 KB

// Dynamic shared memory: the two rings, reused after the main loop for the
// partial tile on its way out (128 rows of NT + 4 floats: rows stay 16-byte
// aligned, and with 16-byte stores the eight rows of one store phase fall on
// distinct banks).
__host__ __device__ constexpr int ringB_off() { return kStagesA * kStageA; }
__host__ __device__ constexpr int ring_bytes(int NT) { return kStagesA * kStageA + kStagesB * NT * kBK * 2; }
__host__ __device__ constexpr int tile_pitch(int NT) { return NT + 4; }
__host__ __device__ constexpr int tile_bytes(int NT) { return kTM * tile_pitch(NT) * 4; }
__host__ __device__ constexpr int head_smem(int NT) {
  return (ring_bytes(NT) > tile_bytes(NT) ? ring_bytes(NT) : tile_bytes(NT)) + 1024;
}

// ---------------------------------------------------------------------------
// PTX wrappers (tensor memory, tcgen05 MMA, TMA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// the same box delivered to every CTA of ctamask (same shared-memory offset,
// each CTA's own mbarrier at the same offset)
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                               uint32_t mbar, uint16_t ctamask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, "
      "{%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar), "h"(ctamask)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 in, fp32 accumulate (one thread issues)
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// the mbarrier completes one arrival once every MMA issued before it is done
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}

// one arrival on the mbarrier at this offset in every CTA of ctamask once
// every MMA issued before it is done
__device__ __forceinline__ void mma_commit_mc(uint32_t mbar, uint16_t ctamask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                   "r"(mbar),
               "h"(ctamask)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Shared-memory matrix descriptor of a K-major operand tile as the TMA's
// 128-byte swizzle lays it out: rows of 128 bytes (64 bf16 of K), eight-row
// swizzle atoms of 1024 bytes one after another along M (or N).  Fields:
// start address >> 4 (bits 0-13), leading-dimension offset (16-29; not used
// by swizzled K-major tiles, 1), stride-dimension offset >> 4 (32-45: the
// 1024 bytes between atoms), the descriptor version of this architecture
// (bit 46), base offset 0 (49-51: tiles are 1024-byte aligned), swizzle mode
// 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 D (bits 4-5 = 1), bf16 A and B
// (7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 (17-22),
// M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

struct HeadArgs {
  float *part;     // [ntiles][kKSplit][Mpad][NT] fp32 partial products (the workspace)
  int32_t M;       // positions (N k)
  int32_t Mpad;    // rows per partial block: M rounded up to a cluster's row tiles
  int32_t nkb;     // 64-wide K blocks of H
  int32_t kb_per;  // K blocks per K quarter
  int32_t NT;      // columns of this launch's W1 tiles (a multiple of 16, <= 256)
};

struct HeadSmem {
  unsigned long long fullA[kStagesA], emptyA[kStagesA];
  unsigned long long fullB[kStagesB], emptyB[kStagesB];
  unsigned long long acc;  // every MMA done
  uint32_t tmem;
  int32_t err;
  int32_t consumed;  // K blocks the MMA thread consumed
  int32_t issuedA, issuedB;
};

__global__ void __launch_bounds__(kMmaThreads, 1)
    length_head_mma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, HeadArgs a) {
  extern __shared__ __align__(1024) unsigned char dyn_raw[];
  __shared__ HeadSmem sm;
  const uint32_t raw = smem_u32(dyn_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-byte aligned: the swizzle atoms' alignment
  unsigned char *ring = dyn_raw + (base - raw);
  const int NT = a.NT;
  const int stageB = NT * kBK * 2;
  const int shareB = stageB / kMGroup;  // the part of a W1 tile each CTA loads (a multiple of 1024 bytes)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // blockIdx.x = (row group * kKSplit + K quarter) * kMGroup + rank in the cluster
  const int mh = static_cast<int>(blockIdx.x % kCluster);  // which row tile of the cluster's group
  const int kr = static_cast<int>((blockIdx.x / kCluster) % kKSplit);  // K quarter
  const int mtile = static_cast<int>(blockIdx.x / (kCluster * kKSplit)) * kMGroup + mh;
  const int ntile = static_cast<int>(blockIdx.y);
  const int kb0 = kr * a.kb_per;
  const int kb1 = min(a.nkb, kb0 + a.kb_per);
  const int nkb = max(0, kb1 - kb0);
  const uint16_t group = static_cast<uint16_t>((1u << kCluster) - 1u);  // the CTAs sharing W1 tiles

  // the reducing kernel may be scheduled now; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&sm.fullA[s], 1);
      mbar_init(&sm.emptyA[s], 1);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&sm.fullB[s], 1);
      mbar_init(&sm.emptyB[s], kMGroup);  // every CTA of the group must be done with the stage
    }
    mbar_init(&sm.acc, 1);
    sm.err = 0;
    sm.consumed = 0;
    sm.issuedA = 0;
    sm.issuedB = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem), kTN);
    tmem_relinquish();
  }
  tc_fence_before();
  cg::this_cluster().sync();  // every CTA's barriers exist before a peer multicasts into it
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp == 0 && lane == 0) {
    // ---- producer of A: this CTA's X tiles (128 rows x 64 of K) ----
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % kStagesA;
      if (i >= kStagesA && !mbar_wait_bounded(&sm.emptyA[s], static_cast<uint32_t>((i / kStagesA - 1) & 1))) {
        atomicOr(&sm.err, 1);
        break;
      }
      mbar_arrive_expect_tx(&sm.fullA[s], static_cast<uint32_t>(kStageA));
      tma_load_2d(base + static_cast<uint32_t>(s * kStageA), &tmA, (kb0 + i) * kBK, mtile * kTM,
                  smem_u32(&sm.fullA[s]));
    }
    sm.issuedA = i;
  } else if (warp == 2 && lane == 0) {
    // ---- producer of B: a quarter of each W1 tile (NT / 4 rows x 64 of K),
    // multicast to the group; the stage's barrier expects the whole tile ----
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % kStagesB;
      if (i >= kStagesB && !mbar_wait_bounded(&sm.emptyB[s], static_cast<uint32_t>((i / kStagesB - 1) & 1))) {
        atomicOr(&sm.err, 1);
        break;
      }
      mbar_arrive_expect_tx(&sm.fullB[s], static_cast<uint32_t>(stageB));
      tma_load_2d_mc(base + static_cast<uint32_t>(ringB_off() + s * stageB + mh * shareB), &tmB, (kb0 + i) * kBK,
                     ntile * kTN + mh * (NT / kMGroup), smem_u32(&sm.fullB[s]), group);
    }
    sm.issuedB = i;
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: four K = 16 steps per K block into the TMEM accumulator ----
    const uint32_t idesc = idesc_bf16(kTM, NT);
    int i = 0;
    for (; i < nkb; ++i) {
      const int sa = i % kStagesA, sb = i % kStagesB;
      if (!mbar_wait_bounded(&sm.fullA[sa], static_cast<uint32_t>((i / kStagesA) & 1)) ||
          !mbar_wait_bounded(&sm.fullB[sb], static_cast<uint32_t>((i / kStagesB) & 1))) {
        atomicOr(&sm.err, 1);
        break;
      }
      tc_fence_after();
      const uint64_t da = sw128_desc(base + static_cast<uint32_t>(sa * kStageA));
      const uint64_t db = sw128_desc(base + static_cast<uint32_t>(ringB_off() + sb * stageB));
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)  // +32 bytes of K per step: +2 in the address field
        mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
      mma_commit(smem_u32(&sm.emptyA[sa]));          // free once these MMAs are done
      mma_commit_mc(smem_u32(&sm.emptyB[sb]), group);  // in every CTA of the group
    }
    sm.consumed = i;
    if (i > 0) mma_commit(smem_u32(&sm.acc));
  }
  __syncthreads();
  // copies issued but never consumed (only after a timeout) land first
  if (warp == 0 && lane == 0)
    for (int i = sm.consumed; i < sm.issuedA; ++i)
      if (!mbar_wait_bounded(&sm.fullA[i % kStagesA], static_cast<uint32_t>((i / kStagesA) & 1))) atomicOr(&sm.err, 1);
  if (warp == 2 && lane == 0)
    for (int i = sm.consumed; i < sm.issuedB; ++i)
      if (!mbar_wait_bounded(&sm.fullB[i % kStagesB], static_cast<uint32_t>((i / kStagesB) & 1))) atomicOr(&sm.err, 1);
  // the accumulator is complete (bounded wait; every thread)
  if (sm.consumed > 0 && !mbar_wait_bounded(&sm.acc, 0)) atomicOr(&sm.err, 1);
  tc_fence_after();
  __syncthreads();
  const bool ok = (sm.err == 0) && (sm.consumed == nkb);

  // ---- the partial tile: TMEM lane = row -> shared memory -> coalesced rows in
  // the workspace (block (ntile, kr), rows of NT floats) ----
  float *P = reinterpret_cast<float *>(ring);
  const int pitch = tile_pitch(NT);
  {
    const int row = warp * 32 + lane;
    float *prow = P + row * pitch;
    for (int c = 0; c < NT; c += 64) {
      float v[64];
      if (nkb > 0 && ok) {
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(c), v);
        if (c + 32 < NT) tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(c + 32), v + 32);
      } else {
        // no K block for this quarter: a zero partial; a wait that gave up: NaN
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = (nkb == 0) ? 0.f : __int_as_float(0x7fffffff);
      }
#pragma unroll
      for (int j = 0; j < 64; j += 4)
        if (c + j < NT) *reinterpret_cast<float4 *>(prow + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
  }
  __syncthreads();
  {
    float *G = a.part + ((static_cast<int64_t>(ntile) * kKSplit + kr) * a.Mpad + static_cast<int64_t>(mtile) * kTM) * NT;
    const int nv = NT / 4;  // 16-byte vectors per row
    for (int row = warp; row < kTM; row += kMmaThreads / 32) {
      if (mtile * kTM + row >= a.M) break;
      const float *prow = P + row * pitch;
      for (int v = lane; v < nv; v += 32)
        st_stream(G + static_cast<int64_t>(row) * NT + 4 * v, prow[4 * v], prow[4 * v + 1], prow[4 * v + 2],
                  prow[4 * v + 3]);
    }
  }
  tc_fence_before();
  cg::this_cluster().sync();  // every commit into a peer's barrier has landed before anyone exits
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTN);
  }
}

// Per request (one CTA): for each of its k positions the four K partials of
// every column are summed in quarter order, then bias and SiLU; the positions
// are averaged, dotted with w2 (a fixed-order block reduction), and b2,
// sigmoid, gamma, floor and clamp give a_hat and k_hat.
constexpr int kReduceThreads = 256;
__global__ void __launch_bounds__(kReduceThreads, 2) length_head_reduce(const float *part, const float *b1, const float *w2,
                                                                     float b2, int32_t k, int32_t Hp, int32_t Mpad,
                                                                     int32_t NT, float gamma, float *a_hat,
                                                                     int32_t *k_hat) {
  __shared__ float red[kReduceThreads / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials are complete
  const int32_t i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float acc = 0.f;
  for (int n = tid; n < Hp; n += kReduceThreads) {
    const int t = n / kTN, c = n % kTN;
    const float bn = __ldg(b1 + n);
    const float *blk = part + static_cast<int64_t>(t) * kKSplit * Mpad * NT + c;
    float s = 0.f;
    for (int p0 = 0; p0 < k; p0 += 8) {
      // the quarters of eight positions in flight before any arithmetic
      float y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        // offsets within the partials (M_pad NT floats per quarter) fit 32 bits
        const int m = i * k + p0 + u;
        y[u] = 0.f;
        if (p0 + u < k) {
#pragma unroll
          for (int q = 0; q < kKSplit; ++q) y[u] += __ldcg(blk + (q * Mpad + m) * NT);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p0 + u < k) {
          const float g = y[u] + bn;
          s += g / (1.f + expf(-g));  // SiLU
        }
    }
    acc = fmaf(__ldg(w2 + n), s / static_cast<float>(k), acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (tid == 0) {
    float z = b2;
    for (int w = 0; w < kReduceThreads / 32; ++w) z += red[w];
    const float av = 1.f / (1.f + expf(-z));
    float kh = floorf(gamma * av * static_cast<float>(k));
    kh = fminf(fmaxf(kh, 1.f), static_cast<float>(k));
    a_hat[i] = av;
    k_hat[i] = (av == av) ? static_cast<int32_t>(kh) : 1;
  }
}

__global__ void length_label_kernel(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                                    float *a_star, float *loss) {
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const int32_t L = __ldg(cu + i + 1) - __ldg(cu + i);
  const int32_t acc = __ldg(accept_len + i);
  if (acc < 0 || L < 1) {
    a_star[i] = __int_as_float(0x7fffffff);
    if (loss) loss[i] = __int_as_float(0x7fffffff);
    return;
  }
  const float as = static_cast<float>(acc) / static_cast<float>(L);
  a_star[i] = as;
  if (loss) {
    const float d = __ldg(a_hat + i) - as;
    loss[i] = d * d;
  }
}

// the driver's tensor-map encoder, looked up once through the runtime
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// a 2-D bf16 tensor [rows, H] (row pitch H * 2 bytes) read in boxes of 64 x box_rows, 128-byte swizzle
bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t H, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// the partial-product blocks' geometry: column tiles, their width, padded rows
static void head_geometry(int32_t N, int32_t k, int32_t Hp, int *ntiles, int *NT, int64_t *Mpad) {
  *ntiles = (Hp + kTN - 1) / kTN;
  // the MMA's N: a multiple of 16; of 32 here, so that each CTA's quarter of a
  // W1 tile starts on a 1024-byte swizzle atom
  *NT = (*ntiles == 1) ? (Hp + 31) / 32 * 32 : kTN;
  const int64_t rows = static_cast<int64_t>(kTM) * kMGroup;
  *Mpad = (static_cast<int64_t>(N) * k + rows - 1) / rows * rows;
}

size_t length_head_gemm_bytes(int32_t N, int32_t k, int32_t Hp) {
  int ntiles = 0, NT = 0;
  int64_t Mpad = 0;
  head_geometry(N, k, Hp, &ntiles, &NT, &Mpad);
  return (static_cast<size_t>(ntiles) * kKSplit * Mpad * NT * sizeof(float) + 255) / 256 * 256;
}

int launch_length_head(const void *hidden, const void *w1, const float *b1, const float *w2, float b2, int32_t N,
                       int32_t k, int32_t H, int32_t Hp, float gamma, float *a_hat, int32_t *k_hat,
                       void *workspace, size_t workspace_bytes, cudaStream_t st) {
  if (workspace_bytes < length_head_gemm_bytes(N, k, Hp)) return 4;
  int ntiles = 0, NT = 0;
  int64_t Mpad = 0;
  head_geometry(N, k, Hp, &ntiles, &NT, &Mpad);
  const int64_t M = static_cast<int64_t>(N) * k;
  CUtensorMap mA, mB;
  if (!make_map(&mA, hidden, M, H, kTM) || !make_map(&mB, w1, Hp, H, NT / kMGroup)) return 2;
  HeadArgs a;
  a.part = static_cast<float *>(workspace);
  a.M = static_cast<int32_t>(M);
  a.Mpad = static_cast<int32_t>(Mpad);
  a.nkb = (H + kBK - 1) / kBK;
  a.kb_per = (a.nkb + kKSplit - 1) / kKSplit;
  a.NT = NT;
  const size_t smem = static_cast<size_t>(head_smem(NT));
  // the largest launch's shared memory, once per device
  static std::mutex mu;
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(length_head_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, head_smem(kTN)) !=
          cudaSuccess)
        return 1;
      attr_done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(Mpad / (kTM * kMGroup) * kKSplit * kCluster), static_cast<unsigned>(ntiles), 1);
  cfg.blockDim = dim3(kMmaThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *tm = timer_before("length_head_mma", st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, length_head_mma, mA, mB, a);
  timer_after(tm, st);
  if (e != cudaSuccess) return 1;
  // the per-request reduction: a programmatic dependent of the projection
  cudaLaunchConfig_t f = {};
  cudaLaunchAttribute fa[1];
  fa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  fa[0].val.programmaticStreamSerializationAllowed = 1;
  f.gridDim = dim3(static_cast<unsigned>(N), 1, 1);
  f.blockDim = dim3(kReduceThreads, 1, 1);
  f.stream = st;
  f.attrs = fa;
  f.numAttrs = 1;
  tm = timer_before("length_head_reduce", st);
  e = cudaLaunchKernelEx(&f, length_head_reduce, static_cast<const float *>(a.part), b1, w2, b2, k, Hp, a.Mpad, NT,
                         gamma, a_hat, k_hat);
  timer_after(tm, st);
  if (e != cudaSuccess) return 1;
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_length_label(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                        float *a_star, float *loss, cudaStream_t st) {
  length_label_kernel<<<(N + 255) / 256, 256, 0, st>>>(accept_len, cu, a_hat, N, a_star, loss);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace svw
