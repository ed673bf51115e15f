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
// CTAs share the work at the benchmark's shape; the four K quarters of a row
// tile form a thread-block cluster.  X tiles come from DRAM (the ones beyond
// the ring's first round requested into L2 once that round is on its way)
// through a five-stage ring, W1 tiles (2 MB in all, read by every row tile: L2 hits) through a
// four-stage ring, each fed by its own producer thread; one thread issues the
// MMAs.  The K quarters are then summed inside the cluster: CTA q
// of the cluster takes rows [32 q, 32 q + 32) of the tile, and every CTA
// sends each 32-row block of its fp32 partial tile from tensor memory into
// the owning CTA's shared memory (distributed shared memory, one slot per
// quarter).  The owner adds the four quarters in quarter order and finishes
// each of its rows: bias, SiLU and the dot with w2 over the tile's columns,
// one float per position and column tile.  Since the mean over positions and
// the dot with w2 commute, a request only needs the sum of its positions'
// dots: when its k positions lie in one 32-row block (k divides 32, H' <= 256)
// the owning CTA adds them and applies b2, sigmoid, gamma, floor and clamp;
// otherwise a small programmatic-dependent kernel does, from the dots in the
// workspace (the same order, the same arithmetic).  No partial product
// leaves the chip.
//
// Every mbarrier wait is bounded by a clock deadline; a CTA that gives up
// stops issuing work, lets the copies it started land (again bounded), sends
// NaN for its rows, still joins every cluster barrier and frees its tensor
// memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace svw {

namespace {

constexpr int kTM = 128;          // rows of X per CTA (the MMA's M)
constexpr int kTN = 256;          // columns of W1 rows per CTA (the MMA's N at most)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int kStagesA = 5;       // X tiles (16 KB; requested into L2 ahead)
constexpr int kStagesB = 4;       // W1 tiles (32 KB; L2 hits): bytes in flight in proportion
constexpr int kKSplit = 4;        // K quarters: the CTAs of a cluster
constexpr int kMmaThreads = 256;  // eight warps; warp w reads TMEM lanes [32 (w % 4), 32 (w % 4) + 32)
constexpr int kWarps = kMmaThreads / 32;
constexpr int kStageA = kTM * kBK * 2;  // 16 KB
constexpr int kBlock = kTM / kKSplit;   // rows each CTA of the cluster finishes (32)

// Dynamic shared memory: the two rings, reused after the main loop for the
// four K quarters of this CTA's 32-row block (slot q from quarter q, float4
// entry (c / 4) * 32 + row holding columns c .. c + 3 of that row).
__host__ __device__ constexpr int ringB_off() { return kStagesA * kStageA; }
__host__ __device__ constexpr int ring_bytes(int NT) { return kStagesA * kStageA + kStagesB * NT * kBK * 2; }
__host__ __device__ constexpr int slot_bytes(int NT) { return kBlock * NT * 4; }
__host__ __device__ constexpr int head_smem(int NT) {
  return (ring_bytes(NT) > kKSplit * slot_bytes(NT) ? ring_bytes(NT) : kKSplit * slot_bytes(NT)) + 1024;
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

// the box at (x, y) fetched into L2 ahead of its load (no completion to wait for)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// 16 bytes into the shared memory of a CTA of this cluster (address from mapa)
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// start loading 32 consecutive fp32 columns of this thread's TMEM lane; the
// registers hold them after tmem_wait_ld()
__device__ __forceinline__ void tmem_ld32_start(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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
  float *s;         // [ntiles][M] per position and column tile: sum_c w2[c] SiLU(y[c] + b1[c])
  float *a_hat;     // [N] out, when fuse
  int32_t *k_hat;   // [N] out, when fuse
  int32_t N, k;     // requests, positions per request
  float b2, gamma;
  int32_t fuse;     // 1: each CTA finishes its block's requests (k divides 32, one column tile)
  const float *b1;  // [Hp]
  const float *w2;  // [Hp]
  int32_t M;        // positions (N k)
  int32_t Hp;       // columns of W1 (H')
  int32_t nkb;      // 64-wide K blocks of H
  int32_t kb_per;   // K blocks per K quarter
  int32_t NT;       // columns of this launch's W1 tiles (a multiple of 32, <= 256)
};

struct HeadSmem {
  unsigned long long fullA[kStagesA], emptyA[kStagesA];
  unsigned long long fullB[kStagesB], emptyB[kStagesB];
  unsigned long long acc;  // every MMA done
  uint32_t tmem;
  int32_t err;
  int32_t consumed;  // K blocks the MMA thread consumed
  int32_t issuedA, issuedB;
  float red[kWarps][32];            // the row dots of the eight column groups
  float dot[kBlock];                // the block's position dots (fuse)
  float b1[kTN], w2[kTN];           // this column tile's bias and output weights
};

// a_hat and k_hat of request i from the sum z of its position dots
__device__ __forceinline__ void head_finish(float z, int32_t k, float b2, float gamma, float *a_hat, int32_t *k_hat,
                                            int32_t i) {
  z = b2 + z / static_cast<float>(k);
  const float av = 1.f / (1.f + expf(-z));
  float kh = floorf(gamma * av * static_cast<float>(k));
  kh = fminf(fmaxf(kh, 1.f), static_cast<float>(k));
  a_hat[i] = av;
  k_hat[i] = (av == av) ? static_cast<int32_t>(kh) : 1;
}

__global__ void __launch_bounds__(kMmaThreads, 1)
    length_head_mma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, HeadArgs a) {
  extern __shared__ __align__(1024) unsigned char dyn_raw[];
  __shared__ HeadSmem sm;
  const uint32_t raw = smem_u32(dyn_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-byte aligned: the swizzle atoms' alignment
  unsigned char *ring = dyn_raw + (base - raw);
  const int NT = a.NT;
  const int stageB = NT * kBK * 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // blockIdx.x = row tile * kKSplit + K quarter (the rank in the cluster)
  const int kr = static_cast<int>(blockIdx.x % kKSplit);
  const int mtile = static_cast<int>(blockIdx.x / kKSplit);
  const int ntile = static_cast<int>(blockIdx.y);
  const int kb0 = kr * a.kb_per;
  const int kb1 = min(a.nkb, kb0 + a.kb_per);
  const int nkb = max(0, kb1 - kb0);

  // the finishing kernel may be scheduled now; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&sm.fullA[s], 1);
      mbar_init(&sm.emptyA[s], 1);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&sm.fullB[s], 1);
      mbar_init(&sm.emptyB[s], 1);
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
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  // the set-up above overlaps the kernel ahead; its output (the hidden
  // states, an updated W1) is read only from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int c = tid; c < NT; c += kMmaThreads) {
    const int col = ntile * kTN + c;
    sm.b1[c] = (col < a.Hp) ? __ldg(a.b1 + col) : 0.f;
    sm.w2[c] = (col < a.Hp) ? __ldg(a.w2 + col) : 0.f;  // padding columns contribute nothing
  }

  if (warp == 0 && lane == 0) {
    // ---- producer of A: this CTA's X tiles (128 rows x 64 of K) through
    // the ring; once the ring's first round is on its way, the rest are
    // requested into L2 (DRAM sees the whole projection's reads together) ----
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % kStagesA;
      if (i == kStagesA)
        for (int j = kStagesA; j < nkb; ++j) tma_prefetch_2d(&tmA, (kb0 + j) * kBK, mtile * kTM);
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
    // ---- producer of B: this CTA's W1 tiles (NT rows x 64 of K), the ones
    // beyond the ring's first round requested into L2 as for A ----
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % kStagesB;
      if (i == kStagesB)
        for (int j = kStagesB; j < nkb; ++j) tma_prefetch_2d(&tmB, (kb0 + j) * kBK, ntile * kTN);
      if (i >= kStagesB && !mbar_wait_bounded(&sm.emptyB[s], static_cast<uint32_t>((i / kStagesB - 1) & 1))) {
        atomicOr(&sm.err, 1);
        break;
      }
      mbar_arrive_expect_tx(&sm.fullB[s], static_cast<uint32_t>(stageB));
      tma_load_2d(base + static_cast<uint32_t>(ringB_off() + s * stageB), &tmB, (kb0 + i) * kBK, ntile * kTN,
                  smem_u32(&sm.fullB[s]));
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
      mma_commit(smem_u32(&sm.emptyA[sa]));  // free once these MMAs are done
      mma_commit(smem_u32(&sm.emptyB[sb]));
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

  // ---- the K quarters summed inside the cluster ----
  // every CTA of the cluster is past its main loop: its rings may be written
  cluster_barrier();
  {
    // warp w holds tile rows [32 q, 32 q + 32), q = w % 4 (its TMEM lanes),
    // and sends them to CTA q, slot kr: the 32-column chunks of parity w / 4
    const int q = warp & 3;
    const uint32_t slot = base + static_cast<uint32_t>(kr * slot_bytes(NT));
    const uint32_t dst = (q == kr) ? slot : mapa_shared(slot, static_cast<uint32_t>(q));
    const bool have = (nkb > 0 && ok);
    // no K block for this quarter: a zero partial; a wait that gave up: NaN
    const uint32_t fill = (nkb == 0) ? 0u : 0x7fffffffu;
    // two chunks per round: both TMEM loads in flight, then 16 stores of 16 bytes
    for (int c = (warp >> 2) * 32; c < NT; c += 128) {
      const bool two = (c + 64 < NT);
      uint32_t v[64];
      if (have) {
        const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c);
        tmem_ld32_start(ta, v);
        if (two) tmem_ld32_start(ta + 64, v + 32);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = fill;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int cc = c + ((j < 8) ? 4 * j : 64 + 4 * (j - 8));  // first column of the 16-byte piece
        if (j < 8 || two) {
          const uint32_t off = static_cast<uint32_t>(((cc >> 2) * 32 + lane) * 16);
          st_cluster_v4(dst + off, __uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
    }
  }
  tc_fence_before();
  cluster_barrier();  // every quarter of this CTA's rows has landed
  {
    // thread (g, r): row r of the block, columns [g NT / 8, (g + 1) NT / 8)
    const int r = lane, g = warp;
    const float4 *S = reinterpret_cast<const float4 *>(ring);
    const int sl = slot_bytes(NT) / 16;  // float4 entries per slot
    const int q0 = g * (NT / 32), q1 = q0 + NT / 32;
    float acc = 0.f;
#pragma unroll 4
    for (int c4 = q0; c4 < q1; ++c4) {
      const int e = c4 * 32 + r;
      float4 y = S[e];
#pragma unroll
      for (int q = 1; q < kKSplit; ++q) {  // quarter order
        const float4 t = S[q * sl + e];
        y.x += t.x;
        y.y += t.y;
        y.z += t.z;
        y.w += t.w;
      }
      const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = yv[j] + sm.b1[c4 * 4 + j];
        acc = fmaf(sm.w2[c4 * 4 + j], __fdividef(x, 1.f + __expf(-x)), acc);  // w2 SiLU
      }
    }
    sm.red[g][r] = acc;
    __syncthreads();
    if (g == 0) {
      const int64_t m0 = static_cast<int64_t>(mtile) * kTM + kr * kBlock;  // the block's first position
      float d = sm.red[0][r];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) d += sm.red[w][r];  // column-group order
      if (!a.fuse) {
        if (m0 + r < a.M) a.s[static_cast<int64_t>(ntile) * a.M + m0 + r] = d;
      } else {
        sm.dot[r] = d;
        __syncwarp();
        // lane j finishes the block's j-th request (positions in order)
        const int64_t i = m0 / a.k + r;
        if (r < kBlock / a.k && i < a.N) {
          float z = 0.f;
          for (int p = 0; p < a.k; ++p) z += sm.dot[r * a.k + p];
          head_finish(z, a.k, a.b2, a.gamma, a.a_hat, a.k_hat, static_cast<int32_t>(i));
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTN);
  }
}

// Per request: the positions' dots summed over column tiles and positions
// (fixed order), then the mean, b2, sigmoid, gamma, floor and clamp give
// a_hat and k_hat.
__global__ void length_head_final(const float *s, int32_t ntiles, int32_t M, int32_t N, int32_t k, float b2,
                                  float gamma, float *a_hat, int32_t *k_hat) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the dots are complete
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  float z = 0.f;
  for (int t = 0; t < ntiles; ++t) {
    const float *st = s + static_cast<int64_t>(t) * M + static_cast<int64_t>(i) * k;
#pragma unroll 8
    for (int p = 0; p < k; ++p) z += __ldcg(st + p);
  }
  head_finish(z, k, b2, gamma, a_hat, k_hat, i);
}

__global__ void length_label_kernel(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                                    float *a_star, float *loss) {
  // the length head's projection may set up now (it waits for this grid
  // before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the accepted lengths are complete
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

// column tiles of W1 and their width (the MMA's N: a multiple of 16; of 32
// here, so that the tile's 32-column TMEM loads stay whole)
static void head_geometry(int32_t Hp, int *ntiles, int *NT) {
  *ntiles = (Hp + kTN - 1) / kTN;
  *NT = (*ntiles == 1) ? (Hp + 31) / 32 * 32 : kTN;
}

size_t length_head_gemm_bytes(int32_t N, int32_t k, int32_t Hp) {
  int ntiles = 0, NT = 0;
  head_geometry(Hp, &ntiles, &NT);
  return (static_cast<size_t>(ntiles) * N * k * sizeof(float) + 255) / 256 * 256;
}

int launch_length_head(const void *hidden, const void *w1, const float *b1, const float *w2, float b2, int32_t N,
                       int32_t k, int32_t H, int32_t Hp, float gamma, float *a_hat, int32_t *k_hat,
                       void *workspace, size_t workspace_bytes, cudaStream_t st) {
  if (workspace_bytes < length_head_gemm_bytes(N, k, Hp)) return 4;
  int ntiles = 0, NT = 0;
  head_geometry(Hp, &ntiles, &NT);
  const int64_t M = static_cast<int64_t>(N) * k;
  CUtensorMap mA, mB;
  if (!make_map(&mA, hidden, M, H, kTM) || !make_map(&mB, w1, Hp, H, NT)) return 2;
  HeadArgs a;
  a.s = static_cast<float *>(workspace);
  a.b1 = b1;
  a.w2 = w2;
  a.M = static_cast<int32_t>(M);
  a.Hp = Hp;
  a.nkb = (H + kBK - 1) / kBK;
  a.kb_per = (a.nkb + kKSplit - 1) / kKSplit;
  a.NT = NT;
  a.a_hat = a_hat;
  a.k_hat = k_hat;
  a.N = N;
  a.k = k;
  a.b2 = b2;
  a.gamma = gamma;
  a.fuse = (ntiles == 1 && kBlock % k == 0) ? 1 : 0;
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
  // the projection: clusters of the four K quarters of a row tile, a
  // programmatic dependent of the kernel ahead (its set-up overlaps that
  // kernel's tail)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kKSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>((M + kTM - 1) / kTM * kKSplit), static_cast<unsigned>(ntiles), 1);
  cfg.blockDim = dim3(kMmaThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void *tm = timer_before("length_head_mma", st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, length_head_mma, mA, mB, a);
  timer_after(tm, st);
  if (e != cudaSuccess) return 1;
  if (a.fuse) return cudaGetLastError() == cudaSuccess ? 0 : 1;
  // the per-request finish: a programmatic dependent of the projection
  cudaLaunchConfig_t f = {};
  cudaLaunchAttribute fa[1];
  fa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  fa[0].val.programmaticStreamSerializationAllowed = 1;
  f.gridDim = dim3(static_cast<unsigned>((N + 127) / 128), 1, 1);
  f.blockDim = dim3(128, 1, 1);
  f.stream = st;
  f.attrs = fa;
  f.numAttrs = 1;
  tm = timer_before("length_head_final", st);
  e = cudaLaunchKernelEx(&f, length_head_final, static_cast<const float *>(a.s), static_cast<int32_t>(ntiles),
                         a.M, N, k, b2, gamma, a_hat, k_hat);
  timer_after(tm, st);
  if (e != cudaSuccess) return 1;
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_length_label(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                        float *a_star, float *loss, cudaStream_t st) {
  // a programmatic dependent of the kernel ahead (it waits for it first), so
  // that its launch overlaps that kernel's tail
  cudaLaunchConfig_t f = {};
  cudaLaunchAttribute fa[1];
  fa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  fa[0].val.programmaticStreamSerializationAllowed = 1;
  f.gridDim = dim3(static_cast<unsigned>((N + 255) / 256), 1, 1);
  f.blockDim = dim3(256, 1, 1);
  f.stream = st;
  f.attrs = fa;
  f.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&f, length_label_kernel, accept_len, cu, a_hat, N, a_star, loss);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? 0 : 1;
}

}  // namespace svw
