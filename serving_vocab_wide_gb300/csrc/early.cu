// early.cu -- early-exit verification by thread-block clusters (sm_103a).
//
// Method ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.2, Algorithm 1;
// "AdaFlash：基于在策略蒸馏扩散草稿器的自适应投机解码" §3.3, Figure 2(c)):
// leftmost rejection makes every row after a request's first rejected
// position irrelevant to its result, and acceptance falls along the block,
// so a verifier that walks each request's positions in order and stops at
// the first rejection reads a fraction of the logits and returns the same
// accepted lengths and tokens.
//
// GPU design.  A cluster of CL CTAs (CL <= 16) takes one request at a time
// from a queue ordered longest first (the plan kernel's records) and walks
// its positions in order.  CTA r owns vocabulary slice [r SL, (r+1) SL): per
// position it bulk-copies its slice of the target row (and of the draft row)
// into shared memory (cp.async.bulk, mbarrier completion), reduces it to
// (max, sum 2^((x - max) log2e/T)) per row -- (max, first argmax) when greedy
// -- and pushes that partial into every peer's inbox (st.async completing the
// peer's mbarrier).  Every CTA merges the CL partials in the same fixed order,
// so all of them reach the same accept decision and go on, or stop, together
// with no further communication.  The next request's slot is drawn by rank 0
// (one atomic) and sent to the peers the same way.  Per request the kernel
// records the stop position and the row statistics there; the finalize
// kernel validates the request, writes accept_len and draws the next token.
// Every wait is bounded: on expiry a CTA records SVW_DEV_TIMEOUT, issues no
// more copies and keeps taking part in the exchanges (marked aborted), so no
// peer can hang.
#include <cfloat>
#include <climits>
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <mutex>

#include "svw_device.cuh"
#include "svw_internal.h"

namespace cg = cooperative_groups;

namespace svw {

namespace {

constexpr int kENT = 256;  // threads per CTA
constexpr int kEWarps = kENT / 32;
constexpr int kEMaxCluster = 16;
constexpr int kSliceTarget = 32768;      // bytes of one row per CTA the cluster size aims at
constexpr int kSliceMax = 64 * 1024;     // largest slice of one row a CTA holds

struct EGeo {
  int32_t SL;           // slice length in elements (multiple of 8)
  int32_t slice_bytes;  // bytes reserved per row slice (multiple of 128)
};

struct ESmem {
  unsigned long long mbar;     // the slice copies of the current position
  unsigned long long xbar[2];  // partial exchange, two slots
  unsigned long long qbar[2];  // request broadcast, two slots
  float4 inbox[2][kEMaxCluster];
  float4 red[2][kEWarps];  // warp partials of two consecutive positions
  int32_t req[2];
  int32_t slot;
  int32_t dec;  // 0: go on, 1: stop here, 2: bad request
  int32_t abort;
  uint32_t abort_parity;
};

// merge of row-statistic partials held by the warp's lanes, by a fixed
// butterfly: every lane, and every CTA merging the same partials, gets the
// same bits.  T > 0: (mT, sT, mD, sD); greedy: (max, first argmax, NaN seen).
template <bool GREEDY>
__device__ __forceinline__ float4 merge_parts(float4 p, float k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float4 q = make_float4(__shfl_xor_sync(0xffffffffu, p.x, o), __shfl_xor_sync(0xffffffffu, p.y, o),
                                 __shfl_xor_sync(0xffffffffu, p.z, o), __shfl_xor_sync(0xffffffffu, p.w, o));
    if (GREEDY) {
      float v = p.x;
      int32_t i = __float_as_int(p.y);
      amax_combine(v, i, q.x, __float_as_int(q.y));
      p = make_float4(v, __int_as_float(i), (p.z != 0.f || q.z != 0.f) ? 1.f : 0.f, 0.f);
    } else {
      lse_combine(p.x, p.y, q.x, q.y, k);
      lse_combine(p.z, p.w, q.z, q.w, k);
    }
  }
  return p;
}

template <bool GREEDY>
__device__ __forceinline__ float4 empty_part() {
  return GREEDY ? make_float4(-INFINITY, __int_as_float(INT32_MAX), 0.f, 0.f)
                : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
}

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kENT) verify_early_cluster(VerifyArgs a, EGeo geo) {
  using E = Elem<DT>;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ ESmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;
  const int64_t lo = static_cast<int64_t>(rank) * geo.SL;
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(geo.SL), V - lo)));
  const int nvec = n / E::kPerVec;  // rows are 16-byte pitched on this path
  const uint32_t bytes = static_cast<uint32_t>(n) * E::kSize;
  unsigned char *tbuf = dyn;
  unsigned char *dbuf = dyn + geo.slice_bytes;
  const uint32_t tb = smem_u32(tbuf), db = smem_u32(dbuf);
  const float k = a.k;

  if (tid == 0) {
    mbar_init(&sm.mbar, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.xbar[s], 1);
      mbar_init(&sm.qbar[s], 1);
    }
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster.sync();  // every barrier exists before any peer sends
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the finalize grid may be scheduled
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the plan kernel's records and reset state
  const int32_t nvalid = __ldcg(a.nvalid);

  uint32_t it = 0;  // exchanges so far (slot and parity)
  uint32_t cp = 0;  // copy phases so far
  unsigned long long nbytes = 0;  // logit bytes this CTA copied
  for (uint32_t rq = 0;; ++rq) {
    // ---- the next request: rank 0 draws a slot and sends it to every CTA ----
    if (tid == 0) {
      const int qs = static_cast<int>(rq & 1);
      mbar_arrive_expect_tx(&sm.qbar[qs], 4);
      if (rank == 0) {
        const int32_t s = atomicAdd(a.qnext, 1);
        for (int q = 0; q < CL; ++q)
          st_async4(mapa_shared(smem_u32(&sm.req[qs]), q), static_cast<uint32_t>(s),
                    mapa_shared(smem_u32(&sm.qbar[qs]), q));
      }
      int32_t slot = INT32_MAX;
      if (mbar_wait_bounded(&sm.qbar[qs], (rq >> 1) & 1)) {
        slot = sm.req[qs];
      } else if (a.status) {
        atomicOr(a.status, SVW_DEV_TIMEOUT);
      }
      sm.slot = slot;
    }
    __syncthreads();
    const int32_t slot = sm.slot;
    if (slot >= nvalid) break;
    const int4 info = __ldcg(a.pinfo + slot);
    const int32_t i = info.x, L = info.z;
    const int64_t c_i = info.y;

    // one thread: start the copies of this CTA's slices of the rows at
    // position jj (the target row; the draft row too unless jj is the bonus)
    auto issue = [&](int32_t jj) {
      const bool pr = !GREEDY && jj < L;
      if (!sm.abort && bytes > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&sm.mbar, (pr ? 2u : 1u) * bytes);
        nbytes += (pr ? 2u : 1u) * bytes;
        bulk_g2s(tbuf, static_cast<const char *>(a.target) + ((c_i + i + jj) * V + lo) * E::kSize, bytes, &sm.mbar);
        if (pr) bulk_g2s(dbuf, static_cast<const char *>(a.draft) + ((c_i + jj) * V + lo) * E::kSize, bytes, &sm.mbar);
      } else {
        mbar_arrive(&sm.mbar);
      }
    };
    auto land = [&]() {  // every thread: wait for the copies in flight
      // after a timeout the barrier's phases are no longer tracked: no waits
      if (!sm.abort && !mbar_wait_bounded(&sm.mbar, cp & 1)) {
        if (tid == 0) {
          if (a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
          sm.abort_parity = cp & 1;
        }
        sm.abort = 1;
      }
      ++cp;
    };
    // every thread: this CTA's warp partial of the slices now in the buffers
    // (position jj), into sm.red[jj & 1]
    auto reduce_slices = [&](int32_t jj) {
      float4 P = empty_part<GREEDY>();
      if (!sm.abort) {
        if (GREEDY) {
          float best;
          int32_t idx, nan;
          warp_amax_smem<DT, kEWarps>(tb, nvec, static_cast<int32_t>(lo), warp, lane, best, idx, nan);
          P = make_float4(best, __int_as_float(idx), nan ? 1.f : 0.f, 0.f);
        } else {
          warp_lse_smem<DT, kEWarps>(tb, nvec, warp, lane, k, P.x, P.y);
          if (jj < L) warp_lse_smem<DT, kEWarps>(db, nvec, warp, lane, k, P.z, P.w);
        }
      }
      if (lane == 0) sm.red[jj & 1][warp] = P;
    };
    // warp 0: this CTA's partial of position jj (warps merged) to every CTA
    // of the cluster, in exchange slot it & 1
    auto send = [&](int32_t jj) {
      const int xs = static_cast<int>(it & 1);
      float4 Pc = merge_parts<GREEDY>(lane < kEWarps ? sm.red[jj & 1][lane] : empty_part<GREEDY>(), k);
      if (sm.abort) {
        // poison the partial so that every CTA judges the request bad alike
        if (GREEDY) Pc.z = 1.f;
        else Pc.y = Pc.w = __int_as_float(0x7fffffff);
      }
      if (lane == 0) mbar_arrive_expect_tx(&sm.xbar[xs], static_cast<uint32_t>(CL) * 16u);
      __syncwarp();
      if (lane < CL) {
        const uint4 w = make_uint4(__float_as_uint(Pc.x), __float_as_uint(Pc.y), __float_as_uint(Pc.z),
                                   __float_as_uint(Pc.w));
        st_async16(mapa_shared(smem_u32(&sm.inbox[xs][rank]), lane), w, mapa_shared(smem_u32(&sm.xbar[xs]), lane));
      }
    };

    // Two-stage pipeline: while position j's partials are being exchanged,
    // the slices of position j + 1 land and are reduced.  A request that
    // stops at j has read (and reduced) one position ahead for nothing.
    if (tid == 0) issue(0);
    land();
    reduce_slices(0);
    __syncthreads();  // position 0's warp partials are in; the buffers are free
    if (tid == 0 && 0 < L) issue(1);
    if (warp == 0) send(0);
    for (int32_t j = 0;; ++j) {
      const bool pair = !GREEDY && j < L;
      const bool ahead = j < L;
      // the token, its logits and the uniform of position j
      int32_t x = 0;
      bool xok = true;
      float yx = 0.f, zx = 0.f, u = 0.f;
      if (tid == 0 && j < L) {
        const int64_t trow = c_i + i + j, drow = c_i + j;
        x = __ldg(a.tokens + drow);
        xok = (x >= 0 && static_cast<int64_t>(x) < V);
        if (!GREEDY && xok) {
          yx = E::load(a.target, trow * V + x);
          zx = E::load(a.draft, drow * V + x);
          u = philox_uniform(a.seed, static_cast<uint32_t>(i), static_cast<uint32_t>(j), 0u);
        }
      }
      // ---- position j + 1: its slices land and are reduced ----
      if (ahead) {
        land();
        reduce_slices(j + 1);
      }
      __syncthreads();  // position j + 1's warp partials are in; the buffers are free
      // ---- position j: the exchange completes; the decision ----
      if (warp == 0) {
        const int xs = static_cast<int>(it & 1);
        bool got = mbar_wait_bounded(&sm.xbar[xs], (it >> 1) & 1);
        if (!got && lane == 0 && a.status) atomicOr(a.status, SVW_DEV_TIMEOUT);
        const float4 M = merge_parts<GREEDY>((got && lane < CL) ? sm.inbox[xs][lane] : empty_part<GREEDY>(), k);
        got = __all_sync(0xffffffffu, got);
        if (lane == 0) {
          // the same decision in every CTA: it depends only on the merged
          // partials, the token and the uniform
          int32_t bad = got ? 0 : 1;
          bool acc = true;
          float lT = 0.f, lD = 0.f;
          if (GREEDY) {
            bad |= (M.z != 0.f) ? 1 : 0;
            if (j < L) acc = xok && (x == __float_as_int(M.y));
          } else {
            lT = lg2(M.y);
            bad |= (M.y > 0.f && M.y <= FLT_MAX) ? 0 : 1;
            if (pair) {
              lD = lg2(M.w);
              bad |= (M.w > 0.f && M.w <= FLT_MAX) ? 0 : 1;
            }
            if (j < L) acc = xok && !bad && accept_token(u, yx, zx, M.x, lT, M.z, lD, k);
          }
          if (j < L && !xok) bad = 1;
          const int32_t dec = bad ? 2 : ((j == L || !acc) ? 1 : 0);
          sm.dec = dec;
          if (dec != 0 && rank == 0) {
            a.eres[i] = make_int4(j, dec == 2 ? 1 : 0, GREEDY ? __float_as_int(M.y) : 0, 0);
            a.erow[i] = make_float4(M.x, lT, M.z, lD);
          }
        }
      }
      ++it;
      __syncthreads();
      if (sm.dec != 0) break;  // no copy is in flight
      // ---- go on: position j + 2's slices in flight, position j + 1's partial out ----
      if (tid == 0 && j + 1 < L) issue(j + 2);
      if (warp == 0) send(j + 1);
    }
  }
  if (tid == 0 && a.bytes_read && nbytes) atomicAdd(a.bytes_read, nbytes);
  // after a timeout no copy is issued; let the one that timed out land if it can
  if (tid == 0 && sm.abort) mbar_wait_bounded(&sm.mbar, sm.abort_parity);
  cluster.sync();  // peers may still read or write this CTA's shared memory
}

}  // namespace

// the cluster geometry for rows of V elements of esize bytes; CL = 0 if the
// rows are too wide for this path
EarlyClusterPlan early_cluster_plan(int64_t V, int esize, bool greedy) {
  EarlyClusterPlan p{};
  const int64_t row = V * esize;
  int64_t CL = (row + kSliceTarget - 1) / kSliceTarget;
  if (CL < 1) CL = 1;
  if (CL > kEMaxCluster) CL = kEMaxCluster;
  int64_t SL = (V + CL - 1) / CL;
  SL = (SL + 7) / 8 * 8;
  const int64_t sb = (SL * esize + 127) / 128 * 128;
  if (sb > kSliceMax) return p;
  p.CL = static_cast<int>(CL);
  p.SL = static_cast<int>(SL);
  p.slice_bytes = static_cast<int>(sb);
  p.smem = static_cast<size_t>(sb) * (greedy ? 1 : 2);
  return p;
}

namespace {

template <int DT, bool GREEDY>
cudaError_t launch_cluster_t(const VerifyArgs &a, const EarlyClusterPlan &p, cudaStream_t st) {
  auto kern = verify_early_cluster<DT, GREEDY>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.smem));
  if (e != cudaSuccess) return e;
  if (p.CL > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kENT, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // as many clusters as fit at once (cached per device, kernel and shape)
  struct Entry {
    int dev;
    const void *fn;
    int CL;
    size_t smem;
    int n;
  };
  static Entry cache[32];
  static int ncache = 0;
  static std::mutex mu;  // calls from several host threads share the cache
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int maxc = 0;
  std::unique_lock<std::mutex> lk(mu);
  for (int q = 0; q < ncache; ++q)
    if (cache[q].dev == dev && cache[q].fn == reinterpret_cast<const void *>(kern) && cache[q].CL == p.CL &&
        cache[q].smem == p.smem)
      maxc = cache[q].n;
  if (maxc == 0) {
    cfg.gridDim = dim3(p.CL * 1024, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (maxc <= 0) return cudaErrorInvalidConfiguration;
    if (ncache < 32) cache[ncache++] = Entry{dev, reinterpret_cast<const void *>(kern), p.CL, p.smem, maxc};
  }
  lk.unlock();
  int64_t nclusters = maxc;
  if (nclusters > a.N) nclusters = a.N;
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * p.CL), 1, 1);
  EGeo geo;
  geo.SL = p.SL;
  geo.slice_bytes = p.slice_bytes;
  void *tm = timer_before("verify_early_cluster", st);
  e = cudaLaunchKernelEx(&cfg, kern, a, geo);
  timer_after(tm, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_early_cluster(const VerifyArgs &a, int dtype, bool greedy, const EarlyClusterPlan &p,
                                 cudaStream_t st) {
  if (dtype == SVW_BF16) return greedy ? launch_cluster_t<1, true>(a, p, st) : launch_cluster_t<1, false>(a, p, st);
  return greedy ? launch_cluster_t<0, true>(a, p, st) : launch_cluster_t<0, false>(a, p, st);
}

}  // namespace svw
