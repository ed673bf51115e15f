// api.cu -- the exported C ABI (see include/svw.h): host-side validation,
// workspace carving, and dispatch to the kernel launchers.  No allocation,
// no host synchronisation, no device-memory reads from the host.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda_runtime.h>

#include "svw_internal.h"

namespace svw {
bool opd_supported(int64_t V, int esize);
}

namespace {

constexpr int64_t kMaxV = 1 << 20;  // sampler span cap (256 threads x 512 groups x 8)
constexpr int64_t kMaxHeadPositions = 1 << 20;  // length head: N k (32-bit offsets into its partials)

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int esize_of(svw_dtype d) { return d == SVW_BF16 ? 2 : 4; }

}  // namespace

// one-shot kernel timer, per host thread (svw_time_next_launch)
namespace {
struct ArmedTimer {
  char kernel[64];
  cudaEvent_t begin;
  cudaEvent_t end;
  bool armed;
};
thread_local ArmedTimer g_timer = {};
}  // namespace

namespace svw {
void *timer_before(const char *kernel, cudaStream_t st) {
  if (!g_timer.armed || std::strncmp(kernel, g_timer.kernel, sizeof(g_timer.kernel)) != 0) return nullptr;
  g_timer.armed = false;
  if (cudaEventRecord(g_timer.begin, st) != cudaSuccess) return nullptr;
  return reinterpret_cast<void *>(g_timer.end);
}
void timer_after(void *end_event, cudaStream_t st) {
  if (end_event) cudaEventRecord(reinterpret_cast<cudaEvent_t>(end_event), st);
}

// test hooks: the wait deadline of every translation unit, and an injected fault
namespace {
constexpr int kMaxWaitSetters = 32;
std::mutex g_wait_mu;
cudaError_t (*g_wait_set[kMaxWaitSetters])(long long);
int g_nwait = 0;
std::atomic<int32_t> g_fault{0};
}  // namespace
cudaError_t register_wait_limit(cudaError_t (*set)(long long)) {
  std::lock_guard<std::mutex> lk(g_wait_mu);
  if (g_nwait < kMaxWaitSetters) g_wait_set[g_nwait++] = set;
  return cudaSuccess;
}
int32_t test_fault() { return g_fault.load(std::memory_order_relaxed); }
}  // namespace svw

// a new tag for every OPD call (never 0): flags set by an earlier call never
// match it
static int32_t next_epoch() {
  static std::atomic<uint32_t> g_epoch{0x3c5a0000u};
  uint32_t ep = ++g_epoch;
  if (ep == 0) ep = ++g_epoch;
  return static_cast<int32_t>(ep);
}

extern "C" {

int32_t svw_version(void) { return 100; }

svw_status svw_set_wait_limit(int64_t cycles) {
  if (cycles <= 0) return SVW_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(svw::g_wait_mu);
  for (int q = 0; q < svw::g_nwait; ++q)
    if (svw::g_wait_set[q](static_cast<long long>(cycles)) != cudaSuccess) return SVW_ERR_CUDA;
  return SVW_OK;
}

svw_status svw_set_fault(int32_t kind) {
  if (kind < 0 || kind > 1) return SVW_ERR_INVALID_ARG;
  svw::g_fault.store(kind, std::memory_order_relaxed);
  return SVW_OK;
}

const char *svw_status_string(svw_status s) {
  switch (s) {
    case SVW_OK: return "SVW_OK";
    case SVW_ERR_INVALID_ARG: return "SVW_ERR_INVALID_ARG: invalid argument";
    case SVW_ERR_UNSUPPORTED: return "SVW_ERR_UNSUPPORTED: dtype or size not supported";
    case SVW_ERR_MISALIGNED: return "SVW_ERR_MISALIGNED: pointer alignment";
    case SVW_ERR_WORKSPACE: return "SVW_ERR_WORKSPACE: workspace missing or too small";
    case SVW_ERR_CUDA: return "SVW_ERR_CUDA: CUDA runtime or launch failure";
    case SVW_ERR_BAD_INPUT: return "SVW_ERR_BAD_INPUT: the device found an invalid or non-finite request / row";
    case SVW_ERR_TIMEOUT: return "SVW_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
  }
  return "unknown svw_status";
}

svw_status svw_device_status(int32_t status_word) {
  if (status_word & SVW_DEV_TIMEOUT) return SVW_ERR_TIMEOUT;
  if (status_word & SVW_DEV_BAD_INPUT) return SVW_ERR_BAD_INPUT;
  return SVW_OK;
}

size_t svw_verify_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                 svw_dtype dtype) {
  if (n_requests <= 0 || total_draft_rows < 0 || V <= 0 || V > kMaxV) return 0;
  if (dtype != SVW_F32 && dtype != SVW_BF16) return 0;
  return svw::verify_layout(n_requests, total_draft_rows, V, esize_of(dtype)).total;
}

}  // extern "C"

// spec_verify and spec_verify_early: same validation, same results.  With
// check_only, every check that does not involve the workspace runs and the
// call returns SVW_OK without launching (spec_verify_noalloc's first step).
static svw_status verify_entry(bool early, const void *target_logits, const void *draft_logits, svw_dtype dtype,
                               int32_t V, int32_t N, const int32_t *cu_draft, int64_t total_draft_rows,
                               int32_t max_len, const int32_t *draft_tokens, float temperature, uint64_t seed,
                               int32_t *accept_len, int32_t *next_token, int32_t *status,
                               unsigned long long *bytes_read, void *workspace, size_t workspace_bytes,
                               void *stream, bool check_only = false) {
  if (dtype != SVW_F32 && dtype != SVW_BF16) return SVW_ERR_UNSUPPORTED;
  if (V <= 0 || N <= 0 || total_draft_rows < 0 || max_len < 1) return SVW_ERR_INVALID_ARG;
  if (max_len > SVW_MAX_LEN || V > kMaxV) return SVW_ERR_UNSUPPORTED;
  const bool have_ws = check_only || workspace;
  if (!target_logits || !draft_logits || !cu_draft || !draft_tokens || !accept_len || !next_token || !have_ws)
    return have_ws ? SVW_ERR_INVALID_ARG : SVW_ERR_WORKSPACE;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SVW_ERR_INVALID_ARG;
  const double kd = (temperature > 0.f) ? 1.4426950408889634 / static_cast<double>(temperature) : 0.0;
  if (temperature > 0.f && !(kd < 3.0e38)) return SVW_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(cu_draft, 4) ||
      !aligned(draft_tokens, 4) || !aligned(accept_len, 4) || !aligned(next_token, 4) ||
      (status && !aligned(status, 4)) || (bytes_read && !aligned(bytes_read, 8)) ||
      (!check_only && !aligned(workspace, 256)))
    return SVW_ERR_MISALIGNED;
  if (early && total_draft_rows + N >= (int64_t{1} << 31)) return SVW_ERR_UNSUPPORTED;  // int32 row records
  if (check_only) return SVW_OK;
  const svw::VerifyLayout lay = svw::verify_layout(N, total_draft_rows, V, es);
  const svw::EarlyLayout elay = svw::early_layout(N, total_draft_rows, V, es);
  if (workspace_bytes < (early ? elay.total : lay.total)) return SVW_ERR_WORKSPACE;

  const svw::ChunkPlan plan = svw::plan_chunks(V, es);
  const bool greedy = (temperature == 0.f);
  const bool vec = ((static_cast<int64_t>(V) * es) % 16 == 0) && aligned(target_logits, 16) &&
                   aligned(draft_logits, 16);
  svw::VerifyArgs a{};
  a.fault = svw::test_fault();
  a.target = target_logits;
  a.draft = draft_logits;
  a.V = V;
  a.N = N;
  a.cu = cu_draft;
  a.total_rows = total_draft_rows;
  a.rows_t = total_draft_rows + N;
  a.max_len = max_len;
  a.tokens = draft_tokens;
  a.k = static_cast<float>(kd);
  a.seed = seed;
  a.accept_len = accept_len;
  a.next_token = next_token;
  a.status = status;
  char *ws = static_cast<char *>(workspace);
  a.part = reinterpret_cast<svw::Partial *>(ws + lay.part_off);
  a.csr_bad = reinterpret_cast<int32_t *>(ws + lay.csr_bad_off);
  a.stats_grid = 0;  // set by the launcher
  a.C = plan.C;
  a.chunk_len = plan.chunk_len;
  const int64_t rows = greedy ? (total_draft_rows + N) : (2 * total_draft_rows + N);
  a.total_items = rows * plan.C;
  cudaError_t e;
  if (early) {
    a.cnt = reinterpret_cast<int32_t *>(ws + elay.cnt_off);
    a.rej = reinterpret_cast<int32_t *>(ws + elay.rej_off);
    a.badpos = reinterpret_cast<int32_t *>(ws + elay.badpos_off);
    a.stop = reinterpret_cast<int32_t *>(ws + elay.stop_off);
    a.pinfo = reinterpret_cast<int4 *>(ws + elay.pinfo_off);
    a.W = reinterpret_cast<int64_t *>(ws + elay.wave_off);
    a.waveA = reinterpret_cast<int32_t *>(ws + elay.wave_off + (SVW_MAX_LEN + 2) * sizeof(int64_t));
    a.nvalid = a.waveA + (SVW_MAX_LEN + 1);
    a.qnext = a.nvalid + 1;
    a.eres = reinterpret_cast<int4 *>(ws + elay.eres_off);
    a.erow = reinterpret_cast<float4 *>(ws + elay.erow_off);
    a.bytes_read = bytes_read;
    e = svw::launch_verify_early(a, dtype, vec, greedy, static_cast<cudaStream_t>(stream));
  } else {
    e = svw::launch_verify(a, dtype, vec, greedy, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? SVW_OK : SVW_ERR_CUDA;
}

namespace svw {
svw_status verify_check_args(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                             int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                             const int32_t *draft_tokens, float temperature, int32_t *accept_len,
                             int32_t *next_token, int32_t *status) {
  return verify_entry(false, target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len,
                      draft_tokens, temperature, 0, accept_len, next_token, status, nullptr, nullptr, 0, nullptr,
                      true);
}
}  // namespace svw

extern "C" {

svw_status spec_verify(const void *target_logits, const void *draft_logits, svw_dtype dtype,
                       int32_t V, int32_t N, const int32_t *cu_draft, int64_t total_draft_rows,
                       int32_t max_len, const int32_t *draft_tokens, float temperature,
                       uint64_t seed, int32_t *accept_len, int32_t *next_token, int32_t *status,
                       void *workspace, size_t workspace_bytes, void *stream) {
  return verify_entry(false, target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len,
                      draft_tokens, temperature, seed, accept_len, next_token, status, nullptr, workspace,
                      workspace_bytes, stream);
}

size_t svw_verify_early_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                       svw_dtype dtype) {
  if (n_requests <= 0 || total_draft_rows < 0 || V <= 0 || V > kMaxV) return 0;
  if (dtype != SVW_F32 && dtype != SVW_BF16) return 0;
  return svw::early_layout(n_requests, total_draft_rows, V, esize_of(dtype)).total;
}

static_assert(svw::kFilterMaxK == SVW_FILTER_MAX_K, "one top-k limit");

static size_t filtered_lists_bytes(int32_t N, int64_t R) {
  const size_t rows = static_cast<size_t>(2 * R + N);
  return (rows * 4 + 255) / 256 * 256 + 2 * ((rows * svw::kFilterMaxK * 4 + 255) / 256 * 256);
}

size_t svw_verify_filtered_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                          svw_dtype dtype) {
  const size_t v = svw_verify_workspace_size(n_requests, total_draft_rows, V, dtype);
  if (v == 0) return 0;
  const size_t f = filtered_lists_bytes(n_requests, total_draft_rows);
  return v > f ? v : f;
}

svw_status spec_verify_filtered(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                                int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                                const int32_t *draft_tokens, float temperature, int32_t top_k, float top_p,
                                uint64_t seed, int32_t *accept_len, int32_t *next_token, int32_t *status,
                                void *workspace, size_t workspace_bytes, void *stream) {
  if (dtype != SVW_F32 && dtype != SVW_BF16) return SVW_ERR_UNSUPPORTED;
  if (V <= 0 || N <= 0 || total_draft_rows < 0 || max_len < 1) return SVW_ERR_INVALID_ARG;
  if (max_len > SVW_MAX_LEN || V > kMaxV) return SVW_ERR_UNSUPPORTED;
  if (!(top_p > 0.f && top_p <= 1.f)) return SVW_ERR_INVALID_ARG;
  if (top_k < 1) return SVW_ERR_INVALID_ARG;
  if (top_k > SVW_FILTER_MAX_K) return SVW_ERR_UNSUPPORTED;
  if (!target_logits || !draft_logits || !cu_draft || !draft_tokens || !accept_len || !next_token ||
      !workspace)
    return workspace ? SVW_ERR_INVALID_ARG : SVW_ERR_WORKSPACE;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SVW_ERR_INVALID_ARG;
  if (temperature == 0.f)
    // filtering keeps the argmax: greedy verification is unchanged
    return spec_verify(target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len, draft_tokens,
                       0.f, seed, accept_len, next_token, status, workspace, workspace_bytes, stream);
  const double kd = 1.4426950408889634 / static_cast<double>(temperature);
  if (!(kd < 3.0e38)) return SVW_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(cu_draft, 4) ||
      !aligned(draft_tokens, 4) || !aligned(accept_len, 4) || !aligned(next_token, 4) ||
      (status && !aligned(status, 4)) || !aligned(workspace, 256))
    return SVW_ERR_MISALIGNED;
  if (workspace_bytes < svw_verify_filtered_workspace_size(N, total_draft_rows, V, dtype)) return SVW_ERR_WORKSPACE;
  if (svw::filter_smem_bytes(V, es, top_k) > 200 * 1024) return SVW_ERR_UNSUPPORTED;
  const size_t rows = static_cast<size_t>(2 * total_draft_rows + N);
  char *ws = static_cast<char *>(workspace);
  svw::FilterArgs a{};
  a.target = target_logits;
  a.draft = draft_logits;
  a.V = V;
  a.N = N;
  a.cu = cu_draft;
  a.R = total_draft_rows;
  a.rows_t = total_draft_rows + N;
  a.max_len = max_len;
  a.tokens = draft_tokens;
  a.k = static_cast<float>(kd);
  a.top_k = top_k;
  a.top_p = top_p;
  a.cand = svw::filter_candidates(top_k);
  a.gs = svw::filter_group(top_k);
  a.seed = seed;
  a.accept_len = accept_len;
  a.next_token = next_token;
  a.status = status;
  a.cnt = reinterpret_cast<int32_t *>(ws);
  const size_t off1 = (rows * 4 + 255) / 256 * 256;
  a.lidx = reinterpret_cast<int32_t *>(ws + off1);
  a.lp = reinterpret_cast<float *>(ws + off1 + (rows * svw::kFilterMaxK * 4 + 255) / 256 * 256);
  const bool vec = ((static_cast<int64_t>(V) * es) % 16 == 0) && aligned(target_logits, 16) &&
                   aligned(draft_logits, 16);
  const cudaError_t e = svw::launch_filtered(a, dtype, vec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SVW_OK : SVW_ERR_CUDA;
}

svw_status spec_verify_early(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                             int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                             const int32_t *draft_tokens, float temperature, uint64_t seed, int32_t *accept_len,
                             int32_t *next_token, int32_t *status, unsigned long long *bytes_read,
                             void *workspace, size_t workspace_bytes, void *stream) {
  return verify_entry(true, target_logits, draft_logits, dtype, V, N, cu_draft, total_draft_rows, max_len,
                      draft_tokens, temperature, seed, accept_len, next_token, status, bytes_read, workspace,
                      workspace_bytes, stream);
}

// OPD workspace: flags int32 [R] | row constants float4 [R], each 256-aligned
static size_t opd_flags_bytes(int64_t R) { return static_cast<size_t>((R * 4 + 255) / 256 * 256); }
static size_t opd_rowc_bytes(int64_t R) { return static_cast<size_t>((R * 16 + 255) / 256 * 256); }

// flags [R] int32 | row constants [R] float4 | clamped-sum partials [R][kOpdFixParts] float2
size_t svw_opd_workspace_size(int64_t total_draft_rows) {
  if (total_draft_rows <= 0 || total_draft_rows > (int64_t{1} << 40)) return 0;
  return opd_flags_bytes(total_draft_rows) + opd_rowc_bytes(total_draft_rows) +
         static_cast<size_t>(total_draft_rows) * svw::kOpdFixParts * sizeof(float2);
}

svw_status opd_loss(const void *target_logits, const void *draft_logits, svw_dtype dtype,
                    int32_t V, int32_t N, const int32_t *cu_draft, int64_t total_draft_rows,
                    int32_t target_has_bonus_row, float temperature, float clip_c,
                    float lambda_ce, float grad_scale, float *loss, float *dlogits,
                    int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
  if (dtype != SVW_F32 && dtype != SVW_BF16) return SVW_ERR_UNSUPPORTED;
  if (V <= 0 || total_draft_rows <= 0) return SVW_ERR_INVALID_ARG;
  if (target_has_bonus_row && (N <= 0 || !cu_draft)) return SVW_ERR_INVALID_ARG;
  if (!target_logits || !draft_logits || !loss) return SVW_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SVW_ERR_INVALID_ARG;
  if (!(clip_c > 0.f) || !std::isfinite(lambda_ce) || !std::isfinite(grad_scale))
    return SVW_ERR_INVALID_ARG;
  const double kd = 1.4426950408889634 / static_cast<double>(temperature);
  if (!(kd < 3.0e38)) return SVW_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!svw::opd_supported(V, es)) return SVW_ERR_UNSUPPORTED;
  if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(loss, 4) ||
      (dlogits && !aligned(dlogits, 16)) || (cu_draft && !aligned(cu_draft, 4)) ||
      (status && !aligned(status, 4)) || (workspace && !aligned(workspace, 256)))
    return SVW_ERR_MISALIGNED;
  if (workspace && workspace_bytes < svw_opd_workspace_size(total_draft_rows)) return SVW_ERR_WORKSPACE;
  const bool bulk = ((static_cast<int64_t>(V) * es) % 16 == 0) && aligned(target_logits, 16) &&
                    aligned(draft_logits, 16);
  svw::OpdArgs a;
  a.fault = svw::test_fault();
  a.target = target_logits;
  a.draft = draft_logits;
  a.V = V;
  a.N = target_has_bonus_row ? N : 0;
  a.cu = cu_draft;
  a.R = total_draft_rows;
  a.has_bonus = target_has_bonus_row ? 1 : 0;
  a.k = static_cast<float>(kd);
  a.invT = static_cast<float>(1.0 / static_cast<double>(temperature));
  a.clip_c = clip_c;
  a.lambda_ce = lambda_ce;
  a.grad_scale = grad_scale;
  a.loss = loss;
  a.dlogits = dlogits;
  a.status = status;
  a.flags = static_cast<int32_t *>(workspace);
  a.epoch = next_epoch();
  a.rowc = workspace ? reinterpret_cast<float4 *>(static_cast<char *>(workspace) + opd_flags_bytes(total_draft_rows))
                     : nullptr;
  a.fixp = workspace ? reinterpret_cast<float2 *>(static_cast<char *>(workspace) + opd_flags_bytes(total_draft_rows) +
                                                  opd_rowc_bytes(total_draft_rows))
                     : nullptr;
  a.nbonus = 0;
  a.bpart = nullptr;
  a.csr_bad = nullptr;
  const cudaError_t e = svw::launch_opd(a, dtype, bulk, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SVW_OK : SVW_ERR_CUDA;
}

svw_status svw_time_next_launch(const char *kernel, void *begin_event, void *end_event) {
  if (!kernel) {
    g_timer.armed = false;
    return SVW_OK;
  }
  if (!begin_event || !end_event || std::strlen(kernel) >= sizeof(g_timer.kernel)) return SVW_ERR_INVALID_ARG;
  std::strncpy(g_timer.kernel, kernel, sizeof(g_timer.kernel));
  g_timer.begin = reinterpret_cast<cudaEvent_t>(begin_event);
  g_timer.end = reinterpret_cast<cudaEvent_t>(end_event);
  g_timer.armed = true;
  return SVW_OK;
}

size_t svw_verify_opd_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V, svw_dtype dtype) {
  if (n_requests <= 0 || total_draft_rows < 0 || V <= 0 || V > kMaxV) return 0;
  if (dtype != SVW_F32 && dtype != SVW_BF16) return 0;
  return svw::fused_layout(n_requests, total_draft_rows, V).total;
}

size_t svw_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V, int32_t max_len) {
  if (max_len < 1 || max_len > SVW_MAX_LEN) return 0;
  if (n_requests <= 0 || total_draft_rows < 0 || V <= 0 || V > kMaxV) return 0;
  size_t need = 0;
  for (svw_dtype dt : {SVW_F32, SVW_BF16}) {
    need = std::max(need, svw_verify_workspace_size(n_requests, total_draft_rows, V, dt));
    need = std::max(need, svw_verify_early_workspace_size(n_requests, total_draft_rows, V, dt));
    need = std::max(need, svw_verify_filtered_workspace_size(n_requests, total_draft_rows, V, dt));
    need = std::max(need, svw_verify_opd_workspace_size(n_requests, total_draft_rows, V, dt));
  }
  if (total_draft_rows > 0) need = std::max(need, svw_opd_workspace_size(total_draft_rows));
  return need;
}

svw_status spec_verify_opd(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                           int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                           const int32_t *draft_tokens, float temperature, float opd_temperature, uint64_t seed,
                           float clip_c, float lambda_ce, float grad_scale, int32_t *accept_len,
                           int32_t *next_token, float *loss, float *dlogits, int32_t *status, void *workspace,
                           size_t workspace_bytes, void *stream) {
  if (dtype != SVW_F32 && dtype != SVW_BF16) return SVW_ERR_UNSUPPORTED;
  if (V <= 0 || N <= 0 || total_draft_rows <= 0 || max_len < 1) return SVW_ERR_INVALID_ARG;
  if (max_len > SVW_MAX_LEN || V > kMaxV) return SVW_ERR_UNSUPPORTED;
  if (!target_logits || !draft_logits || !cu_draft || !draft_tokens || !accept_len || !next_token || !loss ||
      !workspace)
    return workspace ? SVW_ERR_INVALID_ARG : SVW_ERR_WORKSPACE;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SVW_ERR_INVALID_ARG;
  if (!(opd_temperature > 0.f) || !std::isfinite(opd_temperature)) return SVW_ERR_INVALID_ARG;
  if (temperature > 0.f && temperature != opd_temperature) return SVW_ERR_INVALID_ARG;  // shared softmaxes
  if (!(clip_c > 0.f) || !std::isfinite(lambda_ce) || !std::isfinite(grad_scale)) return SVW_ERR_INVALID_ARG;
  const double kd = 1.4426950408889634 / static_cast<double>(opd_temperature);
  if (!(kd < 3.0e38)) return SVW_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!aligned(target_logits, 16) || !aligned(draft_logits, 16) || !aligned(cu_draft, 4) ||
      !aligned(draft_tokens, 4) || !aligned(accept_len, 4) || !aligned(next_token, 4) || !aligned(loss, 4) ||
      (dlogits && !aligned(dlogits, 16)) || (status && !aligned(status, 4)) || !aligned(workspace, 256))
    return SVW_ERR_MISALIGNED;
  // one pass needs the 16-byte-pitched register-resident path
  if ((static_cast<int64_t>(V) * es) % 16 != 0 || !svw::opd_fast_supported(V, es)) return SVW_ERR_UNSUPPORTED;
  const svw::FusedLayout lay = svw::fused_layout(N, total_draft_rows, V);
  if (workspace_bytes < lay.total) return SVW_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool greedy = (temperature == 0.f);

  svw::OpdArgs o;
  o.fault = svw::test_fault();
  o.target = target_logits;
  o.draft = draft_logits;
  o.V = V;
  o.N = N;
  o.cu = cu_draft;
  o.R = total_draft_rows;
  o.has_bonus = 1;
  o.k = static_cast<float>(kd);
  o.invT = static_cast<float>(1.0 / static_cast<double>(opd_temperature));
  o.clip_c = clip_c;
  o.lambda_ce = lambda_ce;
  o.grad_scale = grad_scale;
  o.loss = loss;
  o.dlogits = dlogits;
  o.status = status;
  o.flags = reinterpret_cast<int32_t *>(ws + lay.flags_off);
  o.rowc = reinterpret_cast<float4 *>(ws + lay.rowc_off);
  o.fixp = reinterpret_cast<float2 *>(ws + lay.fixp_off);
  o.epoch = next_epoch();
  o.nbonus = N;
  o.bpart = reinterpret_cast<float4 *>(ws + lay.bpart_off);
  o.csr_bad = reinterpret_cast<int32_t *>(ws + lay.csr_bad_off);
  int grid = 0;
  cudaError_t e = svw::launch_opd_fused_fast(o, dtype, &grid, st);
  if (e != cudaSuccess) return SVW_ERR_CUDA;

  svw::FusedArgs f;
  f.target = target_logits;
  f.draft = draft_logits;
  f.V = V;
  f.N = N;
  f.cu = cu_draft;
  f.total_rows = total_draft_rows;
  f.max_len = max_len;
  f.tokens = draft_tokens;
  f.k = o.k;
  f.seed = seed;
  f.rowc = o.rowc;
  f.bpart = o.bpart;
  f.bparts = svw::opd_cluster_size(V, es);
  f.csr_bad = o.csr_bad;
  f.csr_grid = grid;
  f.accept_len = accept_len;
  f.next_token = next_token;
  f.status = status;
  // the parts grid (tiny) first, so that the gradient fix-up can run beside
  // the finalize kernel's draw
  e = svw::launch_opd_fix(o, dtype, svw::kFixParts, st);
  if (e != cudaSuccess) return SVW_ERR_CUDA;
  e = svw::launch_fused_finalize(f, dtype, greedy, st);
  if (e != cudaSuccess) return SVW_ERR_CUDA;
  e = svw::launch_opd_fix(o, dtype, svw::kFixGradLast, st);  // rows with a clipped term, exactly
  return e == cudaSuccess ? SVW_OK : SVW_ERR_CUDA;
}

size_t svw_length_head_workspace_size(int32_t n_requests, int32_t k, int32_t hidden_out) {
  if (n_requests <= 0 || k <= 0 || k > SVW_MAX_LEN || hidden_out <= 0) return 0;
  if (static_cast<int64_t>(n_requests) * k > kMaxHeadPositions) return 0;
  return svw::length_head_gemm_bytes(n_requests, k, hidden_out);
}

svw_status length_head(const void *hidden, const void *w1, const float *b1, const float *w2, float b2, int32_t N,
                       int32_t k, int32_t H, int32_t hidden_out, float gamma, float *a_hat, int32_t *k_hat,
                       void *workspace, size_t workspace_bytes, void *stream) {
  if (N <= 0 || k <= 0 || H <= 0 || hidden_out <= 0) return SVW_ERR_INVALID_ARG;
  if (k > SVW_MAX_LEN || static_cast<int64_t>(N) * k > kMaxHeadPositions) return SVW_ERR_UNSUPPORTED;
  if (!hidden || !w1 || !b1 || !w2 || !a_hat || !k_hat) return SVW_ERR_INVALID_ARG;
  if (!workspace) return SVW_ERR_WORKSPACE;
  if (!(gamma > 0.f) || !std::isfinite(gamma) || !std::isfinite(b2)) return SVW_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w1, 16) || !aligned(b1, 4) || !aligned(w2, 4) || !aligned(a_hat, 4) ||
      !aligned(k_hat, 4) || !aligned(workspace, 256))
    return SVW_ERR_MISALIGNED;
  if (H % 8 != 0) return SVW_ERR_UNSUPPORTED;  // 16-byte rows for the GEMM
  if (workspace_bytes < svw_length_head_workspace_size(N, k, hidden_out)) return SVW_ERR_WORKSPACE;
  const int rc = svw::launch_length_head(hidden, w1, b1, w2, b2, N, k, H, hidden_out, gamma, a_hat, k_hat,
                                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  return rc == 0 ? SVW_OK : SVW_ERR_CUDA;
}

svw_status length_head_label(const int32_t *accept_len, const int32_t *cu_draft, const float *a_hat, int32_t N,
                             float *a_star, float *loss, void *stream) {
  if (N <= 0 || !accept_len || !cu_draft || !a_star || (loss && !a_hat)) return SVW_ERR_INVALID_ARG;
  if (!aligned(accept_len, 4) || !aligned(cu_draft, 4) || (a_hat && !aligned(a_hat, 4)) || !aligned(a_star, 4) ||
      (loss && !aligned(loss, 4)))
    return SVW_ERR_MISALIGNED;
  const int rc = svw::launch_length_label(accept_len, cu_draft, a_hat, N, a_star, loss,
                                          static_cast<cudaStream_t>(stream));
  return rc == 0 ? SVW_OK : SVW_ERR_CUDA;
}

}  // extern "C"
