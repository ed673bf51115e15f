// svw_internal.h -- host-side declarations shared by the C-ABI layer and the
// kernel launchers.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/svw.h"

namespace svw {

// Measurement hook behind svw_time_next_launch: a launcher calls
// timer_before(name) just before launching kernel `name` and timer_after with
// what it returned just after; both do nothing unless the calling host thread
// armed a timer for that kernel.
void *timer_before(const char *kernel, cudaStream_t stream);
void timer_after(void *end_event, cudaStream_t stream);

// per-(row, chunk) partial result of the streaming row-statistics pass
struct alignas(16) Partial {
  float m;      // raw maximum of the chunk (argmax value in greedy mode)
  float s;      // sum of 2^((x - m) * log2(e)/T) over the chunk (unused when greedy)
  int32_t idx;  // argmax index (greedy), INT32_MAX if none
  int32_t nan;  // chunk holds a NaN (greedy)
};

// how one vocabulary row is split into work items
struct ChunkPlan {
  int32_t C;          // chunks per row (1..32)
  int32_t chunk_len;  // elements per chunk (multiple of 8)
};
ChunkPlan plan_chunks(int64_t V, int esize);

struct VerifyLayout {
  size_t part_off, csr_bad_off, total;
};
VerifyLayout verify_layout(int32_t N, int64_t total_rows, int64_t V, int esize);
constexpr int kMaxStatsGrid = 1024;  // CTAs of the stats kernel (one CSR check flag each)

struct VerifyArgs {
  const void *target;
  const void *draft;
  int64_t V;
  int32_t N;
  const int32_t *cu;
  int64_t total_rows;
  int64_t rows_t;  // total_rows + N
  int32_t max_len;
  const int32_t *tokens;
  float k;  // log2(e) / T  (T > 0)
  uint64_t seed;
  int32_t *accept_len;
  int32_t *next_token;
  int32_t *status;
  Partial *part;                     // [(rows_t + total_rows) * C * 16] per-warp chunk partials
  int32_t *csr_bad;                  // [stats grid] CSR offsets inconsistent (per stats CTA)
  int32_t stats_grid;                // CTAs of the stats kernel
  int32_t C;
  int32_t chunk_len;
  int64_t total_items;
  // early exit (spec_verify_early); unused otherwise
  int32_t *cnt;                    // [N * max_len] partials delivered per accept test (by slot)
  int32_t *rej;                    // [N] first rejected position found (INT32_MAX: none yet)
  int32_t *badpos;                 // [N] first position with a bad row or token found
  int32_t *stop;                   // [N] by slot: first position that stops the request
  int4 *pinfo;                     // [valid requests] {request, first draft row, L, 0}, longest first
  int64_t *W;                      // [max_len + 2] first item of each position wave
  int32_t *waveA;                  // [max_len + 1] requests longer than each position
  unsigned long long *bytes_read;  // logit bytes streamed (may be NULL)
  int32_t *nvalid;                 // valid requests (the plan's record count)
  int32_t *qnext;                  // cluster path: next record slot to hand out
  int4 *eres;                      // cluster path, per request: {stop position, bad, greedy argmax, 0}
  float4 *erow;                    // cluster path, per request: {m_T, l_T, m_D, l_D} at the stop position
  int32_t fault;                   // test-only (svw_set_fault): 1 = the stats kernel's CTA 0 issues no copy
};

cudaError_t launch_verify(const VerifyArgs &a, int dtype, bool vec, bool greedy,
                          cudaStream_t stream);
// workspace of spec_verify_early: spec_verify's, then the early-exit state
struct EarlyLayout {
  size_t part_off, csr_bad_off, cnt_off, rej_off, badpos_off, stop_off, pinfo_off, wave_off, eres_off, erow_off,
      total;
};
// the cluster path of spec_verify_early (early.cu): CL = 0 if not applicable
struct EarlyClusterPlan {
  int CL;
  int SL;
  int slice_bytes;
  size_t smem;
};
EarlyClusterPlan early_cluster_plan(int64_t V, int esize, bool greedy);
cudaError_t launch_early_cluster(const VerifyArgs &a, int dtype, bool greedy, const EarlyClusterPlan &p,
                                 cudaStream_t stream);
EarlyLayout early_layout(int32_t N, int64_t total_rows, int64_t V, int esize);
cudaError_t launch_verify_early(const VerifyArgs &a, int dtype, bool vec, bool greedy, cudaStream_t stream);
// workspace of spec_verify_opd (fused verification + OPD)
struct FusedLayout {
  size_t flags_off, rowc_off, bpart_off, fixp_off, csr_bad_off, total;
};
FusedLayout fused_layout(int32_t N, int64_t total_rows, int64_t V);

// per-request step of spec_verify_opd: validation, accept tests from the
// fast kernel's row constants, leftmost rejection, next token / sampling row
struct FusedArgs {
  const void *target;
  const void *draft;
  int64_t V;
  int32_t N;
  const int32_t *cu;
  int64_t total_rows;
  int32_t max_len;
  const int32_t *tokens;
  float k;  // log2(e) / T of the verification (T > 0)
  uint64_t seed;
  const float4 *rowc;  // [R] Ct, dC = Cd - Ct, x*, target row (NaN: bad row)
  const float4 *bpart;  // [N * kBonusParts] bonus-row partials of the fast kernel's CTAs
  int32_t bparts;       // partials per bonus row (the fast kernel's cluster size)
  const int32_t *csr_bad;
  int32_t csr_grid;
  int32_t *accept_len;
  int32_t *next_token;
  int32_t *status;
};
int draw_cluster(int N);
int32_t test_fault();  // the fault set by svw_set_fault (0: none)  // CTAs per request of a finalize grid that draws (T > 0)
cudaError_t launch_fused_finalize(const FusedArgs &a, int dtype, bool greedy, cudaStream_t stream);

// adaptive length head (lengthhead.cu); 0 on success
size_t length_head_gemm_bytes(int32_t N, int32_t k, int32_t Hp);  // per-position partial dots
int launch_length_head(const void *hidden, const void *w1, const float *b1, const float *w2, float b2, int32_t N,
                       int32_t k, int32_t H, int32_t Hp, float gamma, float *a_hat, int32_t *k_hat,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream);
int launch_length_label(const int32_t *accept_len, const int32_t *cu, const float *a_hat, int32_t N,
                        float *a_star, float *loss, cudaStream_t stream);

// top-k / top-p filtered verification (filtered.cu)
constexpr int kFilterMaxK = 1024;  // largest top_k (one kept entry per thread of a CTA)
struct FilterArgs {
  const void *target;
  const void *draft;
  int64_t V;
  int32_t N;
  const int32_t *cu;
  int64_t R;       // draft rows
  int64_t rows_t;  // target rows (R + N)
  int32_t max_len;
  const int32_t *tokens;
  float k;  // log2(e) / T  (T > 0)
  int32_t top_k;
  float top_p;
  int32_t cand;  // candidate slots per CTA
  int32_t gs;    // entries per group (8 .. 128, a power of two)
  uint64_t seed;
  int32_t *accept_len;
  int32_t *next_token;
  int32_t *status;
  int32_t *cnt;   // [rows_t + R] kept entries per row (-1: the row has no softmax)
  int32_t *lidx;  // [rows_t + R][kFilterMaxK] kept indices, ascending
  float *lp;      // [rows_t + R][kFilterMaxK] their filtered probabilities
};
int filter_candidates(int32_t top_k);
int filter_group(int32_t top_k);
size_t filter_smem_bytes(int64_t V, int esize, int32_t top_k);
cudaError_t launch_filtered(const FilterArgs &a, int dtype, bool vec, cudaStream_t stream);

constexpr int kOpdFixChunks = 64;  // vocabulary chunks per row of the OPD fix-up grid (one warp each)
constexpr int kOpdFixParts = 128;  // partial sums per row from the fast kernel (one per warp of the cluster)
constexpr int kBonusParts = 8;  // bonus-row partial slots per request (the largest OPD cluster)

struct OpdArgs {
  const void *target;
  const void *draft;
  int64_t V;
  int32_t N;
  const int32_t *cu;
  int64_t R;  // draft rows
  int32_t has_bonus;
  float k;     // log2(e) / T
  float invT;  // 1 / T
  float clip_c;
  float lambda_ce;
  float grad_scale;
  float *loss;
  float *dlogits;
  int32_t *status;
  // workspace of the fast path (NULL: the exact kernel takes every row)
  int32_t *flags;  // [R] == epoch: rows the fix-up must redo; == epoch ^ 0x40000000: only their loss
  float4 *rowc;    // [R] row constants of the fast kernel: Ct, dC = Cd - Ct, x*, target row (NaN: bad row)
  float2 *fixp;    // [R][kOpdFixParts] per-warp partials of the fast kernel (clamped sum, S - 1; nats)
  int32_t epoch;   // this call's tag (never 0)
  // fused verification (spec_verify_opd): after the R draft rows the fast
  // kernel also reduces the N bonus target rows, one partial per CTA of the
  // cluster (bpart[i * kBonusParts + rank] = {max, exp-sum, first argmax,
  // flags}), and checks the CSR offsets (csr_bad[CTA])
  int32_t nbonus;
  float4 *bpart;
  int32_t *csr_bad;
  int32_t fault;  // test-only (svw_set_fault): 1 = cluster 0 of the fast kernel issues no copy
};

cudaError_t launch_opd(const OpdArgs &a, int dtype, bool bulk, cudaStream_t stream);
// fast kernel with bonus rows and CSR checks, then the fix-up kernel is left
// to launch_opd_fix; returns the fast kernel's grid size in *grid
bool opd_fast_supported(int64_t V, int esize);
int opd_cluster_size(int64_t V, int esize);  // CTAs per row in the OPD kernels
cudaError_t launch_opd_fused_fast(const OpdArgs &a, int dtype, int *grid, cudaStream_t stream);
// which fix-up grids launch_opd_fix launches (see opd.cu)
constexpr int kFixNone = 0, kFixBoth = 1, kFixParts = 2, kFixGradLast = 3;
cudaError_t launch_opd_fix(const OpdArgs &a, int dtype, int which, cudaStream_t stream);

}  // namespace svw
