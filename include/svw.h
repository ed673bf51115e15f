/*
 * svw.h -- C ABI of the vocabulary-wide speculative-verification library
 * (serving_vocab_wide_gb300).  Hand-written CUDA for sm_103a (GB300).
 *
 * Two operations, both over full-vocabulary logits (and spec_verify_opd,
 * both on the same batch in one pass), two variants of the verification
 * (spec_verify_early: stops reading each request at its first rejection;
 * spec_verify_filtered: top-k / top-p filtered distributions), plus the
 * adaptive length head that sets the next round's verified lengths
 * (length_head, length_head_label):
 *
 *  spec_verify  batched speculative verification of a ragged batch.  Defined
 *               by "DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.1 (greedy
 *               rule), §5.2 eqs. (6)-(8) and Algorithm 1, and by "AdaFlash:
 *               Taming Variance in Diffusion Speculative Decoding", section
 *               "Speculative Decoding: The Basic Idea", steps 3-4.  Requests
 *               are packed by CSR offsets ("AdaFlash：基于在策略蒸馏扩散草稿器
 *               的自适应投机解码" §2.3: the verify batch holds each request's
 *               own length, not N x k).
 *
 *  opd_loss     entry-wise clipped reverse KL(q||p) + lambda * CE on the
 *               target top-1 token, and its gradient wrt the draft logits.
 *               Defined by "AdaFlash: Taming Variance in Diffusion Speculative
 *               Decoding", sections "The Reverse-KL + Hard-Label Mixture Loss,
 *               Derived" and "Algorithm 2: Entry-Wise Clipped Reverse-KL".
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device pointers (cudaMalloc / PyTorch
 *    CUDA tensors) on the current device.  The caller owns all memory; the
 *    library allocates and frees no device memory and keeps no per-call state
 *    (length_head's GEMM library keeps a host handle and per-shape plans).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are stream-ordered and never synchronise the host.
 *  - The return value covers host-side validation and launch errors only.
 *    Problems that only the device can see (bad CSR offsets, out-of-range
 *    tokens, non-finite rows) are reported by OR-ing SVW_DEV_* bits into
 *    *status (device int32, may be NULL); the caller clears it.
 *  - Logits are row-major [rows, V] in fp32 or bf16.  Rows whose byte pitch
 *    V * sizeof(dtype) is a multiple of 16 with 16-byte aligned bases take the
 *    vectorised / bulk-copy path; any other shape takes a scalar path with the
 *    same results.
 *  - Inputs are read-only; outputs must not alias inputs.
 */
#ifndef SVW_H_
#define SVW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum svw_status {
  SVW_OK = 0,
  SVW_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad temperature ... */
  SVW_ERR_UNSUPPORTED = 2, /* dtype or size outside what the kernels handle         */
  SVW_ERR_UNSUPPORTED_DTYPE = SVW_ERR_UNSUPPORTED, /* the same code, by its other name */
  SVW_ERR_MISALIGNED = 3,  /* a pointer violates its documented alignment            */
  SVW_ERR_WORKSPACE = 4,   /* workspace missing or smaller than its *_workspace_size  */
  SVW_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed            */
  SVW_ERR_BAD_INPUT = 6,   /* device-detected: see svw_device_status()               */
  SVW_ERR_TIMEOUT = 7      /* device-detected: see svw_device_status()               */
} svw_status;

typedef enum svw_dtype { SVW_F32 = 0, SVW_BF16 = 1 } svw_dtype;

/*
 * Bits OR-ed into the device status word.  The word is a bit set, not an
 * svw_status: many CTAs of one call may each find a problem, and an atomic OR
 * of bits is the only way they can report without ordering.  No entry point
 * returns SVW_ERR_BAD_INPUT or SVW_ERR_TIMEOUT from the host (the host never
 * waits for the device); svw_device_status() turns a word the caller has read
 * back into those codes.
 */
#define SVW_DEV_BAD_INPUT 1 /* some request / row was invalid or non-finite   */
#define SVW_DEV_TIMEOUT 2   /* a bounded wait inside a kernel gave up         */

/*
 * The svw_status of a device status word read back by the caller:
 * SVW_ERR_TIMEOUT if SVW_DEV_TIMEOUT is set (results of that call are not
 * valid), else SVW_ERR_BAD_INPUT if SVW_DEV_BAD_INPUT is set (the bad
 * requests / rows carry -1 / NaN, the others are valid), else SVW_OK.
 */
svw_status svw_device_status(int32_t status_word);

/* Largest draft length (positions per request) spec_verify accepts. */
#define SVW_MAX_LEN 32

/*
 * svw_workspace_size -- one workspace size for every entry point on a batch
 * shape: the largest of svw_verify_workspace_size, svw_verify_early_workspace_size,
 * svw_verify_filtered_workspace_size (both dtypes), svw_opd_workspace_size and
 * svw_verify_opd_workspace_size for (n_requests, total_draft_rows, V), so
 * that a caller can size one buffer before it knows which call or dtype it
 * will make.  max_len (1..SVW_MAX_LEN) is checked only.  Returns 0 for
 * invalid arguments.  The per-call functions below give the exact (smaller)
 * sizes.
 */
size_t svw_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V, int32_t max_len);

/*
 * Bytes of device workspace spec_verify needs for this batch shape (any
 * temperature).  Depends only on (n_requests, total_draft_rows, V, dtype).
 * Returns 0 for invalid arguments.
 */
size_t svw_verify_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                 svw_dtype dtype);

/*
 * spec_verify -- verify every request of a ragged batch in one call.
 *
 * Request i owns L_i = cu_draft[i+1] - cu_draft[i] draft positions.
 *   draft_logits  device [total_draft_rows, V]; request i's rows are
 *                 cu_draft[i] .. cu_draft[i+1]-1 (position j at cu_draft[i]+j).
 *   target_logits device [total_draft_rows + N, V]; request i's rows are
 *                 cu_draft[i]+i .. cu_draft[i]+i+L_i: row j is the target's
 *                 distribution at draft position j, the last (j = L_i) is the
 *                 bonus row used when every candidate passes.
 *   cu_draft      device int32 [N+1], cu_draft[0] = 0, non-decreasing,
 *                 cu_draft[N] = total_draft_rows (passed on the host so that
 *                 the call never reads device memory from the host).
 *   max_len       1..SVW_MAX_LEN; requests with L_i outside [1, max_len] are bad.
 *   draft_tokens  device int32 [total_draft_rows], x_j drawn from
 *                 softmax(draft row j / temperature); must be in [0, V).
 *   temperature   0 => greedy: accept x_j iff it is the target argmax of row j
 *                 (raw logits, smallest index wins); next_token is the argmax
 *                 of the first rejected row, or of the bonus row.
 *                 > 0 => accept x_j iff u_j < min(1, p_j(x_j) / q_j(x_j)) with
 *                 p = softmax(target/T), q = softmax(draft/T); the accepted
 *                 length is the leftmost-rejection prefix; next_token is drawn
 *                 by inverse CDF (vocabulary order, smallest v with C_v > w Z)
 *                 from max(0, p - q) at the rejected row, or from p at the
 *                 bonus row.
 *   seed          Philox4x32-10 key (lo 32 bits, hi 32 bits).  u_j uses counter
 *                 {i, j, 0, 0}; the sampling uniform w uses {i, j*, 1, 0}, j*
 *                 the sampled row.  Uniform = (word0 >> 8) * 2^-24.
 *   accept_len    device int32 [N] out; -1 for a bad request.
 *   next_token    device int32 [N] out; -1 for a bad request.
 *   status        device int32 scalar, may be NULL; SVW_DEV_BAD_INPUT is
 *                 OR-ed in if any request is bad (invalid length, token out of
 *                 range, a NaN row, or at T > 0 a row with +Inf or only -Inf).
 *   workspace     device, 256-byte aligned, >= svw_verify_workspace_size(...)
 *                 bytes; contents need not be initialised; not preserved.
 */
svw_status spec_verify(const void *target_logits, const void *draft_logits, svw_dtype dtype,
                       int32_t V, int32_t N, const int32_t *cu_draft, int64_t total_draft_rows,
                       int32_t max_len, const int32_t *draft_tokens, float temperature,
                       uint64_t seed, int32_t *accept_len, int32_t *next_token, int32_t *status,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_early -- spec_verify that stops reading a request at its first
 * rejection.
 *
 * Leftmost rejection ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.2,
 * Algorithm 1) makes every row after a request's first rejected position
 * irrelevant to its result, and acceptance falls with the position
 * ("AdaFlash：基于在策略蒸馏扩散草稿器的自适应投机解码" §3.3, Figure 2(c):
 * from about 0.9 at the first position to 0.13-0.26 at the fifteenth).  The
 * rows are streamed position by position across the batch and each accept
 * test runs as soon as its two rows are reduced; rows at positions after a
 * known rejection are skipped.  Which later rows still get read depends on
 * timing, the results do not.
 *
 * Arguments and results as for spec_verify (same accept_len and next_token,
 * bit for bit, same uniforms), with these differences:
 *   - a request is bad (accept_len = next_token = -1) if a row at or before
 *     its first rejected position (the bonus row when none is rejected) is
 *     non-finite, or if any of its tokens is out of range; rows after the
 *     first rejection are not checked (they need not be read);
 *   bytes_read    device uint64 scalar out, may be NULL: the logit bytes this
 *                 call streamed from the two tensors (without the one row
 *                 pair the draw reads again).  Reset by the call.  8-byte
 *                 aligned.
 *   workspace     >= svw_verify_early_workspace_size(...) bytes.
 */
size_t svw_verify_early_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                       svw_dtype dtype);

svw_status spec_verify_early(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                             int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                             const int32_t *draft_tokens, float temperature, uint64_t seed, int32_t *accept_len,
                             int32_t *next_token, int32_t *status, unsigned long long *bytes_read,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Largest top_k spec_verify_filtered accepts. */
#define SVW_FILTER_MAX_K 1024

/*
 * spec_verify_filtered -- spec_verify with both distributions top-k / top-p
 * filtered.
 *
 * The pages verify with the full temperature softmax; serving stacks usually
 * filter first.  This variant is not on the pages and follows this reading:
 * p and q are filtered with the same (temperature, top_k, top_p) -- entries
 * ordered by raw logit descending, the smaller index first among equal
 * logits; the first top_k kept; of those, the shortest prefix whose
 * probability reaches top_p times their total kept; renormalised -- and the
 * method of spec_verify ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.2
 * eqs. (6)-(8), Algorithm 1) runs on the filtered p' and q': x_j is accepted
 * iff u_j < min(1, p'(x_j) / q'(x_j)) (a token outside the target's kept set
 * is rejected; q'(x_j) = 0 with p'(x_j) > 0 is accepted), the next token is
 * drawn from [p' - q']_+ at the rejected row or from p' at the bonus row, by
 * the same inverse CDF in vocabulary order.  draft_tokens are drawn from q'.
 *
 * Arguments and results as for spec_verify, plus:
 *   top_k         1 .. SVW_FILTER_MAX_K (a larger value returns
 *                 SVW_ERR_UNSUPPORTED; values >= V keep every entry).
 *   top_p         (0, 1]; 1 keeps the whole top-k set.
 *   temperature   0 => greedy spec_verify (filtering keeps the argmax).
 *   workspace     >= svw_verify_filtered_workspace_size(...) bytes.
 * V is limited by shared memory (about 200 KB per CTA: V <= ~600 k for bf16
 * at top_k <= 256); larger rows return SVW_ERR_UNSUPPORTED.
 */
size_t svw_verify_filtered_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                          svw_dtype dtype);

svw_status spec_verify_filtered(const void *target_logits, const void *draft_logits, svw_dtype dtype, int32_t V,
                                int32_t N, const int32_t *cu_draft, int64_t total_draft_rows, int32_t max_len,
                                const int32_t *draft_tokens, float temperature, int32_t top_k, float top_p,
                                uint64_t seed, int32_t *accept_len, int32_t *next_token, int32_t *status,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * opd_loss -- per draft row r (0 <= r < total_draft_rows), paired with one
 * target row:
 *   lp = log softmax(target/T), lq = log softmax(draft/T), q = exp(lq)
 *   t_v = q_v (lq_v - lp_v)          (t_v := 0 where q_v = 0)
 *   loss[r] = sum_v clamp(t_v, -clip_c, clip_c) + lambda_ce * (-lq[x*]),
 *             x* = argmax of the raw target row (smallest index wins)
 *   dlogits[r, v] = grad_scale / T * ( q_v (a_v - S) + lambda_ce (q_v - [v == x*]) ),
 *             a_v = [-clip_c < t_v < clip_c] (lq_v - lp_v + 1), S = sum_v q_v a_v
 * i.e. dlogits is grad_scale times the gradient of sum_r loss[r] wrt the
 * draft logits (the target is frozen).  Pass grad_scale = 1/k for the mean
 * over k positions.
 *
 *   target_has_bonus_row  1: verify layout -- target has total_draft_rows + N
 *                 rows and draft row r of request i pairs with target row r + i
 *                 (cu_draft device [N+1] required).  0: rows pair 1:1, target
 *                 has total_draft_rows rows, cu_draft and N are ignored.
 *   temperature   > 0 (the reverse-KL temperature; 1.0 in the review).
 *   clip_c        > 0 (may be +inf: no clipping).
 *   loss          device float [total_draft_rows] out (NaN for a bad row).
 *   dlogits       device float [total_draft_rows, V] out, 16-byte aligned;
 *                 NULL computes the loss only.
 *   status        as for spec_verify (SVW_DEV_BAD_INPUT for a non-finite row
 *                 or a row outside its request's CSR range; SVW_DEV_TIMEOUT if
 *                 a bounded wait on a bulk copy gave up).
 *   workspace     device, 256-byte aligned, >= svw_opd_workspace_size(
 *                 total_draft_rows) bytes (per row: a flag, the row
 *                 constants, 128 partial clamped sums; about 1 KB), contents
 *                 need not be initialised, not preserved; or NULL.  With a
 *                 workspace, rows whose byte pitch is a multiple of 16 take
 *                 a one-exchange fast pass, which also leaves each row's
 *                 exact clamped sum as partials, and only the gradient of
 *                 rows where some term reaches the clip (or the draft has
 *                 masked entries) is written again; the results are the same
 *                 either way (up to float rounding order).
 */
size_t svw_opd_workspace_size(int64_t total_draft_rows);

svw_status opd_loss(const void *target_logits, const void *draft_logits, svw_dtype dtype,
                    int32_t V, int32_t N, const int32_t *cu_draft, int64_t total_draft_rows,
                    int32_t target_has_bonus_row, float temperature, float clip_c,
                    float lambda_ce, float grad_scale, float *loss, float *dlogits,
                    int32_t *status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_opd -- spec_verify and opd_loss (verify layout) on the same
 * batch in one pass over the logits.  The distillation signal is a byproduct
 * of verification ("AdaFlash: Taming Variance in Diffusion Speculative
 * Decoding", "Method Part 1: On-Policy Distillation (OPD) for Diffusion
 * Drafters", "Algorithm, Step by Step" step 3 and Figure 2: the target's
 * distribution at every drafted position is already computed by
 * verification), so both results come from one read of both logit tensors:
 * the OPD kernel's row softmaxes serve the accept tests, and the bonus rows
 * are reduced in the same pass.
 *
 * Arguments as for spec_verify and opd_loss, plus:
 *   temperature      verification temperature (0: greedy).
 *   opd_temperature  > 0, the reverse-KL temperature; must equal temperature
 *                    when temperature > 0 (the softmaxes are shared), else
 *                    SVW_ERR_INVALID_ARG.
 *   loss, dlogits    as for opd_loss with target_has_bonus_row = 1.
 *   workspace        device, 256-byte aligned, >= svw_verify_opd_workspace_size
 *                    bytes; contents need not be initialised; not preserved.
 * accept_len / next_token equal spec_verify's and loss / dlogits equal
 * opd_loss's on the same inputs, with one difference: a request with a
 * non-finite row (NaN, +Inf, or only -Inf in any of its target, bonus or
 * draft rows) is reported bad at every temperature (spec_verify at T = 0
 * only rejects NaN target rows).  Needs 16-byte aligned bases and a 16-byte
 * row pitch (V * sizeof(dtype) % 16 == 0) and a row the one-pass kernel can
 * hold on chip (V = 151936 bf16 fits); otherwise SVW_ERR_UNSUPPORTED.
 */
size_t svw_verify_opd_workspace_size(int32_t n_requests, int64_t total_draft_rows, int32_t V,
                                     svw_dtype dtype);

svw_status spec_verify_opd(const void *target_logits, const void *draft_logits, svw_dtype dtype,
                           int32_t V, int32_t N, const int32_t *cu_draft, int64_t total_draft_rows,
                           int32_t max_len, const int32_t *draft_tokens, float temperature,
                           float opd_temperature, uint64_t seed, float clip_c, float lambda_ce,
                           float grad_scale, int32_t *accept_len, int32_t *next_token, float *loss,
                           float *dlogits, int32_t *status, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * length_head -- the adaptive length head's forward pass ("AdaFlash: Taming
 * Variance in Diffusion Speculative Decoding", "Algorithm 3: Adaptive Length
 * Head, Forward Pass"; "AdaFlash：基于在策略蒸馏扩散草稿器的自适应投机解码" §2.2):
 * for each request i, from its drafter hidden states h_i (k positions x H),
 *   h'_p = SiLU(W1 h_i[p] + b1),  hbar = (1/k) sum_p h'_p,
 *   a_hat[i] = sigmoid(w2 . hbar + b2),
 *   k_hat[i] = clamp(floor(gamma a_hat[i] k), 1, k)   (next round's verified length).
 *   hidden     device bf16 [N, k, H] row-major, 16-byte aligned, H % 8 == 0;
 *              N k <= 2^20 positions and k <= SVW_MAX_LEN (else
 *              SVW_ERR_UNSUPPORTED, and a workspace size of 0).
 *   w1         device bf16 [hidden_out, H] row-major (H' = hidden_out < H).
 *   b1, w2     device float [hidden_out];  b2, gamma > 0 on the host.
 *   a_hat      device float [N] out (before the gamma scaling);  k_hat device int32 [N] out.
 *   workspace  device, 256-byte aligned, >= svw_length_head_workspace_size(N, k,
 *              hidden_out) bytes: one fp32 per position and 256-wide column
 *              tile of W1 (N k ceil(H'/256) floats, rounded up to 256 bytes);
 *              contents need not be initialised.
 * The projection of the N k positions runs on the tensor cores (tcgen05 MMA,
 * operands staged by TMA, fp32 accumulation in tensor memory) in four K
 * quarters, one thread-block cluster per 128 positions; the quarters are
 * summed inside the cluster (distributed shared memory), and the same kernel
 * applies bias and SiLU and dots each position with w2.  A second, small
 * kernel adds each request's position dots and applies the mean, b2,
 * sigmoid, gamma, floor and clamp.  Two kernel launches, each a programmatic
 * dependent of the one ahead (its set-up overlaps that kernel's tail); no
 * library call; the host only encodes the two TMA descriptors.  If a bounded
 * wait inside the projection gives up, the affected requests get a_hat = NaN.
 */
size_t svw_length_head_workspace_size(int32_t n_requests, int32_t k, int32_t hidden_out);

svw_status length_head(const void *hidden, const void *w1, const float *b1, const float *w2, float b2,
                       int32_t N, int32_t k, int32_t H, int32_t hidden_out, float gamma, float *a_hat,
                       int32_t *k_hat, void *workspace, size_t workspace_bytes, void *stream);

/*
 * length_head_label -- the length head's training signal ("AdaFlash: Taming
 * Variance in Diffusion Speculative Decoding", "Online Update of the Length
 * Head, Derived"): a_star[i] = accept_len[i] / L_i, the accepted fraction of
 * the L_i = cu_draft[i+1] - cu_draft[i] verified tokens, and (loss not NULL)
 * loss[i] = (a_hat[i] - a_star[i])^2.  A bad request (accept_len < 0) gets
 * NaN.  All pointers device; a_hat may be NULL when loss is NULL.
 */
svw_status length_head_label(const int32_t *accept_len, const int32_t *cu_draft, const float *a_hat, int32_t N,
                             float *a_star, float *loss, void *stream);

/*
 * spec_verify_noalloc -- spec_verify for callers that cannot allocate device
 * memory.  No counterpart on the pages: it exists only because some callers
 * have no allocator to hand over a workspace (a plain C serving loop, a
 * plug-in inside an engine whose memory pool is sized up front and which
 * forbids cudaMalloc -- a device-synchronising call -- mid-step, a thin launch
 * wrapper that only forwards tensors).
 *
 * Same arguments and results as spec_verify, minus the workspace: the library
 * keeps one fixed scratch area of SVW_NOALLOC_SCRATCH_BYTES per GPU (a
 * file-scope device array, resident for the life of the process on every GPU
 * that loads the library).  This call allocates nothing and frees nothing.
 *  - Batches whose svw_verify_workspace_size(...) exceeds the scratch return
 *    SVW_ERR_UNSUPPORTED without launching (e.g. N = 256 requests, 4096 draft
 *    rows at V = 151936 bf16 fit).
 *  - Argument checks run first and give spec_verify's codes; only a batch
 *    that passes them and needs more than the scratch gets SVW_ERR_UNSUPPORTED.
 *  - `stream` must belong to the current device (the scratch used is the
 *    current device's); otherwise SVW_ERR_INVALID_ARG, nothing launched.
 *  - The first call on each device looks the scratch's device address up
 *    (cudaGetSymbolAddress with that device current); make that first call
 *    before capturing the stream into a graph.
 *  - All calls share the scratch.  Calls whose kernels may overlap on the GPU
 *    (different streams without ordering, several host threads) race on it and
 *    corrupt each other's results; serialise them on one stream.
 */
#define SVW_NOALLOC_SCRATCH_BYTES (32u << 20)
svw_status spec_verify_noalloc(const void *target_logits, const void *draft_logits, svw_dtype dtype,
                               int32_t V, int32_t N, const int32_t *cu_draft,
                               int64_t total_draft_rows, int32_t max_len,
                               const int32_t *draft_tokens, float temperature, uint64_t seed,
                               int32_t *accept_len, int32_t *next_token, int32_t *status,
                               void *stream);

/*
 * svw_time_next_launch -- measurement hook, not part of the method.  Arms a
 * one-shot timer on the calling host thread: the next launch of the named
 * kernel made from this thread ("early_plan", "verify_stats",
 * "verify_finalize", "verify_early_cluster", "filter_rows", "filtered_finalize",
 * "opd_fast_kernel", "opd_fix_parts", "opd_fix_grad", "opd_exact_kernel",
 * "fused_finalize", "length_head_mma", "length_head_final") records
 * begin_event just before it and end_event just after it on the launch stream (cudaEvent_t handles passed as void*, owned
 * by the caller).  kernel = NULL disarms.  The library records nothing
 * unless armed.  Lets a benchmark time one kernel of a multi-kernel call with
 * CUDA events on the launch stream.
 */
svw_status svw_time_next_launch(const char *kernel, void *begin_event, void *end_event);

/*
 * Test hooks for the bounded waits, not part of the method ("failure
 * detection": a wait that runs out is reported, never a hang).
 *
 * svw_set_wait_limit -- the deadline, in SM clock cycles, of every bounded
 * wait in the library's kernels on the current device (default 4e9, about
 * 2 s).  cycles > 0, else SVW_ERR_INVALID_ARG.  Takes effect for kernels
 * launched after it returns.  A limit far below a copy's latency makes
 * healthy waits give up too; use it with svw_set_fault, at about 1e6 cycles,
 * so that only the injected wait runs out.
 *
 * svw_set_fault -- 0: none (default); 1: in the next calls until reset, CTA 0
 * of verify_stats (spec_verify) and cluster 0 of opd_fast_kernel
 * (opd_loss, spec_verify_opd) issue no bulk copy, so their first wait
 * runs out with nothing in flight: the call returns, its status word holds
 * SVW_DEV_TIMEOUT, and the results of the affected rows are void.  Other
 * values: SVW_ERR_INVALID_ARG.  Host-side state, shared by all threads.
 */
svw_status svw_set_wait_limit(int64_t cycles);
svw_status svw_set_fault(int32_t kind);

/* Human-readable name of a status code (static string). */
const char *svw_status_string(svw_status s);

/* Library ABI version: 100 * major + minor. */
int32_t svw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SVW_H_ */
