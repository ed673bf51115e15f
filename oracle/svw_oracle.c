/*
 * svw_oracle.c -- the CPU oracle for batched speculative verification and the
 * on-policy-distillation (OPD) loss.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the GPU path computes.  It is compiled into its own shared
 * library and loaded only by the tests, by __graft_entry__.smoke() and by the
 * CPU-baseline leg of bench.py.  It shares no code, header, table or helper
 * with the CUDA library under serving_vocab_wide_gb300/csrc, and never calls it.
 *
 * Arithmetic: IEEE binary64 throughout.  Every bf16 / fp32 input element is
 * converted exactly to double before use.  Sums run sequentially in vocabulary
 * index order.  No blocking, fusion or reordering beyond what the definitions
 * state.
 *
 * Sources (page title, then the section / equation used):
 *  [DF]  "DFlash 阅读笔记：并行起草、目标特征与精确验证" (reading notes on
 *        "DFlash: Block Diffusion for Flash Speculative Decoding"):
 *        §5.1 greedy verification; §5.2 eq. (6) acceptance probability,
 *        eq. (7) residual distribution, eq. (8) losslessness; Algorithm 1
 *        (the exact speculative cycle: left-to-right check, residual on first
 *        rejection, bonus token when every candidate passes).
 *  [AR]  "AdaFlash: Taming Variance in Diffusion Speculative Decoding"
 *        (technical review): "Speculative Decoding: The Basic Idea" steps 3-4;
 *        "The Reverse-KL + Hard-Label Mixture Loss, Derived" (l_hard with the
 *        target top-1 token, l_rkl); "Algorithm 2: Entry-Wise Clipped
 *        Reverse-KL" and the closed form after it; "A Fully Worked Numeric
 *        Example".
 *  [AP]  "AdaFlash：基于在策略蒸馏扩散草稿器的自适应投机解码" §2.3: the verify
 *        batch packs each request's own verified length (sum of k_i tokens,
 *        not N x k), expressed here by CSR offsets; §2.2 the
 *        adaptive length head (k_hat = clamp(floor(gamma a_hat k), 1, k)).
 *  [AR]  also "Method Part 2: The Adaptive Length Head": "Algorithm 3:
 *        Adaptive Length Head, Forward Pass" and "Online Update of the Length
 *        Head, Derived" (l_len = (a_hat - a*)^2, a* the accepted fraction of
 *        the verified tokens).
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes of the repository):
 *  - Clipping: each (position, vocab entry) term is clamped to [-c, c] before
 *    the vocabulary sum.  The review's Algorithm 2 writes a one-sided
 *    min(term, delta); for c >= 1/e the lower bound can never bind (a term
 *    q log(q/p) is >= -p/e >= -1/e), so the two readings agree there.
 *  - Loss mixture: loss = rkl_clip + lambda * CE per position (the review's
 *    alpha form equals (1 - alpha) times this with lambda = alpha/(1-alpha)).
 *    No 1/k mean: the loss is per position and the gradient is that of the sum
 *    of per-position losses, times grad_scale.
 *  - The gradient is not printed on the pages; it is the chain rule through
 *    the temperature softmax of the draft logits (target frozen):
 *      dL/dz_v = grad_scale/T * ( q_v (a_v - S) + lambda (q_v - [v == x*]) ),
 *      a_v = [-c < t_v < c] (lq_v - lp_v + 1),   S = sum_v q_v a_v.
 *  - Argmax (greedy verify and x*) is over raw logits, smallest index wins.
 *  - Inverse-CDF order is vocabulary index order with the strict rule
 *    next = min{ v : C_v > w Z }.
 *  - q(x) == 0 for a drawn token: threshold 1 (accept).  Z == 0 after a
 *    rejection: sample from p at that row instead, flagged "degenerate".
 *  - Uniforms: U(seed, i, j, s) = (Philox4x32-10(key = {lo32 seed, hi32 seed},
 *    counter = {i, j, s, 0}).word0 >> 8) * 2^-24; stream s = 0 for the accept
 *    test of position j, s = 1 for the token drawn at row j.  Philox4x32-10 is
 *    written from its published definition (Salmon, Moraes, Dror, Shaw,
 *    "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).
 *  - A row holding NaN, +Inf, or only -Inf has no softmax: the request (or
 *    OPD row) is reported bad.  At temperature 0 only NaN makes a row bad.
 *  - Top-k / top-p filtered verification is not on the pages (a serving
 *    variant).  This build's reading: both distributions are filtered with
 *    the same (T, top_k, top_p) before the method runs.  Entries are ordered
 *    by raw logit descending, smaller index first among equal logits; the
 *    first K = min(top_k, V) are kept; of those, the shortest prefix whose
 *    cumulative probability reaches top_p times their total (summed in that
 *    order) is kept; the kept probabilities are renormalised.  The accept
 *    test, residual and bonus draw then use the filtered p' and q'; a token
 *    outside the target's kept set has p'(x) = 0 and is rejected.  At T = 0
 *    filtering keeps the argmax, so greedy verification is unchanged.
 *  - Length head: the pages fix the layer order (per-position Linear + SiLU,
 *    mean over the k positions, Linear + sigmoid, times gamma, floor, clamp)
 *    but not the projected width H' (only H' < H); it is an argument.  The
 *    MSE label compares the unscaled sigmoid output a_hat with a* =
 *    accept_len / L (gamma is a serving knob applied after the prediction).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* flag bits reported per request (verify) or per row (OPD) */
#define FLAG_NEAR_ACCEPT 1 /* |u_j - thr_j| < 1e-5 at a decided position */
#define FLAG_NEAR_CDF 2    /* a CDF boundary within 1e-5 * Z of w * Z     */
#define FLAG_DEGENERATE 4  /* Z == 0 after a rejection                    */
#define FLAG_BAD 8         /* invalid request / non-finite row            */
#define FLAG_NEAR_CLIP 16  /* some |t_v| within 1e-5 * c of the clip c    */
#define FLAG_NEAR_FLOOR 32 /* gamma a_hat k within 1e-4 of an integer       */
#define FLAG_NEAR_FILTER 64 /* a top-p cut within 1e-5 of the threshold     */

#define BAND 1e-5

/* ------------------------------------------------------------------ */
/* element access                                                      */
/* ------------------------------------------------------------------ */
static double elem(const void *base, int dtype, int64_t row, int64_t V, int64_t v) {
  int64_t k = row * V + v;
  if (dtype == ORACLE_BF16) {
    uint16_t b = ((const uint16_t *)base)[k];
    uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
  }
  return (double)((const float *)base)[k];
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11)                                 */
/* ------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u; /* round multipliers */
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u; /* key schedule (Weyl) */
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { /* the key is bumped before every round after the first */
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

double oracle_uniform(uint64_t seed, uint32_t i, uint32_t j, uint32_t s) {
  uint32_t ctr[4] = {i, j, s, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------ */
/* row helpers                                                         */
/* ------------------------------------------------------------------ */

/* 1 if the row has a NaN; 2 if it has +Inf; 4 if every entry is -Inf */
static int row_defects(const void *x, int dtype, int64_t row, int64_t V) {
  int has_nan = 0, has_pinf = 0, all_minf = 1;
  for (int64_t v = 0; v < V; ++v) {
    double a = elem(x, dtype, row, V, v);
    if (isnan(a)) has_nan = 1;
    else if (isinf(a) && a > 0) has_pinf = 1;
    if (!(isinf(a) && a < 0)) all_minf = 0;
  }
  return has_nan | (has_pinf << 1) | (all_minf << 2);
}

/* argmax over raw logits, smallest index among equal maxima (NaN ignored) */
static int64_t row_argmax(const void *x, int dtype, int64_t row, int64_t V) {
  int64_t best = -1;
  double bv = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double a = elem(x, dtype, row, V, v);
    if (isnan(a)) continue;
    if (best < 0 || a > bv) {
      best = v;
      bv = a;
    }
  }
  return best;
}

/* out[v] = softmax(x_row / T)[v], max-subtracted, sequential sum in index order */
static void row_softmax(const void *x, int dtype, int64_t row, int64_t V, double T, double *out) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double a = elem(x, dtype, row, V, v) / T;
    if (a > m) m = a;
  }
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    out[v] = exp(elem(x, dtype, row, V, v) / T - m);
    s += out[v];
  }
  for (int64_t v = 0; v < V; ++v) out[v] /= s;
}

/* log-softmax of x_row / T: out[v] = x_v/T - LSE(x/T) */
static void row_log_softmax(const void *x, int dtype, int64_t row, int64_t V, double T, double *out) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double a = elem(x, dtype, row, V, v) / T;
    if (a > m) m = a;
  }
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) s += exp(elem(x, dtype, row, V, v) / T - m);
  double lse = m + log(s);
  for (int64_t v = 0; v < V; ++v) out[v] = elem(x, dtype, row, V, v) / T - lse;
}

/* Inverse CDF over non-negative weights r[0..V) with total Z:
 * next = min{ v : C_v > w Z }, C_v the sequential prefix sum in index order.
 * If rounding leaves no such v, the last index with r_v > 0 is taken.
 * Sets *near when a boundary C_{next-1} or C_next lies within BAND * Z of w Z. */
static int64_t inverse_cdf(const double *r, int64_t V, double Z, double w, int *near) {
  double t = w * Z;
  double C = 0.0, Cprev = 0.0;
  int64_t pick = -1, last_pos = -1;
  for (int64_t v = 0; v < V; ++v) {
    if (r[v] > 0.0) last_pos = v;
    Cprev = C;
    C += r[v];
    if (pick < 0 && C > t) {
      pick = v;
      if (fabs(Cprev - t) < BAND * Z || fabs(C - t) < BAND * Z) *near = 1;
    }
  }
  if (pick < 0) {
    pick = last_pos;
    *near = 1;
  }
  return pick;
}

/* Distance, as a fraction of Z, from t = w Z to the CDF interval
 * [C_{alt-1}, C_alt) of token alt (0 if t lies inside it, i.e. if the inverse
 * CDF of [DF] §5.2 eq. (7) would draw alt): how far another implementation's
 * token is from being this draw's.  +inf for an index outside [0, V). */
static double cdf_interval_distance(const double *r, int64_t V, double Z, double w, int64_t alt) {
  if (alt < 0 || alt >= V) return INFINITY;
  double t = w * Z, C = 0.0;
  for (int64_t v = 0; v < alt; ++v) C += r[v];
  double lo = C, hi = C + r[alt];
  if (t < lo) return (lo - t) / Z;
  if (t >= hi) return (t - hi) / Z;
  return 0.0;
}

/* ------------------------------------------------------------------ */
/* speculative verification                                            */
/* ------------------------------------------------------------------ */
/*
 * target : [total_rows + N, V]; request n owns target rows cu[n] + n .. cu[n] + n + L_n
 *          (L_n + 1 rows; the last is the bonus row).
 * draft  : [total_rows, V]; request n owns draft rows cu[n] .. cu[n+1] - 1.
 * tokens : [total_rows] draft tokens x_j, drawn from softmax(draft row j / T).
 * req_ids: optional [N]; request n uses Philox request index req_ids[n]
 *          (NULL: n).  Lets a caller verify a subset of a batch with the
 *          batch's own uniforms.
 * thr_out: optional [total_rows]; acceptance threshold min(1, p/q) per
 *          position (NaN where not computed).
 * alt_next, alt_dist: optional [N] each; for request n, alt_dist[n] is the
 *          distance (a fraction of Z) from w Z to the CDF interval of token
 *          alt_next[n] in the distribution this oracle drew from (0: the
 *          same draw; at T = 0, 0 if alt_next[n] is the argmax else +inf).
 *          A test passes the GPU's tokens to check that every mismatch it
 *          excuses as near a CDF boundary really is within the band.
 * Returns 0; per-request problems are reported through flags.
 */
int oracle_spec_verify(const void *target, const void *draft, int dtype, int64_t V, int32_t N,
                       const int32_t *cu, const int32_t *tokens, double temperature, uint64_t seed,
                       int32_t max_len, const int32_t *req_ids, int32_t *accept_len,
                       int32_t *next_token, int32_t *flags, double *thr_out, const int32_t *alt_next,
                       double *alt_dist) {
  double *P = (double *)malloc(sizeof(double) * (size_t)V);
  double *Q = (double *)malloc(sizeof(double) * (size_t)V);
  double *R = (double *)malloc(sizeof(double) * (size_t)V);
  if (!P || !Q || !R) {
    free(P); free(Q); free(R);
    return -1;
  }
  for (int32_t n = 0; n < N; ++n) {
    int32_t L = cu[n + 1] - cu[n];
    int64_t trow0 = (int64_t)cu[n] + n; /* first target row of this request */
    int64_t drow0 = (int64_t)cu[n];     /* first draft row of this request  */
    uint32_t rid = req_ids ? (uint32_t)req_ids[n] : (uint32_t)n;
    flags[n] = 0;
    accept_len[n] = -1;
    next_token[n] = -1;
    if (alt_dist) alt_dist[n] = NAN;
    if (thr_out)
      for (int32_t j = 0; j < L && j >= 0; ++j) thr_out[drow0 + j] = NAN;
    if (L < 1 || L > max_len) {
      flags[n] = FLAG_BAD;
      continue;
    }
    int bad = 0;
    for (int32_t j = 0; j < L; ++j)
      if (tokens[drow0 + j] < 0 || tokens[drow0 + j] >= V) bad = 1;
    /* every row the method reads must have a softmax */
    for (int32_t j = 0; j <= L && !bad; ++j) {
      int d = row_defects(target, dtype, trow0 + j, V);
      if (temperature == 0.0 ? (d & 1) : d) bad = 1;
    }
    if (temperature > 0.0)
      for (int32_t j = 0; j < L && !bad; ++j)
        if (row_defects(draft, dtype, drow0 + j, V)) bad = 1;
    if (bad) {
      flags[n] = FLAG_BAD;
      continue;
    }

    if (temperature == 0.0) {
      /* [DF] §5.1: compare each candidate with the target argmax, left to
       * right; the first mismatch emits the target's own choice; when all
       * pass the bonus row's argmax is emitted. */
      int32_t a = L;
      for (int32_t j = 0; j < L; ++j) {
        if ((int64_t)tokens[drow0 + j] != row_argmax(target, dtype, trow0 + j, V)) {
          a = j;
          break;
        }
      }
      accept_len[n] = a;
      next_token[n] = (int32_t)row_argmax(target, dtype, trow0 + a, V);
      if (alt_dist) alt_dist[n] = (alt_next[n] == next_token[n]) ? 0.0 : INFINITY;
      continue;
    }

    /* [DF] §5.2 eq. (6): accept x_j with probability min(1, p(x_j)/q(x_j)),
     * realised as u_j < min(1, p/q) with u_j = U(seed, i, j, 0). */
    int32_t a = L;
    double thr_at[64];
    double u_at[64];
    for (int32_t j = 0; j < L; ++j) {
      row_softmax(target, dtype, trow0 + j, V, temperature, P);
      row_softmax(draft, dtype, drow0 + j, V, temperature, Q);
      int32_t x = tokens[drow0 + j];
      double thr = (Q[x] > 0.0) ? fmin(1.0, P[x] / Q[x]) : 1.0;
      double u = oracle_uniform(seed, rid, (uint32_t)j, 0u);
      if (j < 64) {
        thr_at[j] = thr;
        u_at[j] = u;
      }
      if (thr_out) thr_out[drow0 + j] = thr;
      if (!(u < thr) && a == L) a = j; /* leftmost rejection ([AR] step 4) */
    }
    accept_len[n] = a;
    for (int32_t j = 0; j < L && j <= a && j < 64; ++j)
      if (fabs(u_at[j] - thr_at[j]) < BAND) flags[n] |= FLAG_NEAR_ACCEPT;

    /* token drawn at row j* = a with w = U(seed, i, j*, 1) */
    double w = oracle_uniform(seed, rid, (uint32_t)a, 1u);
    double Z = 0.0;
    if (a < L) {
      /* [DF] §5.2 eq. (7): residual r = [p - q]_+ / Z at the rejected row */
      row_softmax(target, dtype, trow0 + a, V, temperature, P);
      row_softmax(draft, dtype, drow0 + a, V, temperature, Q);
      for (int64_t v = 0; v < V; ++v) {
        R[v] = fmax(0.0, P[v] - Q[v]);
        Z += R[v];
      }
      if (Z == 0.0) {
        /* no rejection can happen when Z = 0 (eq. (8)); only rounding gets here */
        flags[n] |= FLAG_DEGENERATE;
        for (int64_t v = 0; v < V; ++v) {
          R[v] = P[v];
          Z += R[v];
        }
      }
    } else {
      /* [DF] Algorithm 1 step 9: every candidate passed -> bonus token from
       * the target row after the last candidate */
      row_softmax(target, dtype, trow0 + L, V, temperature, P);
      for (int64_t v = 0; v < V; ++v) {
        R[v] = P[v];
        Z += R[v];
      }
    }
    int near = 0;
    next_token[n] = (int32_t)inverse_cdf(R, V, Z, w, &near);
    if (near) flags[n] |= FLAG_NEAR_CDF;
    if (alt_dist) alt_dist[n] = cdf_interval_distance(R, V, Z, w, alt_next[n]);
  }
  free(P);
  free(Q);
  free(R);
  return 0;
}

/* ------------------------------------------------------------------ */
/* top-k / top-p filtered verification (a serving variant; see above)  */
/* ------------------------------------------------------------------ */
static const double *g_sort_keys; /* logits of the row being ordered (single-threaded) */

/* raw logit descending, smaller index first among equal logits */
static int by_logit_desc(const void *a, const void *b) {
  int64_t i = *(const int64_t *)a, j = *(const int64_t *)b;
  double x = g_sort_keys[i], y = g_sort_keys[j];
  if (x > y) return -1;
  if (x < y) return 1;
  return (i < j) ? -1 : (i > j);
}

/* out[v] = filtered softmax(x_row / T): keep the first min(top_k, V) entries
 * in logit order, then the shortest prefix of those whose cumulative
 * probability reaches top_p times their total; renormalise.  *near is set
 * when the cumulative probability at the cut (or just before it) lies within
 * BAND of the threshold.  keys, order: scratch of V entries. */
static void row_filtered(const void *x, int dtype, int64_t row, int64_t V, double T, int32_t top_k, double top_p,
                         double *out, double *keys, int64_t *order, int *near) {
  row_softmax(x, dtype, row, V, T, out);
  for (int64_t v = 0; v < V; ++v) {
    keys[v] = elem(x, dtype, row, V, v);
    order[v] = v;
  }
  g_sort_keys = keys;
  qsort(order, (size_t)V, sizeof(int64_t), by_logit_desc);
  int64_t K = (top_k >= 1 && (int64_t)top_k < V) ? (int64_t)top_k : V;
  double Zk = 0.0;
  for (int64_t n = 0; n < K; ++n) Zk += out[order[n]];
  int64_t keep = K;
  if (top_p < 1.0) {
    double cum = 0.0, prev = 0.0, thr = top_p * Zk;
    for (int64_t n = 0; n < K; ++n) {
      prev = cum;
      cum += out[order[n]];
      if (cum >= thr) {
        keep = n + 1;
        if (fabs(cum - thr) < BAND * Zk || fabs(prev - thr) < BAND * Zk) *near = 1;
        break;
      }
    }
  }
  double Zf = 0.0;
  for (int64_t n = 0; n < keep; ++n) Zf += out[order[n]];
  for (int64_t n = keep; n < V; ++n) out[order[n]] = 0.0;
  for (int64_t n = 0; n < keep; ++n) out[order[n]] /= Zf;
}

/*
 * Arguments as for oracle_spec_verify, plus top_k (1..V; values <= 0 or >= V
 * keep every entry) and top_p (in (0, 1]; 1 keeps every entry of the top-k set).
 * tokens are drawn from the filtered draft distribution q'.
 */
int oracle_spec_verify_filtered(const void *target, const void *draft, int dtype, int64_t V, int32_t N,
                                const int32_t *cu, const int32_t *tokens, double temperature, int32_t top_k,
                                double top_p, uint64_t seed, int32_t max_len, const int32_t *req_ids,
                                int32_t *accept_len, int32_t *next_token, int32_t *flags) {
  if (temperature == 0.0)
    /* filtering keeps the argmax: greedy verification is unchanged */
    return oracle_spec_verify(target, draft, dtype, V, N, cu, tokens, 0.0, seed, max_len, req_ids, accept_len,
                              next_token, flags, NULL, NULL, NULL);
  double *P = (double *)malloc(sizeof(double) * (size_t)V);
  double *Q = (double *)malloc(sizeof(double) * (size_t)V);
  double *R = (double *)malloc(sizeof(double) * (size_t)V);
  double *keys = (double *)malloc(sizeof(double) * (size_t)V);
  int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)V);
  if (!P || !Q || !R || !keys || !order) {
    free(P); free(Q); free(R); free(keys); free(order);
    return -1;
  }
  for (int32_t n = 0; n < N; ++n) {
    int32_t L = cu[n + 1] - cu[n];
    int64_t trow0 = (int64_t)cu[n] + n;
    int64_t drow0 = (int64_t)cu[n];
    uint32_t rid = req_ids ? (uint32_t)req_ids[n] : (uint32_t)n;
    flags[n] = 0;
    accept_len[n] = -1;
    next_token[n] = -1;
    if (L < 1 || L > max_len) {
      flags[n] = FLAG_BAD;
      continue;
    }
    int bad = 0;
    for (int32_t j = 0; j < L; ++j)
      if (tokens[drow0 + j] < 0 || tokens[drow0 + j] >= V) bad = 1;
    for (int32_t j = 0; j <= L && !bad; ++j)
      if (row_defects(target, dtype, trow0 + j, V)) bad = 1;
    for (int32_t j = 0; j < L && !bad; ++j)
      if (row_defects(draft, dtype, drow0 + j, V)) bad = 1;
    if (bad) {
      flags[n] = FLAG_BAD;
      continue;
    }
    /* [DF] §5.2 eq. (6) with the filtered p' and q' */
    int32_t a = L;
    int near_filter = 0;
    for (int32_t j = 0; j < L && a == L; ++j) {
      int nf = 0;
      row_filtered(target, dtype, trow0 + j, V, temperature, top_k, top_p, P, keys, order, &nf);
      row_filtered(draft, dtype, drow0 + j, V, temperature, top_k, top_p, Q, keys, order, &nf);
      near_filter |= nf;
      int32_t x = tokens[drow0 + j];
      double thr = (P[x] == 0.0) ? 0.0 : ((Q[x] > 0.0) ? fmin(1.0, P[x] / Q[x]) : 1.0);
      double u = oracle_uniform(seed, rid, (uint32_t)j, 0u);
      if (fabs(u - thr) < BAND) flags[n] |= FLAG_NEAR_ACCEPT;
      if (!(u < thr)) a = j; /* leftmost rejection */
    }
    accept_len[n] = a;
    double w = oracle_uniform(seed, rid, (uint32_t)a, 1u);
    double Z = 0.0;
    int nf = 0;
    if (a < L) {
      /* eq. (7) on the filtered distributions (P, Q still hold row a) */
      for (int64_t v = 0; v < V; ++v) {
        R[v] = fmax(0.0, P[v] - Q[v]);
        Z += R[v];
      }
      if (Z == 0.0) {
        flags[n] |= FLAG_DEGENERATE;
        for (int64_t v = 0; v < V; ++v) {
          R[v] = P[v];
          Z += R[v];
        }
      }
    } else {
      row_filtered(target, dtype, trow0 + L, V, temperature, top_k, top_p, R, keys, order, &nf);
      for (int64_t v = 0; v < V; ++v) Z += R[v];
    }
    if (near_filter || nf) flags[n] |= FLAG_NEAR_FILTER;
    int near = 0;
    next_token[n] = (int32_t)inverse_cdf(R, V, Z, w, &near);
    if (near) flags[n] |= FLAG_NEAR_CDF;
  }
  free(P); free(Q); free(R); free(keys); free(order);
  return 0;
}

/* ------------------------------------------------------------------ */
/* OPD loss and its gradient with respect to the draft logits          */
/* ------------------------------------------------------------------ */
/*
 * draft row r (0 <= r < R) pairs with target row r + n(r) when has_bonus
 * (verify layout, n(r) the request owning draft row r per cu) and with
 * target row r otherwise (cu unused).
 * loss[r]     = sum_v clamp(t_v, -c, c) + lambda * CE
 *   t_v       = q_v (lq_v - lp_v),  t_v := 0 where q_v == 0
 *   CE        = -lq_{x*},  x* = argmax_v target_v (raw, smallest index)
 * dlogits[r,v]= grad_scale / T * ( q_v (a_v - S) + lambda (q_v - [v == x*]) )
 * dlogits may be NULL (loss only).  flags may be NULL.
 */
int oracle_opd_loss(const void *target, const void *draft, int dtype, int64_t V, int32_t N,
                    const int32_t *cu, int64_t R, int32_t has_bonus, double temperature,
                    double clip_c, double lambda_ce, double grad_scale, double *loss,
                    double *dlogits, int32_t *flags) {
  double *lp = (double *)malloc(sizeof(double) * (size_t)V);
  double *lq = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  double *t = (double *)malloc(sizeof(double) * (size_t)V);
  if (!lp || !lq || !q || !t) {
    free(lp); free(lq); free(q); free(t);
    return -1;
  }
  const double T = temperature, c = clip_c;
  int32_t n = 0;
  for (int64_t r = 0; r < R; ++r) {
    int64_t trow = r;
    if (has_bonus) {
      while (n + 1 <= N && cu[n + 1] <= r) ++n; /* request owning draft row r */
      trow = r + n;
    }
    int32_t fl = 0;
    if (row_defects(target, dtype, trow, V) || row_defects(draft, dtype, r, V)) {
      loss[r] = NAN;
      if (dlogits)
        for (int64_t v = 0; v < V; ++v) dlogits[r * V + v] = NAN;
      if (flags) flags[r] = FLAG_BAD;
      continue;
    }
    row_log_softmax(target, dtype, trow, V, T, lp);
    row_log_softmax(draft, dtype, r, V, T, lq);
    for (int64_t v = 0; v < V; ++v) q[v] = exp(lq[v]);

    /* [AR] Algorithm 2: per-entry term, clipped before the vocabulary sum */
    double rkl = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      t[v] = (q[v] == 0.0) ? 0.0 : q[v] * (lq[v] - lp[v]);
      double cl = t[v] < -c ? -c : (t[v] > c ? c : t[v]);
      rkl += cl;
      if (fabs(fabs(t[v]) - c) < BAND * c) fl |= FLAG_NEAR_CLIP;
    }
    /* [AR] l_hard: cross-entropy on the target's top-1 token */
    int64_t xs = row_argmax(target, dtype, trow, V);
    double ce = -lq[xs];
    loss[r] = rkl + lambda_ce * ce;
    if (flags) flags[r] = fl;

    if (dlogits) {
      /* chain rule through q = softmax(z / T); only unclipped entries pass
       * gradient (strict inequalities) */
      double S = 0.0;
      for (int64_t v = 0; v < V; ++v) {
        if (q[v] == 0.0) continue;
        double av = (t[v] > -c && t[v] < c) ? (lq[v] - lp[v] + 1.0) : 0.0;
        S += q[v] * av;
      }
      for (int64_t v = 0; v < V; ++v) {
        double qa = 0.0;
        if (q[v] != 0.0) {
          double av = (t[v] > -c && t[v] < c) ? (lq[v] - lp[v] + 1.0) : 0.0;
          qa = q[v] * av;
        }
        double g = (qa - q[v] * S) + lambda_ce * (q[v] - (v == xs ? 1.0 : 0.0));
        dlogits[r * V + v] = grad_scale / T * g;
      }
    }
  }
  free(lp);
  free(lq);
  free(q);
  free(t);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Adaptive length head ([AR] "Algorithm 3: Adaptive Length Head, Forward    */
/* Pass"; [AP] §2.2).  For each request i with hidden states h[i] (k x H):   */
/*   h'_p = SiLU(W1 h[i][p] + b1)        per position p, W1 is H' x H        */
/*   hbar = (1/k) sum_p h'_p                                                 */
/*   a_hat = sigmoid(w2 . hbar + b2)                                         */
/*   k_hat = clamp(floor(gamma a_hat k), 1, k)                               */
/* hidden and W1 are bf16 bits (dtype ORACLE_BF16) or fp32.                  */
/* ------------------------------------------------------------------------ */
static double silu(double x) { return x / (1.0 + exp(-x)); }

int oracle_length_head(const void *hidden, const void *w1, int dtype, int32_t N, int32_t k, int32_t H,
                       int32_t Hp, const float *b1, const float *w2, float b2, double gamma, double *a_hat,
                       int32_t *k_hat, int32_t *flags) {
  if (N < 0 || k < 1 || H < 1 || Hp < 1) return 1;
  double *hbar = (double *)malloc(sizeof(double) * (size_t)Hp);
  if (!hbar) return 2;
  for (int32_t i = 0; i < N; ++i) {
    for (int32_t j = 0; j < Hp; ++j) hbar[j] = 0.0;
    for (int32_t p = 0; p < k; ++p) {
      const int64_t row = (int64_t)i * k + p;
      for (int32_t j = 0; j < Hp; ++j) {
        double g = 0.0;
        for (int32_t h = 0; h < H; ++h) g += elem(w1, dtype, j, H, h) * elem(hidden, dtype, row, H, h);
        hbar[j] += silu(g + (double)b1[j]);
      }
    }
    double z = (double)b2;
    for (int32_t j = 0; j < Hp; ++j) z += (double)w2[j] * (hbar[j] / (double)k);
    const double a = 1.0 / (1.0 + exp(-z));
    const double x = gamma * a * (double)k;
    double kh = floor(x);
    if (kh < 1.0) kh = 1.0;
    if (kh > (double)k) kh = (double)k;
    a_hat[i] = a;
    k_hat[i] = (int32_t)kh;
    if (flags) {
      const double frac = x - floor(x);
      flags[i] = (frac < 1e-4 || frac > 1.0 - 1e-4) ? FLAG_NEAR_FLOOR : 0;
    }
  }
  free(hbar);
  return 0;
}

/* Length-head label and loss ([AR] "Online Update of the Length Head,
 * Derived"): a* = accept_len / L (the accepted fraction of the L verified
 * tokens of request i, L = cu[i+1] - cu[i]); loss = (a_hat - a*)^2.  A bad
 * request (accept_len < 0 or L < 1) gets a* = loss = NaN. */
int oracle_length_label(const int32_t *accept_len, const int32_t *cu, const double *a_hat, int32_t N,
                        double *a_star, double *loss) {
  for (int32_t i = 0; i < N; ++i) {
    const int32_t L = cu[i + 1] - cu[i];
    if (accept_len[i] < 0 || L < 1) {
      a_star[i] = NAN;
      loss[i] = NAN;
      continue;
    }
    a_star[i] = (double)accept_len[i] / (double)L;
    const double d = a_hat[i] - a_star[i];
    loss[i] = d * d;
  }
  return 0;
}
