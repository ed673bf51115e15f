"""Pins for the oracle's top-k / top-p filtered verification.

Filtering is not on the pages; the reading (stated in the oracle's header):
both distributions are filtered with the same (T, top_k, top_p) -- order by
raw logit descending, smaller index first among equal logits, keep the first
top_k, then the shortest prefix whose cumulative probability reaches top_p of
their total, renormalise -- and the verification of "DFlash 阅读笔记：并行起草、
目标特征与精确验证" §5.2 eqs. (6)-(8) / Algorithm 1 runs on the filtered p' and q'.

Each pin comes from something other than the oracle's own formula: special
cases that reduce to the pinned unfiltered and greedy routines, hand-computed
filtered distributions checked draw by draw against the uniforms, tie cases,
and the losslessness of eq. (8) (the emitted token is distributed as p').
"""
import math

import numpy as np
from scipy.stats import chisquare

import oracle
import synth


def _lg(p):
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


def test_no_filter_is_the_unfiltered_method():
    for b, T in ((synth.config(1), 1.0),
                 (synth.make_batch("nf", seed=3, lengths=np.array([3, 1, 7, 16], np.int32), V=300, dtype="bf16",
                                   target_sd=2.0, sigma_req=np.array([0.5, 1.0, 2.0, 3.0]), temperatures=(0.6,)),
                  0.6)):
        ref = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[T], T, 5)
        for k in (b.V, 0, 10 ** 9):
            got = oracle.spec_verify_filtered(b.target, b.draft, b.cu, b.tokens[T], T, k, 1.0, 5)
            assert np.array_equal(got["accept_len"], ref["accept_len"])
            assert np.array_equal(got["next_token"], ref["next_token"])


def test_top1_is_greedy_verification():
    """top_k = 1 makes p' and q' one-hot at the argmaxes: a drafted token (the
    draft argmax) passes iff it is the target argmax, and the emitted token is
    the target argmax -- greedy verification ([DF] §5.1)."""
    b = synth.make_batch("t1", seed=4, lengths=np.array([4, 2, 8, 1, 5], np.int32), V=64, dtype="f32",
                         target_sd=1.5, sigma_req=np.array([0.3, 0.5, 1.0, 0.2, 0.4]), temperatures=(1.0,))
    tok = synth.sample_tokens(b.draft, 0.0, 1)  # the draft argmax of every row
    ref = oracle.spec_verify(b.target, b.draft, b.cu, tok, 0.0, 9)
    for T in (1.0, 0.5):
        got = oracle.spec_verify_filtered(b.target, b.draft, b.cu, tok, T, 1, 1.0, 9)
        assert np.array_equal(got["accept_len"], ref["accept_len"])
        assert np.array_equal(got["next_token"], ref["next_token"])


def _bonus_batch(logits, n):
    """n one-position requests whose draft equals the target (p' = q': every
    token passes) and whose bonus row holds `logits`; tokens = argmax."""
    V = len(logits)
    row = np.asarray(logits, np.float32)
    tgt = np.ascontiguousarray(np.broadcast_to(row, (n, 2, V)).reshape(-1, V))
    drf = np.ascontiguousarray(np.broadcast_to(row, (n, V)))
    cu = synth.cu_from_lengths(np.ones(n, np.int32))
    tok = np.full(n, int(np.argmax(row)), np.int32)
    return tgt, drf, cu, tok


def _check_draws(logits, top_k, top_p, kept_probs, n=3000, seed=11):
    """Every request's bonus draw against the hand-computed filtered CDF and
    its own uniform w = U(seed, i, 1, 1)."""
    tgt, drf, cu, tok = _bonus_batch(logits, n)
    got = oracle.spec_verify_filtered(tgt, drf, cu, tok, 1.0, top_k, top_p, seed)
    assert np.all(got["accept_len"] == 1)
    C = np.cumsum(kept_probs)
    checked = 0
    for i in range(n):
        w = oracle.uniform(seed, i, 1, 1)
        if np.min(np.abs(C - w)) < 1e-6:
            continue
        assert got["next_token"][i] == int(np.searchsorted(C, w, side="right")), (i, w)
        checked += 1
    assert checked > 0.99 * n


def test_hand_example_top_p():
    """p = (0.5, 0.3, 0.15, 0.05): top_p = 0.7 keeps the first two (0.8 >= 0.7)
    -> p' = (0.625, 0.375, 0, 0); top_p = 0.8 still two (cumulative 0.8 reaches
    it only in exact arithmetic, so use 0.79); top_p = 0.81 keeps three."""
    lg = _lg([0.5, 0.3, 0.15, 0.05])
    _check_draws(lg, 4, 0.7, [0.625, 0.375])
    _check_draws(lg, 4, 0.79, [0.625, 0.375])
    _check_draws(lg, 4, 0.81, [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95])
    _check_draws(lg, 4, 0.3, [1.0])          # the first entry alone reaches 0.3
    _check_draws(lg, 4, 0.7995, [0.625, 0.375])  # reached, not exceeded by much: still two


def test_hand_example_top_k_then_top_p():
    """top_k = 3 first (mass 0.95), then top_p of that: 0.8 * 0.95 = 0.76 is
    reached by the first two (0.8)."""
    lg = _lg([0.05, 0.5, 0.15, 0.3])        # the order is by logit, not index
    _check_draws(lg, 3, 1.0, [0, 0.5 / 0.95, 0.15 / 0.95, 0.3 / 0.95])
    _check_draws(lg, 3, 0.8, [0, 0.625, 0, 0.375])
    _check_draws(lg, 2, 1.0, [0, 0.625, 0, 0.375])
    # top_p is a fraction of the top-k mass: 0.82 * 0.95 = 0.779 is reached by
    # the first two (0.8), although 0.82 of the whole row would need three
    _check_draws(lg, 3, 0.82, [0, 0.625, 0, 0.375])


def test_ties_keep_the_smaller_index():
    lg = np.array([1.0, 3.0, 3.0, 3.0, 0.0], np.float32)
    _check_draws(lg, 2, 1.0, [0, 0.5, 0.5])
    _check_draws(lg, 1, 1.0, [0, 1.0])


def test_token_outside_the_target_set_is_rejected():
    """A drafted token the target's filter drops has p'(x) = 0: rejected for
    every uniform, and the residual is p' itself (q' vanishes on it)."""
    V = 6
    y = _lg([0.4, 0.3, 0.2, 0.06, 0.03, 0.01])
    z = _lg([0.01, 0.03, 0.06, 0.2, 0.3, 0.4])
    n = 500
    tgt = np.ascontiguousarray(np.broadcast_to(y, (n, 2, V)).reshape(-1, V))
    drf = np.ascontiguousarray(np.broadcast_to(z, (n, V)))
    cu = synth.cu_from_lengths(np.ones(n, np.int32))
    tok = np.full(n, 5, np.int32)  # kept by the draft's top-2, dropped by the target's
    got = oracle.spec_verify_filtered(tgt, drf, cu, tok, 1.0, 2, 1.0, 3)
    assert np.all(got["accept_len"] == 0)
    assert set(np.unique(got["next_token"]).tolist()) <= {0, 1}


def _filtered(y, T, k, p):
    """Test-side filter, written independently, used to draw the tokens."""
    order = sorted(range(len(y)), key=lambda v: (-float(y[v]), v))
    e = np.exp((np.asarray(y, np.float64) - float(np.max(y))) / T)
    e /= e.sum()
    kept = order[:k]
    tot = sum(e[v] for v in kept)
    c, keep = 0.0, []
    for v in kept:
        keep.append(v)
        c += e[v]
        if c >= p * tot:
            break
    out = np.zeros(len(y))
    out[keep] = e[keep] / sum(e[v] for v in keep)
    return out


def test_lossless_chisquare_filtered():
    """[DF] §5.2 eq. (8) with the filtered distributions: the first emitted
    token (the accepted draft token, else the residual draw) is distributed as
    the filtered target p'."""
    rng = np.random.default_rng(21)
    V, n, T, k, p = 8, 200_000, 0.9, 5, 0.85
    y = rng.normal(0, 1.5, size=V).astype(np.float32)
    z = (y + rng.normal(0, 1.0, size=V)).astype(np.float32)
    pf, qf = _filtered(y, T, k, p), _filtered(z, T, k, p)
    tgt = np.ascontiguousarray(np.broadcast_to(np.stack([y, y]), (n, 2, V)).reshape(-1, V))
    drf = np.ascontiguousarray(np.broadcast_to(z, (n, V)))
    cu = synth.cu_from_lengths(np.ones(n, np.int32))
    tok = rng.choice(V, size=n, p=qf).astype(np.int32)
    got = oracle.spec_verify_filtered(tgt, drf, cu, tok, T, k, p, 17)
    first = np.where(got["accept_len"] >= 1, tok, got["next_token"])
    expect = pf * n
    m = expect > 0
    assert np.all(np.bincount(first, minlength=V)[~m] == 0)
    assert chisquare(np.bincount(first, minlength=V)[m], expect[m]).pvalue > 1e-4
    # and the acceptance rate is sum_v min(p'_v, q'_v) (eq. (6) summed over x ~ q')
    rate = float(np.mean(got["accept_len"] >= 1))
    assert abs(rate - float(np.minimum(pf, qf).sum())) < 5 * math.sqrt(0.25 / n)


def test_greedy_unchanged_by_filters():
    b = synth.make_batch("g", seed=8, lengths=np.array([3, 6, 2], np.int32), V=500, dtype="bf16",
                         sigma_req=np.ones(3), temperatures=(0.0,))
    ref = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[0.0], 0.0, 2)
    got = oracle.spec_verify_filtered(b.target, b.draft, b.cu, b.tokens[0.0], 0.0, 3, 0.5, 2)
    assert np.array_equal(got["accept_len"], ref["accept_len"])
    assert np.array_equal(got["next_token"], ref["next_token"])
