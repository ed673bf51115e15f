"""Pins for the oracle's speculative verification (CPU only).

Each test ties the oracle to a fact fixed by the pages or by mathematics, not
to a retyping of its own code:
  * losslessness (eq. (8) of the DFlash notes): the first emitted token is
    distributed as p -- chi-square over 10^6 seeded requests at V = 8;
  * the law of (accepted length, next token) from brute-force enumeration of
    every draft sequence (V <= 4, L <= 3);
  * E[tau] = (1 - a^(m+1)) / (1 - a) on rows built with sum_v min(p, q) = a,
    against the values the DFlash notes print (4.86, 8.15);
  * the residual example after eq. (8): every rejection emits the one token
    that carries the missing mass;
  * the greedy rule with ties, and invalid inputs.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chisquare

import oracle
import synth
from conftest import read_golden


def _uniform_batch(y_rows, z_rows, n_req, T, seed):
    """n_req identical requests: request rows y_rows (L+1) / z_rows (L);
    draft tokens drawn independently per request from softmax(z/T)."""
    L = z_rows.shape[0]
    tgt = np.ascontiguousarray(np.broadcast_to(y_rows, (n_req, L + 1, y_rows.shape[1]))
                               .reshape(-1, y_rows.shape[1]))
    drf = np.ascontiguousarray(np.broadcast_to(z_rows, (n_req, L, z_rows.shape[1]))
                               .reshape(-1, z_rows.shape[1]))
    cu = synth.cu_from_lengths(np.full(n_req, L))
    tok = synth.sample_tokens(drf, T, seed)
    return tgt, drf, cu, tok


def _emitted(acc, nxt, tok, cu, k):
    """k-th emitted token of each request (k < L + 1)."""
    out = np.where(acc > k, tok[cu[:-1] + np.minimum(k, np.diff(cu) - 1)], nxt)
    return out, acc >= k  # defined only when the first k tokens were accepted


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_lossless_first_token_chisquare(T):
    rng = np.random.default_rng(2024)
    V = 8
    y = rng.normal(0, 1.5, size=(2, V)).astype(np.float32)
    z = (y[:1] + rng.normal(0, 1.0, size=(1, V))).astype(np.float32)
    n = 1_000_000
    tgt, drf, cu, tok = _uniform_batch(y, z, n, T, seed=91)
    r = oracle.spec_verify(tgt, drf, cu, tok, T, seed=5)
    first, _ = _emitted(r["accept_len"], r["next_token"], tok, cu, 0)
    p0 = softmax(y[0].astype(np.float64) / T)
    obs = np.bincount(first, minlength=V)
    assert chisquare(obs, p0 * n).pvalue > 1e-4
    # the draft alone is far from p: the test has power
    q0 = softmax(z[0].astype(np.float64) / T)
    assert chisquare(obs, q0 * n).pvalue < 1e-12
    # second token when the first was accepted comes from the bonus row
    second = r["next_token"][r["accept_len"] == 1]
    p1 = softmax(y[1].astype(np.float64) / T)
    obs2 = np.bincount(second, minlength=V)
    assert chisquare(obs2, p1 * obs2.sum()).pvalue > 1e-4


def _enumerate_law(P, Q, Pbonus):
    """Exact joint law of (accepted length A, next token) by enumerating every
    draft sequence x in V^L with weight prod_j Q_j(x_j)."""
    L, V = Q.shape
    law = np.zeros((L + 1, V))
    for xs in itertools.product(range(V), repeat=L):
        w = np.prod([Q[j, x] for j, x in enumerate(xs)])
        if w == 0.0:
            continue
        alive = 1.0
        for j, x in enumerate(xs):
            acc = min(1.0, P[j, x] / Q[j, x])
            rej = alive * (1.0 - acc)
            if rej > 0:
                resid = np.maximum(P[j] - Q[j], 0.0)
                law[j] += w * rej * resid / resid.sum()
            alive *= acc
        law[L] += w * alive * Pbonus
    return law


@pytest.mark.parametrize("V,L,T", [(3, 1, 1.0), (4, 2, 1.0), (3, 3, 0.7), (4, 3, 1.0)])
def test_brute_force_joint_law(V, L, T):
    rng = np.random.default_rng(100 + 10 * V + L)
    y = rng.normal(0, 1.2, size=(L + 1, V)).astype(np.float32)
    z = rng.normal(0, 1.2, size=(L, V)).astype(np.float32)
    P = softmax(y.astype(np.float64) / T, axis=1)
    Q = softmax(z.astype(np.float64) / T, axis=1)
    law = _enumerate_law(P[:L], Q, P[L])
    assert abs(law.sum() - 1.0) < 1e-12
    n = 400_000
    tgt, drf, cu, tok = _uniform_batch(y, z, n, T, seed=17)
    r = oracle.spec_verify(tgt, drf, cu, tok, T, seed=3)
    A, nx = r["accept_len"], r["next_token"]
    obs = np.zeros((L + 1, V))
    np.add.at(obs, (A, nx), 1)
    exp = law * n
    keep = exp.ravel() > 0
    assert obs.ravel()[~keep].sum() == 0, "an impossible outcome was produced"
    assert chisquare(obs.ravel()[keep], exp.ravel()[keep]).pvalue > 1e-4
    # marginal of the first emitted token equals p_0
    first_tok, _ = _emitted(A, nx, tok, cu, 0)
    cnt = np.bincount(first_tok, minlength=V)
    assert chisquare(cnt, P[0] * n).pvalue > 1e-4


def _rows_with_overlap(rng, a, V, L):
    """Target rows p_j and draft rows q_j = a p_j + (1-a) delta_w with p_w = 0,
    so that sum_v min(p_j, q_j) = a at every position."""
    w = V - 1
    y = np.empty((L + 1, V), np.float32)
    z = np.empty((L, V), np.float32)
    for j in range(L + 1):
        yy = rng.normal(0, 1.0, size=V)
        yy[w] = -1e4                       # p_w underflows to exactly 0
        y[j] = yy
    for j in range(L):
        p = softmax(y[j].astype(np.float64))
        q = a * p
        q[w] = 1.0 - a
        z[j] = np.log(q)
    return y, z


@pytest.mark.parametrize("m,a", [(15, 0.8), (15, 0.9), (16, 0.8), (16, 0.9)])
def test_expected_tau_closed_form(m, a):
    printed = {(int(r[0]), float(r[1])): float(r[2]) for r in read_golden("expected_tau.txt")}
    closed = (1 - a ** (m + 1)) / (1 - a)
    if (m, a) in printed:
        assert abs(closed - printed[(m, a)]) < 5e-3
    rng = np.random.default_rng(int(a * 100) + m)
    V = 12
    y, z = _rows_with_overlap(rng, a, V, m)
    n = 60_000
    tgt, drf, cu, tok = _uniform_batch(y, z, n, 1.0, seed=m)
    r = oracle.spec_verify(tgt, drf, cu, tok, 1.0, seed=42)
    tau = r["accept_len"].astype(np.float64) + 1.0
    se = tau.std(ddof=1) / np.sqrt(n)
    assert abs(tau.mean() - closed) < 4 * se, (tau.mean(), closed, se)
    # prefix-survival identity (eq. (2)): E[A + 1] = 1 + sum_k Pr(A >= k)
    A = r["accept_len"]
    surv = sum((A >= k).mean() for k in range(1, m + 1))
    assert abs(tau.mean() - (1.0 + surv)) < 1e-9


def test_residual_example_always_corrects_to_A():
    rows = read_golden("figure3_residual.txt")
    p = np.array([float(r[1]) for r in rows])
    q = np.array([float(r[2]) for r in rows])
    assert abs(np.minimum(p, q).sum() - 0.7) < 1e-12
    y = np.log(np.stack([p, p])).astype(np.float32)
    z = np.log(q)[None, :].astype(np.float32)
    n = 200_000
    tgt, drf, cu, tok = _uniform_batch(y, z, n, 1.0, seed=8)
    r = oracle.spec_verify(tgt, drf, cu, tok, 1.0, seed=1)
    rej = r["accept_len"] == 0
    assert rej.sum() > 0.25 * n
    assert np.all(r["next_token"][rej] == 0)
    # and the rejection rate is the missing mass 0.3
    assert abs(rej.mean() - 0.3) < 5 * np.sqrt(0.21 / n)


def test_greedy_rule_with_ties():
    # request 0: rows 0..2 target, argmax ties resolved to the smallest index
    y = np.array([[1, 3, 3, 2],      # argmax 1
                  [5, 0, 5, 5],      # argmax 0
                  [0, 0, 0, 0],      # bonus: argmax 0
                  [2, 1, 7, 7],      # request 1 row 0: argmax 2
                  [9, 9, 1, 1]],     # request 1 bonus: argmax 0
                 dtype=np.float32)
    z = np.zeros((3, 4), np.float32)
    cu = np.array([0, 2, 3], np.int32)
    tok = np.array([1, 0, 3], np.int32)
    r = oracle.spec_verify(y, z, cu, tok, 0.0, seed=0)
    assert list(r["accept_len"]) == [2, 0]
    assert list(r["next_token"]) == [0, 2]
    tok2 = np.array([1, 2, 2], np.int32)   # request 0 rejects at j=1 (2 != 0)
    r = oracle.spec_verify(y, z, cu, tok2, 0.0, seed=0)
    assert list(r["accept_len"]) == [1, 1]
    assert list(r["next_token"]) == [0, 0]


def test_greedy_ignores_draft_logits_and_uniforms():
    b = synth.config(5, N=6, V=2000)
    tok = b.tokens[0.0]
    r1 = oracle.spec_verify(b.target, b.draft, b.cu, tok, 0.0, seed=1)
    r2 = oracle.spec_verify(b.target, b.draft[::-1].copy(), b.cu, tok, 0.0, seed=99)
    assert np.array_equal(r1["accept_len"], r2["accept_len"])
    assert np.array_equal(r1["next_token"], r2["next_token"])


def test_identical_distributions_accept_everything():
    rng = np.random.default_rng(4)
    y = rng.normal(0, 2, size=(4, 40)).astype(np.float32)
    z = y[:3].copy()
    tgt, drf, cu, tok = _uniform_batch(y, z, 2000, 1.0, seed=2)
    r = oracle.spec_verify(tgt, drf, cu, tok, 1.0, seed=0)
    assert np.all(r["accept_len"] == 3)  # min(1, p/q) = 1 everywhere


def test_uniform_keying():
    """Different requests, positions and streams draw different uniforms; the
    same key gives the same value; the value is a 24-bit dyadic in [0, 1)."""
    vals = {(i, j, s): oracle.uniform(0, i, j, s) for i in range(4) for j in range(4)
            for s in range(2)}
    assert len(set(vals.values())) == len(vals)
    for v in vals.values():
        assert 0.0 <= v < 1.0 and (v * 2 ** 24) == int(v * 2 ** 24)
    assert oracle.uniform(0, 1, 2, 1) == vals[(1, 2, 1)]
    assert oracle.uniform(1 << 32, 1, 2, 1) != vals[(1, 2, 1)]  # high seed word is keyed


def test_philox_statistics():
    words = np.array([oracle.philox4x32_10([i, 7, 1, 0], [123, 456]) for i in range(20000)],
                     dtype=np.uint64)
    # each output word uniform over 64 bins
    for k in range(4):
        cnt = np.bincount((words[:, k] >> 26).astype(np.int64), minlength=64)
        assert chisquare(cnt).pvalue > 1e-4
    # avalanche: flipping one counter bit flips about half the 128 output bits
    base = oracle.philox4x32_10([5, 6, 7, 8], [1, 2])
    flips = []
    for bit in range(32):
        o = oracle.philox4x32_10([5 ^ (1 << bit), 6, 7, 8], [1, 2])
        flips.append(sum(bin(int(a) ^ int(b)).count("1") for a, b in zip(base, o)))
    assert 54 < np.mean(flips) < 74


def test_invalid_requests_are_flagged():
    y = np.zeros((9, 5), np.float32)
    z = np.zeros((6, 5), np.float32)
    cu = np.array([0, 2, 4, 6], np.int32)
    tok = np.array([0, 1, 7, 0, 1, 2], np.int32)    # request 1 holds token 7 >= V
    y[7, 2] = np.nan                                 # request 2, target row 1
    r = oracle.spec_verify(y, z, cu, tok, 1.0, seed=0)
    assert r["flags"][0] == 0 and r["accept_len"][0] >= 0
    assert r["flags"][1] & oracle.FLAG_BAD and r["accept_len"][1] == -1
    assert r["flags"][2] & oracle.FLAG_BAD and r["accept_len"][2] == -1
    r = oracle.spec_verify(y, z, cu, tok, 1.0, seed=0, max_len=1)  # L = 2 > max_len
    assert np.all(r["flags"] & oracle.FLAG_BAD)


def test_threaded_whole_batch_oracle_matches_one_call():
    """The test helper that runs the oracle's requests on host threads (for
    whole-batch GPU parity) returns exactly what one call over the batch does."""
    from helpers import _groups, compare_opd_all, oracle_verify_all
    b = synth.config(5, N=21, V=2048, seed=99)
    for T in (1.0, 0.0):
        one = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[float(T)], T, b.seed)
        many = oracle_verify_all(b, T)
        for k in ("accept_len", "next_token", "flags"):
            assert np.array_equal(one[k], many[k]), k
    ref = oracle.opd_loss(b.target, b.draft, cu_draft=b.cu, has_bonus=True)
    assert compare_opd_all(b, ref["loss"].astype(np.float32), ref["dlogits"].astype(np.float32)) >= 0
    assert sum(e - a for a, e in _groups(21, 64)) == 21


def test_cdf_interval_distance_of_another_token():
    """The oracle's alt_dist output (used to check every mismatch a GPU test
    excuses as near a CDF boundary): for each candidate token, the distance
    from w Z to that token's interval [C_{v-1}, C_v) of the distribution the
    draw used, recomputed here in fp64 from the residual [p - q]_+ ([DF] §5.2
    eq. (7)) or the bonus row."""
    V, T = 7, 1.0
    b = synth.make_batch("alt", seed=5, lengths=np.array([3, 2, 4], np.int32), V=V, dtype="f32",
                         sigma_req=[1.5, 0.3, 2.0], temperatures=(T,))
    base = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[T], T, b.seed)

    def softmax(x):
        e = np.exp(x.astype(np.float64) / T - (x.astype(np.float64) / T).max())
        return e / e.sum()

    for alt_tok in range(-1, V + 1):
        alt = np.full(b.N, alt_tok, np.int32)
        r = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[T], T, b.seed, alt_next=alt)
        assert np.array_equal(r["next_token"], base["next_token"])
        for n in range(b.N):
            L, a = int(b.cu[n + 1] - b.cu[n]), int(base["accept_len"][n])
            t0, d0 = int(b.cu[n]) + n, int(b.cu[n])
            p = softmax(b.target[t0 + a])
            w = oracle.uniform(b.seed, n, a, 1)
            rr = np.maximum(0.0, p - softmax(b.draft[d0 + a])) if a < L else p
            Z = rr.sum()
            if not 0 <= alt_tok < V:
                assert np.isinf(r["alt_dist"][n])
                continue
            lo, hi = rr[:alt_tok].sum(), rr[:alt_tok + 1].sum()
            want = (lo - w * Z) / Z if w * Z < lo else ((w * Z - hi) / Z if w * Z >= hi else 0.0)
            assert abs(r["alt_dist"][n] - want) < 1e-12, (n, alt_tok)
            assert (r["alt_dist"][n] == 0.0) == (alt_tok == base["next_token"][n])
    # greedy: 0 for the argmax, +inf for anything else
    g = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[T], 0.0, b.seed)
    r = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[T], 0.0, b.seed, alt_next=g["next_token"])
    assert np.all(r["alt_dist"] == 0.0)
    r = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[T], 0.0, b.seed, alt_next=(g["next_token"] + 1) % V)
    assert np.all(np.isinf(r["alt_dist"]))
