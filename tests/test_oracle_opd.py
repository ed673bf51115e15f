"""Pins for the oracle's OPD loss and gradient (CPU only).

Each test ties the oracle to something other than itself: the review's worked
example, hand-derived clip values from that example's printed terms, central
finite differences of the oracle's own loss, and exact invariants of the
softmax gradient.
"""
import numpy as np
import pytest
from scipy.special import log_softmax

import oracle
from conftest import read_golden


def _golden_example():
    g = {r[0]: [float(x) for x in r[1:]] for r in read_golden("opd_worked_example.txt")}
    q = np.array(g["q"])
    p = np.array(g["p"])
    return g, np.log(p).astype(np.float32)[None, :], np.log(q).astype(np.float32)[None, :]


def test_worked_example_unclipped():
    g, y, z = _golden_example()
    # no clipping (c above every term), lambda = 0 -> the reverse KL alone
    rkl = oracle.opd_loss(y, z, clip_c=10.0, lambda_ce=0.0, want_grad=False)["loss"][0]
    assert abs(rkl - g["l_rkl"][0]) < 5e-4
    # lambda = 1 adds exactly the hard-label CE on the target top-1 token (A)
    both = oracle.opd_loss(y, z, clip_c=10.0, lambda_ce=1.0, want_grad=False)["loss"][0]
    assert abs((both - rkl) - g["l_hard"][0]) < 5e-4
    # the review's mixture alpha*l_hard + (1-alpha)*l_rkl equals
    # (1-alpha) * (rkl + lambda*CE) with lambda = alpha / (1 - alpha)
    a = g["alpha"][0]
    mix = oracle.opd_loss(y, z, clip_c=10.0, lambda_ce=a / (1 - a), want_grad=False)["loss"][0]
    assert abs((1 - a) * mix - g["l_opd"][0]) < 5e-4


@pytest.mark.parametrize("c", [0.01, 0.05, 0.09, 0.1, 0.2, 0.3])
def test_worked_example_entrywise_clamp(c):
    """Clamp each printed per-entry term to [-c, c] by hand, then sum."""
    g, y, z = _golden_example()
    expected = sum(min(max(t, -c), c) for t in g["term"])
    got = oracle.opd_loss(y, z, clip_c=c, lambda_ce=0.0, want_grad=False)["loss"][0]
    # printed terms carry 3 decimals: 4 terms x 5e-4
    assert abs(got - expected) < 2e-3, (c, got, expected)


def test_clamp_reading_differs_from_one_sided_min_at_small_c():
    """At c = 0.01 the two-sided clamp gives 0.02 while the review's one-sided
    min(term, delta) would give -0.176: the oracle implements the clamp."""
    _, y, z = _golden_example()
    got = oracle.opd_loss(y, z, clip_c=0.01, lambda_ce=0.0, want_grad=False)["loss"][0]
    assert abs(got - 0.02) < 1e-9
    assert abs(got - (-0.176)) > 0.1


def _grid_logits(rng, shape, sd):
    # logits on a 2^-12 grid: exact in float32, and so are +/- 2^-10 steps
    return (np.round(rng.normal(0.0, sd, size=shape) * 4096.0) / 4096.0).astype(np.float32)


def _terms(y, z, T):
    lp = log_softmax(y.astype(np.float64) / T, axis=-1)
    lq = log_softmax(z.astype(np.float64) / T, axis=-1)
    return np.exp(lq) * (lq - lp)


@pytest.mark.parametrize("T,c,lam", [(1.0, 1e9, 0.1), (0.7, 1e9, 0.5), (1.0, 0.02, 0.1),
                                     (1.3, 0.05, 0.0)])
def test_gradient_matches_central_differences(T, c, lam):
    rng = np.random.default_rng(7)
    R, V = 6, 24
    y = _grid_logits(rng, (R, V), 2.0)
    z = _grid_logits(rng, (R, V), 2.0)
    h = 2.0 ** -10
    gs = 0.25
    out = oracle.opd_loss(y, z, temperature=T, clip_c=c, lambda_ce=lam, grad_scale=gs)
    g = out["dlogits"]
    fd = np.zeros_like(g)
    for v in range(V):
        zp = z.copy(); zp[:, v] += h
        zm = z.copy(); zm[:, v] -= h
        # no entry's clamp decision may flip inside the step
        for zz in (zp, zm):
            same = (np.abs(_terms(y, zz, T)) < c) == (np.abs(_terms(y, z, T)) < c)
            assert same.all(), "finite-difference step crosses a clip boundary"
        lp_ = oracle.opd_loss(y, zp, temperature=T, clip_c=c, lambda_ce=lam, want_grad=False)["loss"]
        lm_ = oracle.opd_loss(y, zm, temperature=T, clip_c=c, lambda_ce=lam, want_grad=False)["loss"]
        fd[:, v] = gs * (lp_ - lm_) / (2 * h)
    scale = np.abs(g).max(axis=1, keepdims=True)
    assert np.all(np.abs(g - fd) <= 1e-5 * scale + 1e-9), np.abs(g - fd).max()
    if c < 1e8:
        assert (np.abs(_terms(y, z, T)) >= c).any(), "case meant to exercise clipping"


def test_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(3)
    y = rng.normal(0, 3, size=(8, 300)).astype(np.float32)
    z = (0.7 * y + rng.normal(0, 2, size=y.shape)).astype(np.float32)
    for c in (1.0, 0.01, 1e9):
        g = oracle.opd_loss(y, z, clip_c=c, lambda_ce=0.3)["dlogits"]
        assert np.all(np.abs(g.sum(axis=1)) < 1e-12 * 300 + 1e-14)


def test_equal_distributions():
    """p == q: every reverse-KL term is 0, so the loss is lambda*CE and the
    gradient is lambda (q - e_{x*}) / T."""
    rng = np.random.default_rng(5)
    y = rng.normal(0, 2, size=(3, 50)).astype(np.float32)
    T, lam = 0.8, 0.3
    out = oracle.opd_loss(y, y, temperature=T, clip_c=0.5, lambda_ce=lam)
    lq = log_softmax(y.astype(np.float64) / T, axis=-1)
    xs = np.argmax(y, axis=1)
    ce = -lq[np.arange(3), xs]
    assert np.allclose(out["loss"], lam * ce, rtol=1e-12, atol=1e-14)
    exp_g = lam * np.exp(lq)
    exp_g[np.arange(3), xs] -= lam
    assert np.allclose(out["dlogits"], exp_g / T, rtol=1e-10, atol=1e-15)


def test_top1_tie_takes_smallest_index():
    y = np.array([[0.0, 2.0, 2.0, 1.0]], dtype=np.float32)
    z = np.array([[0.5, -1.0, 3.0, 0.0]], dtype=np.float32)
    out = oracle.opd_loss(y, z, clip_c=10.0, lambda_ce=1.0)
    lq = log_softmax(z.astype(np.float64), axis=-1)[0]
    rkl = oracle.opd_loss(y, z, clip_c=10.0, lambda_ce=0.0, want_grad=False)["loss"][0]
    assert abs(out["loss"][0] - rkl - (-lq[1])) < 1e-12   # x* = 1, not 2


def test_verify_layout_pairing():
    """has_bonus: draft row r pairs with target row r + (request of r)."""
    rng = np.random.default_rng(11)
    cu = np.array([0, 2, 5], dtype=np.int32)
    y = rng.normal(0, 2, size=(7, 16)).astype(np.float32)
    z = rng.normal(0, 2, size=(5, 16)).astype(np.float32)
    got = oracle.opd_loss(y, z, cu_draft=cu, has_bonus=True)
    pair = np.array([0, 1, 3, 4, 5])
    ref = oracle.opd_loss(y[pair], z)
    assert np.array_equal(got["loss"], ref["loss"])
    assert np.array_equal(got["dlogits"], ref["dlogits"])


def test_bad_rows_are_flagged():
    y = np.zeros((3, 8), dtype=np.float32)
    z = np.zeros((3, 8), dtype=np.float32)
    y[1, 3] = np.nan
    z[2, :] = -np.inf
    out = oracle.opd_loss(y, z)
    assert out["flags"][0] == 0 and np.isfinite(out["loss"][0])
    assert out["flags"][1] & oracle.FLAG_BAD and np.isnan(out["loss"][1])
    assert out["flags"][2] & oracle.FLAG_BAD


def test_masked_entries():
    """-inf draft logits have q = 0: their term is 0 and their gradient is 0;
    -inf target logits under q > 0 give an infinite term, clamped to c."""
    y = np.array([[1.0, 0.5, -np.inf, 0.0]], dtype=np.float32)
    z = np.array([[0.0, -np.inf, 0.3, 1.0]], dtype=np.float32)
    out = oracle.opd_loss(y, z, clip_c=0.25, lambda_ce=0.0)
    lq = log_softmax(z.astype(np.float64), axis=-1)[0]
    lp = log_softmax(y.astype(np.float64), axis=-1)[0]
    q = np.exp(lq)
    t0 = q[0] * (lq[0] - lp[0]); t3 = q[3] * (lq[3] - lp[3])
    exp = np.clip(t0, -0.25, 0.25) + 0.0 + 0.25 + np.clip(t3, -0.25, 0.25)
    assert abs(out["loss"][0] - exp) < 1e-12
    assert out["dlogits"][0, 1] == 0.0
