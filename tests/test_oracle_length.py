"""Pins for the oracle's adaptive length head ("AdaFlash: Taming Variance in
Diffusion Speculative Decoding", "Algorithm 3: Adaptive Length Head, Forward
Pass" and "Online Update of the Length Head, Derived"; "AdaFlash：基于在策略
蒸馏扩散草稿器的自适应投机解码" §2.2).

Each pin comes from something other than the oracle's own formula: values
that follow by hand from special weights, identities of SiLU and the mean,
and the clamp's two ends.
"""
import math

import numpy as np

import oracle


def _head(hidden, w1, b1, w2, b2, gamma=1.0):
    return oracle.length_head(np.asarray(hidden, np.float32), np.asarray(w1, np.float32),
                              np.asarray(b1, np.float32), np.asarray(w2, np.float32), b2, gamma)


def test_zero_weights_give_the_bias_rate():
    """W1 = 0, b1 = 0: SiLU(0) = 0, so a_hat = sigmoid(b2): 1/2 at b2 = 0 and
    3/4 at b2 = ln 3; k_hat = floor(gamma a_hat k) by hand."""
    N, k, H, Hp = 2, 16, 8, 4
    h = np.random.default_rng(0).normal(size=(N, k, H))
    r = _head(h, np.zeros((Hp, H)), np.zeros(Hp), np.ones(Hp), 0.0, gamma=1.1)
    assert np.all(r["a_hat"] == 0.5)
    assert np.all(r["k_hat"] == 8)          # floor(1.1 * 0.5 * 16) = floor(8.8)
    r = _head(h, np.zeros((Hp, H)), np.zeros(Hp), np.ones(Hp), math.log(3.0), gamma=1.1)
    assert np.allclose(r["a_hat"], 0.75, atol=1e-15)
    assert np.all(r["k_hat"] == 13)         # floor(1.1 * 0.75 * 16) = floor(13.2)


def test_clamp_at_both_ends():
    N, k, H, Hp = 1, 16, 4, 2
    h = np.ones((N, k, H))
    lo = _head(h, np.zeros((Hp, H)), np.zeros(Hp), np.zeros(Hp), -30.0)
    assert lo["a_hat"][0] < 1e-12 and lo["k_hat"][0] == 1          # at least one position
    hi = _head(h, np.zeros((Hp, H)), np.zeros(Hp), np.zeros(Hp), math.log(3.0), gamma=3.0)
    assert hi["k_hat"][0] == 16                                     # never more than k


def test_silu_odd_part_identity():
    """SiLU(x) - SiLU(-x) = x (sigma(x) + sigma(-x) = 1): with W1 = [[1], [-1]]
    and w2 = [1, -1] the logit is exactly the input, so a_hat = sigmoid(x); and
    through the bias path (W1 = 0, b1 = [x, -x]) the same."""
    xs = np.array([-3.0, -0.5, 0.0, 0.25, 2.0, 7.0])
    for x in xs:
        r = _head([[[x]]], [[1.0], [-1.0]], [0.0, 0.0], [1.0, -1.0], 0.0)
        assert abs(r["a_hat"][0] - 1.0 / (1.0 + math.exp(-x))) < 1e-12
        r = _head([[[5.0]]], [[0.0], [0.0]], [x, -x], [1.0, -1.0], 0.0)
        assert abs(r["a_hat"][0] - 1.0 / (1.0 + math.exp(-x))) < 1e-12


def test_silu_minimum_bounds_the_rate():
    """With one projected feature and w2 = 1, b2 = 0, a_hat = sigmoid(mean SiLU),
    and SiLU >= its minimum m = SiLU(x*), x* the root of 1 + x (1 - sigma(x)) = 0
    (found here by bisection): a_hat >= sigmoid(m), with equality at x*."""
    def sig(x):
        return 1.0 / (1.0 + math.exp(-x))
    lo, hi = -3.0, 0.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if 1.0 + mid * (1.0 - sig(mid)) > 0.0:
            hi = mid
        else:
            lo = mid
    xstar = 0.5 * (lo + hi)
    m = xstar * sig(xstar)
    rng = np.random.default_rng(1)
    x = rng.uniform(-6, 6, size=(50, 3, 1))
    r = _head(x, [[1.0]], [0.0], [1.0], 0.0)
    assert np.all(r["a_hat"] >= sig(m) - 1e-12)
    r = _head([[[xstar]]], [[1.0]], [0.0], [1.0], 0.0)
    assert abs(r["a_hat"][0] - sig(m)) < 1e-9


def test_mean_over_positions():
    """The pool is a mean: the same vector at every position gives the same
    a_hat for any k, and permuting positions changes nothing."""
    rng = np.random.default_rng(2)
    H, Hp = 16, 8
    w1 = rng.normal(size=(Hp, H)) / 4
    b1 = rng.normal(size=Hp)
    w2 = rng.normal(size=Hp)
    v = rng.normal(size=H)
    a = [_head(np.tile(v, (1, k, 1)), w1, b1, w2, 0.3)["a_hat"][0] for k in (1, 5, 16)]
    assert abs(a[0] - a[1]) < 1e-12 and abs(a[0] - a[2]) < 1e-12
    h = rng.normal(size=(1, 16, H))
    perm = rng.permutation(16)
    assert abs(_head(h, w1, b1, w2, 0.3)["a_hat"][0] - _head(h[:, perm], w1, b1, w2, 0.3)["a_hat"][0]) < 1e-12


def test_projection_is_linear_in_the_input():
    """Before the SiLU the projection is linear: scaling the hidden state and
    W1's inverse cancel (same a_hat), bf16 bits and fp32 give the same a_hat
    on bf16-representable inputs."""
    rng = np.random.default_rng(3)
    H, Hp, k = 32, 4, 4
    h = rng.normal(size=(2, k, H)).astype(np.float32)
    w1 = (rng.normal(size=(Hp, H)) / 8).astype(np.float32)
    b1, w2 = rng.normal(size=Hp), rng.normal(size=Hp)
    a1 = _head(h * 4.0, w1 / 4.0, b1, w2, -0.2)["a_hat"]
    a2 = _head(h, w1, b1, w2, -0.2)["a_hat"]
    assert np.allclose(a1, a2, atol=1e-12)
    hb = (np.asarray(h, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    wb = (np.asarray(w1, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    hf = (hb.astype(np.uint32) << 16).view(np.float32)
    wf = (wb.astype(np.uint32) << 16).view(np.float32)
    ab = oracle.length_head(hb, wb, np.float32(b1), np.float32(w2), -0.2)["a_hat"]
    af = _head(hf, wf, b1, w2, -0.2)["a_hat"]
    assert np.array_equal(ab, af)


def test_label_and_loss():
    """a* is the accepted fraction of the verified tokens; the MSE is zero at
    a_hat = a*; a bad request has no label."""
    acc = np.array([3, 0, 16, -1, 2])
    cu = np.array([0, 4, 12, 28, 30, 32])
    a_hat = np.array([0.75, 0.5, 1.0, 0.3, 0.0])
    r = oracle.length_label(acc, cu, a_hat)
    assert np.allclose(r["a_star"][:3], [0.75, 0.0, 1.0])
    assert r["a_star"][4] == 1.0
    assert np.allclose(r["loss"][[0, 2]], 0.0) and abs(r["loss"][1] - 0.25) < 1e-15
    assert r["loss"][4] == 1.0
    assert math.isnan(r["a_star"][3]) and math.isnan(r["loss"][3])
