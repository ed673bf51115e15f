"""GPU parity: the adaptive length head (forward and label) against the oracle.

a_hat within 1e-4 (absolute; it is a probability), k_hat bit-exact except
where the oracle flags gamma a_hat k within 1e-4 of an integer (the floor
could go either way under float rounding); the label within fp32 rounding of
what the oracle computes from the same a_hat.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()


def _bf16_bits(x):
    x = np.ascontiguousarray(x, np.float32)
    u = x.view(np.uint32)
    r = u + 0x7FFF + ((u >> 16) & 1)  # round to nearest even
    return (r >> 16).astype(np.uint16)


def _inputs(seed, N, k, H, Hp):
    rng = np.random.default_rng(seed)
    h = _bf16_bits(rng.normal(size=(N, k, H)))
    w1 = _bf16_bits(rng.normal(size=(Hp, H)) / np.sqrt(H) * 2.0)
    b1 = rng.normal(0, 0.3, size=Hp).astype(np.float32)
    w2 = (rng.normal(size=Hp) / np.sqrt(Hp) * 2.0).astype(np.float32)
    return h, w1, b1, w2


def _gpu(h, w1, b1, w2, b2, gamma):
    import torch
    import serving_vocab_wide_gb300 as svw
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    hb = t(h.view(np.int16)).view(torch.bfloat16)
    wb = t(w1.view(np.int16)).view(torch.bfloat16)
    a, kh = svw.length_head(hb, wb, t(b1), t(w2), b2, gamma)
    return a.cpu().numpy(), kh.cpu().numpy()


def _compare(a, kh, ref, label):
    assert np.all(np.abs(a.astype(np.float64) - ref["a_hat"]) <= 1e-4), \
        f"{label}: a_hat err {np.abs(a - ref['a_hat']).max()}"
    ok = (ref["flags"] & oracle.FLAG_NEAR_FLOOR) == 0
    assert np.array_equal(kh[ok], ref["k_hat"][ok]), label
    assert np.all((kh >= 1) & (kh <= 16))


@pytest.mark.parametrize("N,k,H,Hp,b2,gamma", [(5, 16, 256, 32, 0.5, 1.0), (9, 7, 512, 64, -0.8, 1.3),
                                               (3, 1, 64, 8, 2.0, 0.7), (33, 16, 1024, 128, 0.0, 1.0),
                                               # two 256-wide column tiles of W1, the second partial
                                               (7, 5, 512, 300, 0.1, 1.0),
                                               # K not a multiple of 64 (zero-filled tail); split ranks
                                               # with and without K blocks
                                               (4, 3, 200, 48, -0.3, 1.0), (6, 9, 136, 16, 0.4, 1.2),
                                               # several 128-row tiles, the last one partial
                                               (40, 13, 768, 200, 0.0, 0.9)])
def test_small_shapes(N, k, H, Hp, b2, gamma):
    h, w1, b1, w2 = _inputs(N * 7 + H, N, k, H, Hp)
    a, kh = _gpu(h, w1, b1, w2, b2, gamma)
    _compare(a, kh, oracle.length_head(h, w1, b1, w2, b2, gamma), f"N={N} H={H}")


def test_drafter_scale_all_requests():
    """N = 256 requests, k = 16, H = 4096 (drafter hidden size), H' = 256
    (the benchmark's shape): every request against the oracle (its requests
    split over host threads), and the same bits on a second call."""
    from concurrent.futures import ThreadPoolExecutor
    from helpers import host_threads
    N, k, H, Hp = 256, 16, 4096, 256
    h, w1, b1, w2 = _inputs(77, N, k, H, Hp)
    a, kh = _gpu(h, w1, b1, w2, 0.2, 1.0)
    a2, kh2 = _gpu(h, w1, b1, w2, 0.2, 1.0)
    assert np.array_equal(a, a2) and np.array_equal(kh, kh2)
    groups = np.array_split(np.arange(N), min(N, 2 * host_threads()))
    with ThreadPoolExecutor(host_threads()) as pool:
        refs = list(pool.map(lambda g: oracle.length_head(h[g], w1, b1, w2, 0.2, 1.0), groups))
    ref = {key: np.concatenate([r[key] for r in refs]) for key in ("a_hat", "k_hat", "flags")}
    _compare(a, kh, ref, "drafter scale")
    assert len(np.unique(kh)) > 3  # the lengths actually vary


def test_label():
    import torch
    import serving_vocab_wide_gb300 as svw
    rng = np.random.default_rng(9)
    N = 300
    L = rng.integers(1, 17, size=N)
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    acc = rng.integers(0, L + 1).astype(np.int32)
    acc[[3, 17]] = -1
    a_hat = rng.uniform(0, 1, size=N).astype(np.float32)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    a_star, loss = svw.length_head_label(t(acc), t(cu), t(a_hat))
    ref = oracle.length_label(acc, cu, a_hat.astype(np.float64))
    a_star, loss = a_star.cpu().numpy(), loss.cpu().numpy()
    ok = acc >= 0
    assert np.allclose(a_star[ok], ref["a_star"][ok], rtol=0, atol=1e-7)
    # (a_hat - a*)^2 in fp32: a* and the difference each round once, so the
    # error is about 2 |a_hat - a*| 2^-24 <= 2.4e-7, absolute
    assert np.all(np.abs(loss[ok] - ref["loss"][ok]) <= 1e-6)
    assert np.all(np.isnan(a_star[~ok])) and np.all(np.isnan(loss[~ok]))


@pytest.mark.parametrize("k", [16, 7])
def test_label_then_head_same_stream(k):
    """The label of this round reads last round's a_hat while the head that
    follows it on the same stream (a programmatic launch, which may start
    before the label ends) writes the new a_hat: the label must see only the
    old values, whichever finishing path the head takes (k = 16: the
    projection kernel finishes the requests; k = 7: a second kernel does)."""
    import torch
    import serving_vocab_wide_gb300 as svw
    N, H, Hp = 64, 512, 64
    h, w1, b1, w2 = _inputs(5 + k, N, k, H, Hp)
    rng = np.random.default_rng(17 + k)
    L = rng.integers(1, 17, size=N)
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    acc = rng.integers(0, L + 1).astype(np.int32)
    old = rng.uniform(0, 1, size=N).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    hb = t(h.view(np.int16)).view(torch.bfloat16)
    wb = t(w1.view(np.int16)).view(torch.bfloat16)
    a_hat = t(old)
    k_hat = torch.empty(N, dtype=torch.int32, device="cuda")
    for _ in range(3):  # repeated, so that a late write would show at least once
        a_hat.copy_(t(old))
        a_star, loss = svw.length_head_label(t(acc), t(cu), a_hat)
        svw.length_head(hb, wb, t(b1), t(w2), 0.1, 1.0, a_hat=a_hat, k_hat=k_hat)
        torch.cuda.synchronize()
        ref = oracle.length_label(acc, cu, old.astype(np.float64))
        assert np.all(np.abs(loss.cpu().numpy() - ref["loss"]) <= 1e-6)
        new = oracle.length_head(h, w1, b1, w2, 0.1, 1.0)
        assert np.all(np.abs(a_hat.cpu().numpy().astype(np.float64) - new["a_hat"]) <= 1e-4)
