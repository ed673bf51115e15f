"""GPU parity: spec_verify_filtered (top-k / top-p filtered verification,
through the C ABI) against the oracle.

Filtering is not on the pages; the reading is the oracle's (both
distributions filtered with the same T, top_k, top_p; "DFlash 阅读笔记：并行
起草、目标特征与精确验证" §5.2 on the filtered p' and q').  accept_len and
next_token must be bit-exact except on requests the oracle flags as within
1e-5 of an accept threshold, a CDF boundary or a top-p cut.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import NEAR, to_torch_i32, to_torch_logits

pytestmark = pytest.mark.gpu

NEARF = NEAR | oracle.FLAG_NEAR_FILTER


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()


def _gpu(target, draft, cu, tok, T, k, p, seed, status=None, total_rows=None):
    import serving_vocab_wide_gb300 as svw
    acc, nxt = svw.spec_verify_filtered(to_torch_logits(target), to_torch_logits(draft), to_torch_i32(cu),
                                        to_torch_i32(tok), T, k, p, seed,
                                        total_draft_rows=int(cu[-1]) if total_rows is None else total_rows,
                                        status=status)
    return acc.cpu().numpy(), nxt.cpu().numpy()


def _compare(acc, nxt, ref, label):
    near = (ref["flags"] & NEARF) != 0
    mism = (acc != ref["accept_len"]) | (nxt != ref["next_token"])
    bad = np.nonzero(mism & ~near)[0]
    assert bad.size == 0, (f"{label}: {bad.size} unflagged mismatches, first {bad[:5]}: gpu {acc[bad[:5]]} "
                           f"{nxt[bad[:5]]} oracle {ref['accept_len'][bad[:5]]} {ref['next_token'][bad[:5]]}")
    return int(near.sum())


def _check(b, T, k, p, label, seed=None, reqs=None):
    seed = b.seed if seed is None else seed
    tok = synth.sample_tokens_filtered(b.draft, T, k, p, 31)
    acc, nxt = _gpu(b.target, b.draft, b.cu, tok, T, k, p, seed)
    if reqs is None:
        ref = oracle.spec_verify_filtered(b.target, b.draft, b.cu, tok, T, k, p, seed)
    else:
        sub = b.subset(reqs)
        stok = np.concatenate([tok[b.cu[i]:b.cu[i + 1]] for i in reqs]).astype(np.int32)
        ref = oracle.spec_verify_filtered(sub.target, sub.draft, sub.cu, stok, T, k, p, seed,
                                          req_ids=np.asarray(reqs, np.int32))
        acc, nxt = acc[reqs], nxt[reqs]
    assert np.all(acc >= 0), label
    _compare(acc, nxt, ref, label)
    return acc, nxt


@pytest.mark.parametrize("k,p", [(1, 1.0), (20, 0.9), (50, 1.0), (5, 0.5), (1024, 0.95), (300, 0.6)])
@pytest.mark.parametrize("V,dtype", [(4096, "bf16"), (5003, "bf16"), (4100, "f32"), (1001, "f32")])
def test_shapes_and_filters(V, dtype, k, p):
    lengths = np.array([1, 5, 3, 16, 9, 2], np.int32)
    b = synth.make_batch("flt", seed=V + k, lengths=lengths, V=V, dtype=dtype, target_sd=2.0,
                         sigma_req=np.array([0.3, 1.0, 2.0, 0.5, 1.5, 0.7]), temperatures=(1.0,))
    _check(b, 1.0, k, p, f"V={V} {dtype} k={k} p={p}")


@pytest.mark.parametrize("T,k,p", [(1.0, 50, 0.9), (0.6, 1024, 0.95), (1.0, 1, 1.0)])
def test_wide_vocab_ragged(T, k, p):
    b = synth.config(5, N=10, lengths=np.array([2, 4, 8, 16, 1, 3, 16, 7, 5, 12], np.int32), seed=77)
    _check(b, T, k, p, f"V=151936 T={T} k={k} p={p}")


def test_tiny_rows_keep_everything():
    """V = 8 with top_k >= V: every entry is a candidate."""
    b = synth.make_batch("tiny", seed=2, lengths=np.array([3, 1, 4], np.int32), V=8, dtype="bf16",
                         target_sd=1.0, sigma_req=np.ones(3), temperatures=(1.0,))
    _check(b, 1.0, 16, 1.0, "V=8 k=16")
    _check(b, 1.0, 3, 0.8, "V=8 k=3 p=0.8")


def test_heavy_ties_and_constant_rows():
    """Integer-valued logits (thousands of ties at the top-k key) and
    constant rows: ties are kept in index order."""
    rng = np.random.default_rng(5)
    lengths = np.array([4, 3, 6], np.int32)
    b = synth.make_batch("ties", seed=6, lengths=lengths, V=8192, dtype="bf16", sigma_req=np.ones(3),
                         temperatures=(1.0,))
    t = synth.bf16_bits(np.round(rng.normal(0, 1.0, size=(b.target.shape[0], b.V))).astype(np.float32))
    d = synth.bf16_bits(np.round(rng.normal(0, 1.0, size=(b.draft.shape[0], b.V))).astype(np.float32))
    t[1, :] = synth.bf16_bits(np.full(b.V, 0.5, np.float32))   # a constant target row
    d[2, :] = synth.bf16_bits(np.full(b.V, -1.0, np.float32))  # a constant draft row
    b.target, b.draft = t, d
    for k, p in ((40, 1.0), (700, 0.3), (1024, 1.0)):
        _check(b, 1.0, k, p, f"ties k={k} p={p}")


def test_masked_entries():
    """Rows with -inf entries (a masked vocabulary), fewer finite entries than top_k."""
    b = synth.make_batch("mask", seed=9, lengths=np.array([3, 5], np.int32), V=4096, dtype="bf16",
                         sigma_req=np.ones(2), temperatures=(1.0,))
    t, d = b.target.copy(), b.draft.copy()
    keep = np.zeros(b.V, bool)
    keep[np.random.default_rng(1).choice(b.V, 30, replace=False)] = True
    t[:, ~keep] = 0xFF80
    d[:, ~keep] = 0xFF80
    b.target, b.draft = t, d
    _check(b, 1.0, 100, 1.0, "masked k=100")
    _check(b, 1.0, 10, 0.9, "masked k=10 p=0.9")


def test_bad_rows_and_tokens():
    import torch
    import serving_vocab_wide_gb300 as svw
    V = 512
    b = synth.make_batch("bad", seed=3, lengths=np.array([2, 3, 2, 40], np.int32), V=V, dtype="bf16",
                         sigma_req=np.ones(4), temperatures=(1.0,))
    tok = synth.sample_tokens_filtered(b.draft, 1.0, 20, 0.9, 4)
    tok[int(b.cu[1]) + 1] = V + 3               # request 1: token out of range
    t = b.target.copy()
    t[int(b.cu[2]) + 2 + 1, 17] = 0x7FC0        # request 2: NaN target row
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt = _gpu(t, b.draft, b.cu, tok, 1.0, 20, 0.9, 0, status=status)
    ref = oracle.spec_verify_filtered(t, b.draft, b.cu, tok, 1.0, 20, 0.9, 0)
    assert list(acc[1:]) == [-1, -1, -1] and list(nxt[1:]) == [-1, -1, -1]
    assert np.all(ref["flags"][1:] & oracle.FLAG_BAD)
    assert acc[0] == ref["accept_len"][0] and nxt[0] == ref["next_token"][0]
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT


def test_greedy_is_spec_verify():
    import serving_vocab_wide_gb300 as svw
    b = synth.make_batch("g", seed=8, lengths=np.array([3, 6, 2], np.int32), V=5000, dtype="bf16",
                         sigma_req=np.ones(3), temperatures=(0.0,))
    acc, nxt = _gpu(b.target, b.draft, b.cu, b.tokens[0.0], 0.0, 3, 0.5, 2)
    a0, n0 = svw.spec_verify(to_torch_logits(b.target), to_torch_logits(b.draft), to_torch_i32(b.cu),
                             to_torch_i32(b.tokens[0.0]), 0.0, 2, total_draft_rows=b.total_rows)
    assert np.array_equal(acc, a0.cpu().numpy()) and np.array_equal(nxt, n0.cpu().numpy())


def test_lossless_chisquare_on_gpu():
    """The first emitted token is distributed as the filtered target p'."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(21)
    V, n, T, k, p = 8, 1_000_000, 0.9, 5, 0.85
    y = rng.normal(0, 1.5, size=V).astype(np.float32)
    z = (y + rng.normal(0, 1.0, size=V)).astype(np.float32)

    def filt(row):
        keep = synth.filter_mask(row, T, k, p)
        e = np.exp((row.astype(np.float64) - row.max()) / T) * keep
        return e / e.sum()

    pf, qf = filt(y), filt(z)
    tgt = np.ascontiguousarray(np.broadcast_to(np.stack([y, y]), (n, 2, V)).reshape(-1, V))
    drf = np.ascontiguousarray(np.broadcast_to(z, (n, V)))
    cu = synth.cu_from_lengths(np.ones(n, np.int32))
    tok = rng.choice(V, size=n, p=qf).astype(np.int32)
    acc, nxt = _gpu(tgt, drf, cu, tok, T, k, p, 17)
    first = np.where(acc >= 1, tok, nxt)
    cnt = np.bincount(first, minlength=V)
    m = pf > 0
    assert np.all(cnt[~m] == 0)
    assert chisquare(cnt[m], pf[m] * n).pvalue > 1e-4
    ref = oracle.spec_verify_filtered(tgt[:40000], drf[:20000], cu[:20001], tok[:20000], T, k, p, 17)
    _compare(acc[:20000], nxt[:20000], ref, "chisq subset")


def test_mix_full_size_sampled(mix_batch):
    reqs = np.sort(np.random.default_rng(4).choice(mix_batch.N, 10, replace=False))
    _check(mix_batch, 1.0, 50, 0.9, "mix N=256 k=50 p=0.9", reqs=reqs)


@pytest.fixture(scope="module")
def mix_batch():
    return synth.config(5)
