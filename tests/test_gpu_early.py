"""GPU parity: spec_verify_early (early-exit verification) against the oracle
and spec_verify.

Leftmost rejection ("DFlash 阅读笔记：并行起草、目标特征与精确验证" §5.2,
Algorithm 1) leaves every row after a request's first rejection without
influence on its result, so the early-exit path must return the oracle's
accept_len and next_token (bit-exact outside the oracle's flagged near-ties,
same uniforms) while reading fewer bytes.  Greedy results are exact, so there
it must equal spec_verify everywhere.  bytes_read is bounded below by the rows
the accepted lengths make necessary and above by the whole batch; the
cluster path (16-byte pitched rows) reads at most one position past each
request's first rejection.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare_verify, gpu_verify, to_torch_i32, to_torch_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()


def _early(b, T, seed=None, max_len=32, status=None, tokens=None, target=None, draft=None, cu=None,
           total_rows=None):
    import torch
    import serving_vocab_wide_gb300 as svw
    nbytes = torch.zeros(1, dtype=torch.int64, device="cuda")
    acc, nxt = svw.spec_verify_early(
        to_torch_logits(b.target if target is None else target),
        to_torch_logits(b.draft if draft is None else draft),
        to_torch_i32(b.cu if cu is None else cu),
        to_torch_i32(b.tokens[float(T)] if tokens is None else tokens), T,
        b.seed if seed is None else seed, max_len=max_len,
        total_draft_rows=b.total_rows if total_rows is None else total_rows, status=status, bytes_read=nbytes)
    return acc.cpu().numpy(), nxt.cpu().numpy(), int(nbytes.item())


def _row_bytes(b):
    return b.V * (2 if b.target.dtype == np.uint16 else 4)


def _bounds(b, acc, T):
    """(least, whole-batch) logit bytes: positions 0..j* of every request (the
    bonus row when nothing is rejected) against every row."""
    L = np.diff(b.cu).astype(np.int64)
    per = 1 if T == 0 else 2
    least = np.where(acc < L, per * (acc + 1), per * L + 1)
    return int(least.sum()) * _row_bytes(b), int((per * L + 1).sum()) * _row_bytes(b)


def _ahead(b, acc, T):
    """Bytes the cluster path may read one position ahead: the rows of
    position j* + 1 of every request rejected at j* < L."""
    L = np.diff(b.cu).astype(np.int64)
    nxt_rows = np.where(acc + 1 < L, 1 if T == 0 else 2, 1)
    return int(np.where(acc < L, nxt_rows, 0).sum()) * _row_bytes(b)


def _pitched(b):
    return (_row_bytes(b) % 16) == 0


def _against_spec_verify(b, T, acc, nxt, label, reqs=None):
    """Equal to spec_verify, except (T > 0) on requests the oracle flags as a
    near-tie, where the two fp32 paths may round apart."""
    acc0, nxt0 = gpu_verify(b, T)
    mism = np.nonzero((acc != acc0) | (nxt != nxt0))[0]
    if T == 0 or mism.size == 0:
        assert mism.size == 0, (label, mism[:5])
        return
    assert mism.size <= max(2, b.N // 50), (label, mism)
    sub = b.subset(mism)
    ref = oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[float(T)], T, b.seed,
                             req_ids=np.asarray(mism, np.int32))
    nf, _ = compare_verify(acc[mism], nxt[mism], ref, label + " (differs from spec_verify)")
    assert nf == mism.size, (label, "unflagged difference from spec_verify")


def _check(b, T, label):
    acc, nxt, nbytes = _early(b, T)
    ref = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[float(T)], T, b.seed)
    compare_verify(acc, nxt, ref, label)
    _against_spec_verify(b, T, acc, nxt, label)
    least, whole = _bounds(b, acc, T)
    assert least <= nbytes <= whole, (label, least, nbytes, whole)
    if _pitched(b):
        assert nbytes <= least + _ahead(b, acc, T), (label, least, nbytes)
    return acc, nbytes, least, whole


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
def test_ragged_wide_vocab(T):
    b = synth.config(5, N=10, lengths=np.array([2, 4, 8, 16, 1, 3, 16, 7, 5, 12], np.int32), seed=77)
    if float(T) not in b.tokens:
        b.tokens[float(T)] = synth.sample_tokens(b.draft, T, 77)
    _check(b, T, f"ragged T={T}")


def test_tiny_fp32():
    _check(synth.config(1), 1.0, "tiny")


@pytest.mark.parametrize("V,dtype", [(5003, "bf16"), (1001, "f32"), (4100, "f32"), (8, "bf16"),
                                     (65543, "bf16")])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_odd_shapes(V, dtype, T):
    """Row pitches that are not a multiple of 16 bytes take the plain-load path."""
    lengths = np.array([1, 5, 3, 16, 9, 2], np.int32)
    b = synth.make_batch("odd", seed=V, lengths=lengths, V=V, dtype=dtype, target_sd=2.0,
                         sigma_req=np.array([0.5, 1.0, 2.0, 3.0, 1.5, 0.7]), temperatures=(T,))
    _check(b, T, f"V={V} {dtype} T={T}")


def test_all_accepted_reads_everything():
    """Draft = target: p = q, every token passes, every row (bonus included) is read."""
    b = synth.make_batch("same", seed=5, lengths=np.array([3, 16, 1, 8], np.int32), V=2048, dtype="bf16",
                         sigma_req=np.ones(4), temperatures=(1.0,))
    L = np.diff(b.cu)
    tgt = b.target.copy()
    for i in range(b.N):
        tgt[b.cu[i] + i:b.cu[i + 1] + i] = b.draft[b.cu[i]:b.cu[i + 1]]
    acc, nxt, nbytes = _early(b, 1.0, target=tgt)
    assert np.array_equal(acc, L)
    ref = oracle.spec_verify(tgt, b.draft, b.cu, b.tokens[1.0], 1.0, b.seed)
    compare_verify(acc, nxt, ref, "same")
    assert nbytes == int((2 * L + 1).sum()) * _row_bytes(b)


def test_first_position_rejected_reads_little():
    """p(x_0) = 0 in every request: rejected at position 0 for any uniform.
    The position-major stream must skip nearly all later rows."""
    b = synth.make_batch("rej0", seed=6, lengths=np.full(64, 16, np.int32), V=151936, dtype="bf16",
                         sigma_req=np.full(64, 1.0), temperatures=(1.0,))
    tgt = b.target.copy()
    tok = b.tokens[1.0]
    for i in range(b.N):
        tgt[b.cu[i] + i, tok[b.cu[i]]] = 0xFF80  # -inf at the drafted token of position 0
    acc, nxt, nbytes = _early(b, 1.0, target=tgt)
    assert np.all(acc == 0)
    ref = oracle.spec_verify(tgt[:6 * 17], b.draft[:6 * 16], b.cu[:7], tok[:6 * 16], 1.0, b.seed)
    compare_verify(acc[:6], nxt[:6], ref, "rej0")
    least, whole = _bounds(b, acc, 1.0)
    assert least <= nbytes < 0.3 * whole, (least, nbytes, whole)


def test_rows_after_the_rejection_are_not_checked():
    """A NaN row after a certain rejection does not make the request bad (it is
    never needed); at or before the rejection it does, as with spec_verify."""
    import torch
    import serving_vocab_wide_gb300 as svw
    V = 4096
    b = synth.make_batch("nanafter", seed=8, lengths=np.array([6, 6, 6, 6], np.int32), V=V, dtype="bf16",
                         sigma_req=np.ones(4), temperatures=(1.0,))
    tok = b.tokens[1.0]
    tgt, drf = b.target.copy(), b.draft.copy()
    for i in range(b.N):
        drf[b.cu[i]] = tgt[b.cu[i] + i]                  # p = q at position 0: always accepted
        tgt[b.cu[i] + i + 1, tok[b.cu[i] + 1]] = 0xFF80  # p(x_1) = 0: position 1 always rejected
    clean_t, clean_d = tgt.copy(), drf.copy()
    tgt[b.cu[0] + 0 + 3, 5] = 0x7FC0      # request 0: NaN target row at position 3 (after)
    drf[b.cu[1] + 5, 9] = 0x7FC0          # request 1: NaN draft row at position 5 (after)
    tgt[b.cu[2] + 2 + 1, 7] = 0x7FC0      # request 2: NaN at the rejected position itself
    drf[b.cu[3] + 0, 7] = 0x7FC0          # request 3: NaN before the rejection
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt, _ = _early(b, 1.0, target=tgt, draft=drf, status=status)
    ref = oracle.spec_verify(clean_t, clean_d, b.cu, tok, 1.0, b.seed)
    assert list(acc[:2]) == list(ref["accept_len"][:2]) == [1, 1]
    assert list(nxt[:2]) == list(ref["next_token"][:2])
    assert list(acc[2:]) == [-1, -1] and list(nxt[2:]) == [-1, -1]
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT
    # spec_verify reads every row, so all four are bad there
    acc_full, _ = svw.spec_verify(to_torch_logits(tgt), to_torch_logits(drf), to_torch_i32(b.cu),
                                  to_torch_i32(tok), 1.0, b.seed, total_draft_rows=b.total_rows)
    assert acc_full.cpu().tolist() == [-1, -1, -1, -1]


def test_bad_tokens_lengths_and_csr():
    import torch
    import serving_vocab_wide_gb300 as svw
    V = 256
    b = synth.make_batch("bad", seed=3, lengths=np.array([2, 3, 2, 40], np.int32), V=V, dtype="bf16",
                         sigma_req=np.ones(4), temperatures=(1.0,))
    tok = b.tokens[1.0].copy()
    tok[int(b.cu[1]) + 2] = V + 5         # request 1: last token out of range
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt, _ = _early(b, 1.0, tokens=tok, status=status)
    ref = oracle.spec_verify(b.target, b.draft, b.cu, tok, 1.0, b.seed)
    assert acc[1] == acc[3] == nxt[1] == nxt[3] == -1  # bad token; length above max_len
    for i in (0, 2):
        assert acc[i] == ref["accept_len"][i] and nxt[i] == ref["next_token"][i]
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT
    # offsets that disagree with total_draft_rows: every request is bad
    c = synth.make_batch("csr", seed=4, lengths=np.array([2, 2], np.int32), V=64, sigma_req=np.ones(2),
                         temperatures=(1.0,))
    acc, nxt, _ = _early(c, 1.0, total_rows=3)
    assert list(acc) == [-1, -1] and list(nxt) == [-1, -1]


def test_greedy_ties_and_bonus():
    import serving_vocab_wide_gb300 as svw
    V = 4096
    y = np.zeros((5, V), np.float32)
    y[0, [10, 20]] = 3.0
    y[1, [7, 3000]] = 5.0
    y[2, 99] = 1.0
    y[3, [4095, 4094]] = 2.0
    y[4, :] = -1.0
    tgt = synth.bf16_bits(y)
    drf = np.zeros((3, V), np.uint16)
    cu = np.array([0, 2, 3], np.int32)
    for tok, exp_acc, exp_nxt in (([10, 7, 4094], [2, 1], [99, 0]),
                                  ([20, 7, 4094], [0, 1], [10, 0]),
                                  ([10, 8, 4095], [1, 0], [7, 4094])):
        acc, nxt = svw.spec_verify_early(to_torch_logits(tgt), to_torch_logits(drf), to_torch_i32(cu),
                                         to_torch_i32(tok), 0.0, 0, total_draft_rows=3)
        assert acc.cpu().tolist() == exp_acc and nxt.cpu().tolist() == exp_nxt


def test_deterministic_results():
    b = synth.config(3, N=24, seed=5)
    a1, n1, _ = _early(b, 1.0)
    a2, n2, _ = _early(b, 1.0)
    assert np.array_equal(a1, a2) and np.array_equal(n1, n2)


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
def test_mix_full_size(T, mix_batch):
    """The benchmark's batch: every request equals spec_verify's; a seeded
    sample against the oracle."""
    b = mix_batch
    acc, nxt, nbytes = _early(b, T)
    _against_spec_verify(b, T, acc, nxt, f"mix T={T}")
    least, whole = _bounds(b, acc, T)
    assert least <= nbytes <= least + _ahead(b, acc, T)
    reqs = np.sort(np.random.default_rng(3).choice(b.N, 12, replace=False))
    sub = b.subset(reqs)
    ref = oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[float(T)], T, b.seed,
                             req_ids=np.asarray(reqs, np.int32))
    compare_verify(acc[reqs], nxt[reqs], ref, f"mix T={T}")
    print(f"mix T={T}: read {nbytes / whole:.3f} of the batch (least {least / whole:.3f})")


@pytest.fixture(scope="module")
def mix_batch():
    return synth.config(5)
