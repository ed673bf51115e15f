"""GPU parity: spec_verify (CUDA, through the C ABI) against the oracle.

accept_len and next_token must be bit-exact except on requests the oracle
flags as within 1e-5 of an accept threshold or of a CDF boundary; those are
counted.  Full-size workloads compare every request (the oracle's requests
split over the host's cores, with the batch's own Philox request indices) and
bound the share of flagged requests.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (check_near_ties, compare_verify, gpu_verify, oracle_verify_all, to_torch_i32,
                     to_torch_logits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()


def _oracle(b, T, reqs=None, alt_next=None):
    if reqs is None:
        return oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[float(T)], T, b.seed, alt_next=alt_next)
    sub = b.subset(reqs)
    return oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[float(T)], T, b.seed,
                              req_ids=np.asarray(reqs, np.int32), alt_next=alt_next)


def _check(b, T, reqs=None, label=""):
    acc, nxt = gpu_verify(b, T)
    if reqs is not None:
        acc, nxt = acc[reqs], nxt[reqs]
    ref = _oracle(b, T, reqs, alt_next=nxt)
    nf, nfm = compare_verify(acc, nxt, ref, label)
    assert np.all(acc >= 0)
    return acc, nxt, nf


def test_tiny_fp32():
    b = synth.config(1)
    acc, nxt, _ = _check(b, 1.0, label="tiny")
    assert acc.max() >= 1  # not all rejected at position 0


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
def test_ragged_wide_vocab_all_requests(T):
    b = synth.config(5, N=10, lengths=np.array([2, 4, 8, 16, 1, 3, 16, 7, 5, 12], np.int32),
                     seed=77)
    if float(T) not in b.tokens:
        b.tokens[float(T)] = synth.sample_tokens(b.draft, T, 77)
    _check(b, T, label=f"ragged T={T}")


@pytest.mark.parametrize("V,dtype", [(5003, "bf16"), (1001, "f32"), (8, "bf16"), (1, "f32"),
                                     (4100, "f32"), (65543, "bf16"),
                                     # a 256K vocabulary: 15 chunks per row, and the draw's widest rows
                                     (262144, "bf16")])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_odd_shapes(V, dtype, T):
    lengths = np.array([1, 5, 3, 16], np.int32)
    b = synth.make_batch("odd", seed=V, lengths=lengths, V=V, dtype=dtype, target_sd=2.0,
                         sigma_req=np.array([0.5, 1.0, 2.0, 3.0]), temperatures=(T,))
    _check(b, T, label=f"V={V} {dtype} T={T}")


def test_greedy_ties_and_bonus():
    import torch
    import serving_vocab_wide_gb300 as svw
    V = 4096
    y = np.zeros((5, V), np.float32)
    y[0, [10, 20]] = 3.0          # tie: argmax 10
    y[1, [7, 3000]] = 5.0         # argmax 7
    y[2, 99] = 1.0                # bonus row of request 0
    y[3, [4095, 4094]] = 2.0      # request 1 row 0: argmax 4094
    y[4, :] = -1.0                # request 1 bonus: all equal -> 0
    tgt = synth.bf16_bits(y)
    drf = np.zeros((3, V), np.uint16)
    cu = np.array([0, 2, 3], np.int32)
    for tok, exp_acc, exp_nxt in (([10, 7, 4094], [2, 1], [99, 0]),
                                  ([20, 7, 4094], [0, 1], [10, 0]),
                                  ([10, 8, 4095], [1, 0], [7, 4094])):
        acc, nxt = svw.spec_verify(to_torch_logits(tgt), to_torch_logits(drf), to_torch_i32(cu),
                                   to_torch_i32(tok), 0.0, 0, total_draft_rows=3)
        assert acc.cpu().tolist() == exp_acc
        assert nxt.cpu().tolist() == exp_nxt
        ref = oracle.spec_verify(tgt, drf, cu, np.array(tok, np.int32), 0.0, 0)
        assert ref["accept_len"].tolist() == exp_acc and ref["next_token"].tolist() == exp_nxt


def test_bad_inputs_are_reported():
    import torch
    import serving_vocab_wide_gb300 as svw
    V = 256
    lengths = np.array([2, 3, 2, 2, 40], np.int32)   # the last exceeds max_len
    b = synth.make_batch("bad", seed=3, lengths=lengths, V=V, dtype="bf16",
                         sigma_req=np.ones(5), temperatures=(1.0,))
    tok = b.tokens[1.0].copy()
    tok[2] = V + 5                                # request 1: token out of range
    t = b.target.copy()
    t[int(b.cu[2]) + 2 + 1, 17] = 0x7FC0          # request 2, target row 1: NaN
    d = b.draft.copy()
    d[int(b.cu[3]), :] = 0xFF80                   # request 3, draft row 0: all -inf
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt = svw.spec_verify(to_torch_logits(t), to_torch_logits(d), to_torch_i32(b.cu),
                               to_torch_i32(tok), 1.0, 0, total_draft_rows=b.total_rows,
                               status=status)
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    ref = oracle.spec_verify(t, d, b.cu, tok, 1.0, 0)
    assert list(acc[1:]) == [-1, -1, -1, -1] and list(nxt[1:]) == [-1, -1, -1, -1]
    assert np.all(ref["flags"][1:] & oracle.FLAG_BAD)
    assert acc[0] == ref["accept_len"][0] and nxt[0] == ref["next_token"][0]
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT
    # greedy: only NaN makes a row bad
    tok0 = synth.sample_tokens(d, 0.0, 3)
    tok0[2] = 1
    acc, _ = svw.spec_verify(to_torch_logits(t), to_torch_logits(d), to_torch_i32(b.cu),
                             to_torch_i32(tok0), 0.0, 0, total_draft_rows=b.total_rows)
    ref = oracle.spec_verify(t, d, b.cu, tok0, 0.0, 0)
    assert acc.cpu().numpy().tolist() == ref["accept_len"].tolist()


def test_inconsistent_csr_is_rejected_on_device():
    import torch
    import serving_vocab_wide_gb300 as svw
    V = 64
    b = synth.make_batch("csr", seed=4, lengths=np.array([2, 2], np.int32), V=V,
                         sigma_req=np.ones(2), temperatures=(1.0,))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt = svw.spec_verify(to_torch_logits(b.target), to_torch_logits(b.draft),
                               to_torch_i32(b.cu), to_torch_i32(b.tokens[1.0]), 1.0, 0,
                               total_draft_rows=3, status=status)  # cu[N] = 4 != 3
    assert acc.cpu().tolist() == [-1, -1] and nxt.cpu().tolist() == [-1, -1]
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT


def test_concurrent_host_threads():
    """Calls from several host threads at once, each on its own stream with
    its own workspace, give the results of the same calls made one by one
    (the library's launch caches are shared between threads)."""
    import threading
    import torch
    import serving_vocab_wide_gb300 as svw
    batches = [synth.config(5, N=6, lengths=np.array([3, 16, 1, 8, 5, 2], np.int32), V=32768, seed=300 + q)
               for q in range(4)]
    temps = [1.0, 0.0, 1.0, 0.0]

    def call(b, T, stream):
        with torch.cuda.stream(stream):
            acc, nxt = svw.spec_verify(to_torch_logits(b.target), to_torch_logits(b.draft), to_torch_i32(b.cu),
                                       to_torch_i32(b.tokens[T]), T, b.seed, max_len=32,
                                       total_draft_rows=b.total_rows, stream=stream)
        stream.synchronize()
        return acc.cpu().numpy(), nxt.cpu().numpy()

    ref = [call(b, T, torch.cuda.Stream()) for b, T in zip(batches, temps)]
    out = [None] * len(batches)
    streams = [torch.cuda.Stream() for _ in batches]

    def work(q):
        for _ in range(5):
            out[q] = call(batches[q], temps[q], streams[q])

    threads = [threading.Thread(target=work, args=(q,)) for q in range(len(batches))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    for q in range(len(batches)):
        assert np.array_equal(out[q][0], ref[q][0]) and np.array_equal(out[q][1], ref[q][1])


def test_deterministic_rerun():
    b = synth.config(3, N=12, seed=5)
    a1, n1 = gpu_verify(b, 1.0)
    a2, n2 = gpu_verify(b, 1.0)
    assert np.array_equal(a1, a2) and np.array_equal(n1, n2)


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_lossless_chisquare_on_gpu(T):
    """The CUDA path's first emitted token is distributed as p (eq. (8))."""
    from scipy.special import softmax
    from scipy.stats import chisquare
    import serving_vocab_wide_gb300 as svw
    rng = np.random.default_rng(9)
    V, n = 8, 1_000_000
    y = rng.normal(0, 1.5, size=(2, V)).astype(np.float32)
    z = (y[:1] + rng.normal(0, 1.0, size=(1, V))).astype(np.float32)
    tgt = np.ascontiguousarray(np.broadcast_to(y, (n, 2, V)).reshape(-1, V))
    drf = np.ascontiguousarray(np.broadcast_to(z, (n, 1, V)).reshape(-1, V))
    cu = synth.cu_from_lengths(np.ones(n, np.int32))
    tok = synth.sample_tokens(drf, T, 123)
    acc, nxt = svw.spec_verify(to_torch_logits(tgt), to_torch_logits(drf), to_torch_i32(cu),
                               to_torch_i32(tok), T, 31, total_draft_rows=n)
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    first = np.where(acc >= 1, tok, nxt)
    p0 = softmax(y[0].astype(np.float64) / T)
    assert chisquare(np.bincount(first, minlength=V), p0 * n).pvalue > 1e-4
    ref = oracle.spec_verify(tgt[:40000], drf[:20000], cu[:20001], tok[:20000], T, 31)
    compare_verify(acc[:20000], nxt[:20000], ref, "chisq subset")


# ---------------------------------------------------------------------------
# full-size workloads (the shapes the benchmark times), sampled requests
# ---------------------------------------------------------------------------
def test_fixed_length_full_size():
    b = synth.config(2)
    acc, nxt = _check_all(b, 1.0, "fixed N=32")
    tau = acc.mean() + 1
    assert 2.0 < tau < 12.0


def _check_all(b, T, label):
    """Every request of a full-size batch against the oracle (threaded), with
    the near-tie excusals counted and bounded."""
    acc, nxt = gpu_verify(b, T)
    ref = oracle_verify_all(b, T, alt_next=nxt)
    nf, nfm = compare_verify(acc, nxt, ref, label)
    check_near_ties(ref, nfm, label)
    assert np.all(acc >= 0)
    return acc, nxt


def test_ragged_full_size_all_requests():
    _check_all(synth.config(3), 1.0, "ragged N=128")


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
def test_mix_full_size_all_requests(T, mix_batch):
    _check_all(mix_batch, T, f"mix N=256 T={T}")


@pytest.fixture(scope="module")
def mix_batch():
    return synth.config(5)
