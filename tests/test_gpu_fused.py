"""GPU parity: spec_verify_opd (verification and the OPD loss on the same
batch in one pass) against the oracle's spec_verify and opd_loss.

The same bars as the separate calls: accept_len / next_token bit-exact
outside the oracle's flagged near-ties, loss within 1e-4 relative, each
dlogits row within 1e-4 of its largest |entry|.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (check_near_ties, compare_opd, compare_opd_all, compare_verify, opd_errors,
                     oracle_verify_all, to_torch_i32, to_torch_logits)

pytestmark = pytest.mark.gpu

OPD = dict(clip_c=1.0, lambda_ce=0.1)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()


def _fused(b, T, To=None, status=None, tokens=None, **kw):
    import serving_vocab_wide_gb300 as svw
    tok = b.tokens[float(T)] if tokens is None else tokens
    acc, nxt, loss, g = svw.spec_verify_opd(
        to_torch_logits(b.target), to_torch_logits(b.draft), to_torch_i32(b.cu), to_torch_i32(tok), T,
        b.seed, opd_temperature=To, max_len=32, total_draft_rows=b.total_rows, status=status,
        **dict(OPD, **kw))
    return acc.cpu().numpy(), nxt.cpu().numpy(), loss.cpu().numpy(), g.cpu().numpy()


def _check(b, T, To, reqs=None, label="", **kw):
    acc, nxt, loss, g = _fused(b, T, To, **kw)
    opd_kw = dict(OPD, **kw)
    if reqs is None:
        vref = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[float(T)], T, b.seed)
        oref = oracle.opd_loss(b.target, b.draft, temperature=To, cu_draft=b.cu, has_bonus=True, **opd_kw)
        compare_verify(acc, nxt, vref, label)
        compare_opd(loss, g, oref, label=label)
    else:
        sub = b.subset(reqs)
        vref = oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[float(T)], T, b.seed,
                                  req_ids=np.asarray(reqs, np.int32))
        compare_verify(acc[reqs], nxt[reqs], vref, label)
        rows = np.concatenate([np.arange(b.cu[i], b.cu[i + 1]) for i in reqs])
        oref = oracle.opd_loss(sub.target, sub.draft, temperature=To, cu_draft=sub.cu, has_bonus=True,
                               **opd_kw)
        compare_opd(loss[rows], g[rows], oref, label=label)
    assert np.all(acc >= 0)
    return acc, nxt, loss, g


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_ragged_sampling(T):
    b = synth.config(5, N=9, lengths=np.array([2, 4, 8, 16, 1, 3, 16, 7, 5], np.int32), V=40000, seed=81)
    if float(T) not in b.tokens:
        b.tokens[float(T)] = synth.sample_tokens(b.draft, T, 81)
    _check(b, T, T, label=f"fused T={T}")


@pytest.mark.parametrize("To", [1.0, 0.7])
def test_greedy_with_loss_at_its_own_temperature(To):
    b = synth.config(5, N=6, lengths=np.array([3, 16, 1, 8, 5, 2], np.int32), V=32768, seed=82)
    _check(b, 0.0, To, label=f"fused greedy, loss T={To}")


def test_fp32_rows():
    b = synth.make_batch("f32", seed=83, lengths=np.array([4, 1, 9, 16], np.int32), V=4096, dtype="f32",
                         sigma_pos=synth.sigma_ramp, temperatures=(1.0,))
    _check(b, 1.0, 1.0, label="fused f32")


def test_clipped_rows_are_exact():
    b = synth.config(5, N=6, lengths=np.array([5, 8, 2, 16, 3, 7], np.int32), V=16384, seed=84)
    _check(b, 1.0, 1.0, label="fused c=0.02", clip_c=0.02)


def test_matches_separate_opd_bitwise():
    """The loss pass is the same kernel as opd_loss's: identical results."""
    import serving_vocab_wide_gb300 as svw
    b = synth.config(5, N=12, V=40000, seed=85)
    acc, nxt, loss, g = _fused(b, 1.0, 1.0)
    l2, g2 = svw.opd_loss(to_torch_logits(b.target), to_torch_logits(b.draft), temperature=1.0,
                          cu_draft=to_torch_i32(b.cu), has_bonus=True, **OPD)
    assert np.array_equal(loss, l2.cpu().numpy()) and np.array_equal(g, g2.cpu().numpy())


def test_bad_requests():
    import torch
    import serving_vocab_wide_gb300 as svw
    b = synth.config(5, N=6, lengths=np.array([3, 4, 2, 5, 6, 2], np.int32), V=8192, seed=86)
    t = b.target.copy()
    d = b.draft.copy()
    t[b.cu[1] + 1 + 2, 7] = 0x7FC0           # NaN in request 1's target row 2
    d[b.cu[3] + 0, 100] = 0x7F80             # +Inf in request 3's draft row 0
    t[b.cu[4] + 4 + b.lengths[4], :] = 0xFF80  # request 4's bonus row all -inf
    tok = b.tokens[1.0].copy()
    tok[b.cu[5]] = b.V + 3                   # request 5: token out of range
    bb = synth.Batch(**{**b.__dict__, "target": t, "draft": d})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt, loss, g = _fused(bb, 1.0, 1.0, status=status, tokens=tok)
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT
    assert list(acc[[1, 3, 4, 5]]) == [-1] * 4 and list(nxt[[1, 3, 4, 5]]) == [-1] * 4
    ok = [0, 2]
    sub = b.subset(ok)
    vref = oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[1.0], 1.0, b.seed,
                              req_ids=np.asarray(ok, np.int32))
    compare_verify(acc[ok], nxt[ok], vref, "fused good requests")


def test_inconsistent_csr_rejects_all():
    import torch
    import serving_vocab_wide_gb300 as svw
    b = synth.config(5, N=4, lengths=np.array([3, 4, 2, 5], np.int32), V=4096, seed=87)
    cu = b.cu.copy()
    cu[2], cu[3] = cu[3], cu[2]  # not monotone
    bb = synth.Batch(**{**b.__dict__, "cu": cu})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, nxt, _, _ = _fused(bb, 1.0, 1.0, status=status)
    assert np.all(acc == -1) and np.all(nxt == -1)
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT


@pytest.fixture(scope="module")
def mix_batch():
    return synth.config(5)


@pytest.mark.parametrize("V", [106504, 163840])
def test_wide_clusters(V):
    """Wide rows (up to the one-pass path's widest), several rows and bonus
    rows per cluster."""
    b = synth.config(5, N=20, V=V, seed=V)
    _check(b, 1.0, 1.0, label=f"fused V={V} T=1")
    _check(b, 0.0, 1.0, label=f"fused V={V} T=0")


def test_workspace_contents_do_not_matter(mix_batch):
    """Every workspace word the finalize reads is written by the same call:
    a workspace filled with 0xff bytes (NaN row constants, set flags) before
    each call gives the same results as a zeroed one, call after call."""
    import torch
    import serving_vocab_wide_gb300 as svw
    b = mix_batch
    N, R, V = b.N, b.total_rows, b.target.shape[1]
    t, d = to_torch_logits(b.target), to_torch_logits(b.draft)
    cu, tok = to_torch_i32(b.cu), to_torch_i32(b.tokens[1.0])
    ws = torch.zeros(svw.verify_opd_workspace_size(N, R, V, svw.SVW_BF16), dtype=torch.uint8, device="cuda")
    outs = []
    for rep in range(4):
        if rep:
            ws.fill_(255)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        acc, nxt, loss, _ = svw.spec_verify_opd(t, d, cu, tok, 1.0, b.seed, opd_temperature=1.0, max_len=32,
                                                total_draft_rows=R, status=st, workspace=ws, **OPD)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append((acc.cpu().numpy(), nxt.cpu().numpy(), loss.cpu().numpy()))
    for o in outs[1:]:
        for x, y in zip(outs[0], o):
            assert np.array_equal(x, y)
    assert np.all(outs[0][0] >= 0)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_mix_full_size_all_requests(T, mix_batch):
    """Every request and every loss / gradient row of the benchmark's batch,
    the oracle's requests split over the host's cores; near-tie excusals
    counted and bounded."""
    b = mix_batch
    acc, nxt, loss, g = _fused(b, T, 1.0)
    vref = oracle_verify_all(b, T, alt_next=nxt)
    nf, nfm = compare_verify(acc, nxt, vref, f"fused mix N=256 T={T}")
    check_near_ties(vref, nfm, f"fused mix N=256 T={T}")
    assert np.all(acc >= 0)
    skipped = compare_opd_all(b, loss, g, label=f"fused mix N=256 T={T}", temperature=1.0, **OPD)
    print(f"fused mix T={T}: {skipped} of {b.total_rows} loss rows near the clip bound")
    assert skipped <= 0.01 * b.total_rows


@pytest.mark.parametrize("sigma", [0.05, 0.02])
@pytest.mark.parametrize("lam", [0.1, 0.0])
def test_near_copy_drafts(sigma, lam):
    """Drafts almost equal to their targets (z = y + N(0, sigma^2) at every
    position), V = 151936: the loss within 1e-4 relative with no absolute
    allowance, the verification bit-exact outside flagged near-ties."""
    b = synth.make_batch("nearcopy", seed=int(1000 * sigma) + int(10 * lam) + 91,
                         lengths=np.array([16, 3, 8, 1, 12, 5], np.int32), V=151936, draft_kind="add",
                         sigma_req=[sigma] * 6, temperatures=(1.0,))
    acc, nxt, loss, g = _fused(b, 1.0, 1.0, lambda_ce=lam)
    vref = oracle.spec_verify(b.target, b.draft, b.cu, b.tokens[1.0], 1.0, b.seed)
    compare_verify(acc, nxt, vref, f"near copy sigma={sigma}")
    oref = oracle.opd_loss(b.target, b.draft, temperature=1.0, cu_draft=b.cu, has_bonus=True, clip_c=1.0,
                           lambda_ce=lam)
    lrel, grel = opd_errors(loss, g, oref)
    print(f"fused near copy sigma={sigma} lambda={lam}: max rel loss err {lrel.max():.3g}, "
          f"max rel grad err {grel.max():.3g}, mean accepted {acc.mean():.2f}")
    compare_opd(loss, g, oref, atol=0.0, label=f"fused near copy sigma={sigma} lambda={lam}")


def test_deterministic_rerun(mix_batch):
    r1 = _fused(mix_batch, 1.0, 1.0)
    r2 = _fused(mix_batch, 1.0, 1.0)
    for x, y in zip(r1, r2):
        assert np.array_equal(x, y)


def test_kernel_timer_hook():
    """svw_time_next_launch records the caller's events around one kernel."""
    import torch
    import serving_vocab_wide_gb300 as svw
    b = synth.config(5, N=8, V=32768, seed=88)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    svw.time_next_launch("opd_fast_kernel", e0, e1)
    _fused(b, 1.0, 1.0)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0.0
    # one-shot: a second call leaves the events alone
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    f1.record()
    torch.cuda.synchronize()
    _fused(b, 1.0, 1.0)
    torch.cuda.synchronize()
    assert f0.elapsed_time(f1) >= 0.0
