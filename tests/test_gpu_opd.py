"""GPU parity: opd_loss (CUDA, through the C ABI) against the oracle.

Per-position loss within 1e-4 relative; every dlogits row within 1e-4 of the
row's largest |gradient|.  Rows the oracle flags as having a term within
1e-5 of the clip boundary are skipped and counted.

Both device paths are covered: with a workspace (one-exchange fast pass, then
the exact kernel on rows where a term reaches the clip or the draft has
masked entries) and without one (the exact kernel on every row).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare_opd, compare_opd_all, opd_errors, to_torch_i32, to_torch_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()


def _gpu(tgt, drf, cu=None, has_bonus=False, status=None, want_grad=True, **kw):
    import serving_vocab_wide_gb300 as svw
    loss, g = svw.opd_loss(to_torch_logits(tgt), to_torch_logits(drf),
                           cu_draft=None if cu is None else to_torch_i32(cu),
                           has_bonus=has_bonus, status=status, want_grad=want_grad, **kw)
    return loss.cpu().numpy(), (None if g is None else g.cpu().numpy())


PATHS = pytest.mark.parametrize("exact_only", [False, True], ids=["fast", "exact"])


@PATHS
@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (1024, "bf16"), (5003, "bf16"),
                                     (1001, "f32"), (4096, "f32"), (8, "bf16"), (151936, "f32"),
                                     (2048, "bf16"), (129024, "bf16"), (24, "f32"),
                                     # a 256K vocabulary: wider than the one-pass path, so the
                                     # exact kernel takes every row on both parametrisations
                                     (262144, "bf16")])
def test_paired_rows(V, dtype, exact_only):
    rows = 6
    b = synth.make_batch("opd", seed=V + 1, lengths=np.full(1, rows, np.int32), V=V,
                         dtype=dtype, draft_kind="scaled", temperatures=(), has_bonus=False)
    loss, g = _gpu(b.target, b.draft, exact_only=exact_only)
    ref = oracle.opd_loss(b.target, b.draft)
    compare_opd(loss, g, ref, label=f"V={V} {dtype}")


@pytest.mark.parametrize("V", [40000, 106504, 163840])
def test_many_rows_per_cluster(V):
    """Clusters that each walk several rows (and bonus rows) of the verify
    layout, up to the widest row of the one-pass path (163840 bf16 entries:
    8 CTAs of 2560 16-byte vectors)."""
    b = synth.make_batch("opd", seed=V + 3, lengths=np.full(20, 8, np.int32), V=V, dtype="bf16",
                         draft_kind="scaled", temperatures=(), has_bonus=True)
    loss, g = _gpu(b.target, b.draft, cu=b.cu, has_bonus=True)
    ref = oracle.opd_loss(b.target, b.draft, cu_draft=b.cu, has_bonus=True)
    compare_opd(loss, g, ref, label=f"many rows V={V}")


@PATHS
@pytest.mark.parametrize("T,c,lam,gs", [(1.0, 0.01, 0.1, 1.0), (0.7, 1e30, 0.5, 0.0625),
                                        (1.3, 0.2, 0.0, 1.0), (1.0, float("inf"), 4.0, 0.2)])
def test_parameters(T, c, lam, gs, exact_only):
    b = synth.make_batch("opd", seed=11, lengths=np.full(1, 5, np.int32), V=32768,
                         draft_kind="scaled", temperatures=(), has_bonus=False)
    loss, g = _gpu(b.target, b.draft, temperature=T, clip_c=c, lambda_ce=lam, grad_scale=gs,
                   exact_only=exact_only)
    ref = oracle.opd_loss(b.target, b.draft, temperature=T, clip_c=c, lambda_ce=lam,
                          grad_scale=gs)
    compare_opd(loss, g, ref, label=f"T={T} c={c}")


def _row_max_term(y, z):
    """max_v |q_v (lq_v - lp_v)| per row in fp64 (only to choose a clip bound
    that splits the rows; the parity check itself is against the oracle)."""
    y = synth.as_f32(y).astype(np.float64)
    z = synth.as_f32(z).astype(np.float64)
    lp = y - y.max(1, keepdims=True)
    lp -= np.log(np.exp(lp).sum(1, keepdims=True))
    lq = z - z.max(1, keepdims=True)
    lq -= np.log(np.exp(lq).sum(1, keepdims=True))
    return np.abs(np.exp(lq) * (lq - lp)).max(1)


def test_fix_up_over_several_flag_batches():
    """More rows than one batch of the fix-up's flag scan (4096 rows), with a
    clip bound between the rows' largest terms: the flagged rows of every
    batch are redone exactly and the others keep the one-pass result."""
    b = synth.make_batch("opd", seed=37, lengths=np.full(1, 9000, np.int32), V=1024,
                         draft_kind="scaled", temperatures=(), has_bonus=False)
    mt = _row_max_term(b.target, b.draft)
    c = float(np.median(mt))
    assert (mt > c).sum() > 4096
    loss, g = _gpu(b.target, b.draft, clip_c=c)
    ref = oracle.opd_loss(b.target, b.draft, clip_c=c)
    compare_opd(loss, g, ref, label=f"9000 rows c={c}")


@PATHS
def test_mixed_clipped_and_unclipped_rows(exact_only):
    """About half the rows have a term beyond the clip: the fast pass must hand
    exactly those to the exact kernel and keep the others."""
    b = synth.make_batch("opd", seed=31, lengths=np.full(1, 40, np.int32), V=16384,
                         draft_kind="add", temperatures=(), has_bonus=False,
                         sigma_pos=lambda j: 0.1 + 0.1 * j)
    mt = _row_max_term(b.target, b.draft)
    c = float(np.median(mt))
    assert 8 <= int((mt > c).sum()) <= 32
    loss, g = _gpu(b.target, b.draft, clip_c=c, exact_only=exact_only)
    ref = oracle.opd_loss(b.target, b.draft, clip_c=c)
    compare_opd(loss, g, ref, label=f"c={c}")


@PATHS
def test_masked_entries(exact_only):
    """-inf draft entries (q = 0) and -inf target entries under q > 0 (an
    infinite term, clamped) in otherwise ordinary rows."""
    b = synth.make_batch("opd", seed=32, lengths=np.full(1, 6, np.int32), V=8192,
                         draft_kind="scaled", temperatures=(), has_bonus=False)
    t = b.target.copy()
    d = b.draft.copy()
    d[1, ::7] = 0xFF80                # masked draft entries
    t[2, 100:200] = 0xFF80            # masked target entries
    d[3, ::5] = 0xFF80
    t[3, 1::5] = 0xFF80               # both
    loss, g = _gpu(t, d, clip_c=1.0, exact_only=exact_only)
    ref = oracle.opd_loss(t, d, clip_c=1.0)
    assert np.all(np.isfinite(loss))
    compare_opd(loss, g, ref, label="masked")


def test_loss_only():
    b = synth.make_batch("opd", seed=12, lengths=np.full(1, 4, np.int32), V=20000,
                         draft_kind="scaled", temperatures=(), has_bonus=False)
    loss, g = _gpu(b.target, b.draft, want_grad=False)
    assert g is None
    compare_opd(loss, None, oracle.opd_loss(b.target, b.draft, want_grad=False))


@PATHS
def test_verify_layout_rows(exact_only):
    b = synth.config(5, N=7, V=40000, seed=21)
    loss, g = _gpu(b.target, b.draft, cu=b.cu, has_bonus=True, exact_only=exact_only)
    ref = oracle.opd_loss(b.target, b.draft, cu_draft=b.cu, has_bonus=True)
    compare_opd(loss, g, ref, label="verify layout")


@PATHS
def test_bad_rows(exact_only):
    import torch
    import serving_vocab_wide_gb300 as svw
    b = synth.make_batch("opd", seed=13, lengths=np.full(1, 4, np.int32), V=4096,
                         draft_kind="scaled", temperatures=(), has_bonus=False)
    t = b.target.copy()
    d = b.draft.copy()
    t[1, 5] = 0x7FC0          # NaN
    d[2, :] = 0xFF80          # all -inf
    t[3, 100] = 0x7F80        # +inf
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss, g = _gpu(t, d, status=status, exact_only=exact_only)
    ref = oracle.opd_loss(t, d)
    assert np.isfinite(loss[0]) and np.all(np.isnan(loss[1:]))
    assert np.all(ref["flags"][1:] & oracle.FLAG_BAD)
    assert np.all(np.isnan(g[1:]))
    assert int(status.item()) & svw.SVW_DEV_BAD_INPUT
    compare_opd(loss[:1], g[:1], {k: v[:1] for k, v in ref.items()})


def test_full_size_all_rows():
    """Every row of the 64 x 16-row OPD workload against the oracle."""
    b = synth.config(4)
    loss, g = _gpu(b.target, b.draft, temperature=1.0, clip_c=1.0, lambda_ce=0.1)
    skipped = compare_opd_all(b, loss, g, label="opd 1024 rows", temperature=1.0, clip_c=1.0, lambda_ce=0.1)
    assert skipped <= 0.01 * b.total_rows
    # every row's gradient sums to ~0
    assert np.all(np.abs(g.sum(axis=1)) < 1e-4 * np.abs(g).max(axis=1) + 1e-6)
    assert np.all(np.isfinite(loss))


def test_deterministic_rerun():
    b = synth.config(4, N=3)
    l1, g1 = _gpu(b.target, b.draft)
    l2, g2 = _gpu(b.target, b.draft)
    assert np.array_equal(l1, l2) and np.array_equal(g1, g2)


def test_fast_and_exact_paths_agree_full_size():
    """Every row of the full-size OPD batch: the two device paths agree to
    float rounding (each is checked against the oracle elsewhere)."""
    b = synth.config(4)
    lf, gf = _gpu(b.target, b.draft)
    le, ge = _gpu(b.target, b.draft, exact_only=True)
    assert np.all(np.abs(lf - le) <= 1e-4 * np.abs(le) + 1e-6)
    scale = np.abs(ge).max(axis=1)
    assert np.all(np.abs(gf - ge).max(axis=1) <= 1e-4 * scale + 1e-12)


@PATHS
@pytest.mark.parametrize("sigma", [0.1, 0.05, 0.02])
@pytest.mark.parametrize("lam", [0.1, 0.0])
def test_near_copy_drafts_full_vocabulary(sigma, lam, exact_only):
    """Drafts that nearly equal their targets (z = y + N(0, sigma^2)), the
    regime on-policy distillation converges to: KL ~ sigma^2 / 2, so with
    lambda = 0 the loss is ~1e-3 .. 2e-4 and log q - log p ~ sigma.  Loss
    within 1e-4 relative with no absolute allowance, every gradient row
    within 1e-4 of its largest entry, at V = 151936."""
    R = 24
    b = synth.make_batch("opd", seed=int(1000 * sigma) + int(10 * lam) + 51, lengths=np.full(1, R, np.int32),
                         V=151936, draft_kind="add", sigma_req=[sigma], temperatures=(), has_bonus=False)
    loss, g = _gpu(b.target, b.draft, clip_c=1.0, lambda_ce=lam, exact_only=exact_only)
    ref = oracle.opd_loss(b.target, b.draft, clip_c=1.0, lambda_ce=lam)
    lrel, grel = opd_errors(loss, g, ref)
    print(f"sigma={sigma} lambda={lam} {'exact' if exact_only else 'fast'}: loss {ref['loss'].min():.3g}.."
          f"{ref['loss'].max():.3g}, max rel loss err {lrel.max():.3g}, max rel grad err {grel.max():.3g}")
    compare_opd(loss, g, ref, atol=0.0, label=f"near copy sigma={sigma} lambda={lam}")
