"""Shared test helpers: moving synthetic batches to the GPU and comparing the
CUDA path with the oracle (on whole batches, with the oracle's requests
split over the host's cores)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle

NEAR = oracle.FLAG_NEAR_ACCEPT | oracle.FLAG_NEAR_CDF | oracle.FLAG_DEGENERATE


def to_torch_logits(arr, device="cuda"):
    import torch
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_torch_i32(arr, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).to(device)


def gpu_verify(b, T, seed=None, max_len=32, status=None):
    import serving_vocab_wide_gb300 as svw
    t = to_torch_logits(b.target)
    d = to_torch_logits(b.draft)
    cu = to_torch_i32(b.cu)
    tok = to_torch_i32(b.tokens[float(T)])
    acc, nxt = svw.spec_verify(t, d, cu, tok, T, b.seed if seed is None else seed,
                               max_len=max_len, total_draft_rows=b.total_rows, status=status)
    return acc.cpu().numpy(), nxt.cpu().numpy()


BAND = 1e-5  # the oracle's near-tie band (accept threshold; CDF boundary, as a fraction of Z)


def compare_verify(acc, nxt, ref, label=""):
    """Bit-exact outside the oracle's flagged near-tie requests, and every
    excused mismatch checked: a different accepted length needs a flagged
    accept test; a different token after the same accepted length needs a
    flagged CDF boundary and, when the oracle was given the GPU's tokens
    (ref["alt_dist"]), the GPU's token must lie within the band of the
    oracle's draw point w Z.  Returns (n_flagged, n_flagged_mismatch)."""
    flags = ref["flags"]
    near = (flags & NEAR) != 0
    mism = (acc != ref["accept_len"]) | (nxt != ref["next_token"])
    bad_unflagged = np.nonzero(mism & ~near)[0]
    assert bad_unflagged.size == 0, (
        f"{label}: {bad_unflagged.size} unflagged mismatches, first requests "
        f"{bad_unflagged[:5]}: gpu acc {acc[bad_unflagged[:5]]} nxt {nxt[bad_unflagged[:5]]} "
        f"oracle acc {ref['accept_len'][bad_unflagged[:5]]} nxt {ref['next_token'][bad_unflagged[:5]]}")
    acc_diff = np.nonzero(mism & (acc != ref["accept_len"]))[0]
    assert np.all(flags[acc_diff] & oracle.FLAG_NEAR_ACCEPT), (
        f"{label}: requests {acc_diff} differ in accepted length without a flagged accept test")
    tok_diff = np.nonzero(mism & (acc == ref["accept_len"]))[0]
    assert np.all(flags[tok_diff] & (oracle.FLAG_NEAR_CDF | oracle.FLAG_DEGENERATE)), (
        f"{label}: requests {tok_diff} differ in the drawn token without a flagged CDF boundary")
    if "alt_dist" in ref and tok_diff.size:
        dist = ref["alt_dist"][tok_diff]
        degen = (flags[tok_diff] & oracle.FLAG_DEGENERATE) != 0
        assert np.all((dist <= BAND) | degen), (
            f"{label}: GPU tokens of requests {tok_diff} lie {dist} (fraction of Z) from the oracle's draw")
    return int(near.sum()), int((mism & near).sum())


def near_tie_counts(flags):
    """Requests flagged near an accept threshold and near a CDF boundary."""
    return (int(((flags & oracle.FLAG_NEAR_ACCEPT) != 0).sum()),
            int(((flags & oracle.FLAG_NEAR_CDF) != 0).sum()))


def opd_errors(loss, grad, ref):
    """Per row: relative loss error and the dlogits error as a fraction of the
    row's largest |gradient| (NaN where the oracle has no value)."""
    ol = ref["loss"]
    lrel = np.abs(loss.astype(np.float64) - ol) / np.abs(ol)
    grel = None
    if grad is not None and ref["dlogits"] is not None:
        og = ref["dlogits"]
        grel = np.abs(grad.astype(np.float64) - og).max(axis=1) / np.abs(og).max(axis=1)
    return lrel, grel


def compare_opd(loss, grad, ref, rtol=1e-4, atol=1e-6, label=""):
    """loss within rtol relative (plus atol absolute); each dlogits row within
    rtol * max|row|.  Rows the oracle flags as near a clip boundary are
    skipped and counted."""
    skip = (ref["flags"] & oracle.FLAG_NEAR_CLIP) != 0
    ok = ~skip
    ol = ref["loss"]
    err = np.abs(loss.astype(np.float64) - ol)
    tol = rtol * np.abs(ol) + atol
    assert np.all(err[ok] <= tol[ok]), f"{label}: loss err {err[ok].max()} (tol {tol[ok][np.argmax(err[ok])]})"
    if grad is not None and ref["dlogits"] is not None:
        og = ref["dlogits"]
        gerr = np.abs(grad.astype(np.float64) - og).max(axis=1)
        gscale = np.abs(og).max(axis=1)
        assert np.all(gerr[ok] <= rtol * gscale[ok] + 1e-12), \
            f"{label}: dlogits err {gerr[ok].max()} vs scale {gscale[ok].min()}"
    return int(skip.sum())


# ---------------------------------------------------------------------------
# the oracle on whole batches: requests are independent, so contiguous groups
# of them run on separate threads (the oracle's C calls release the GIL)
# ---------------------------------------------------------------------------
def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _groups(N, n):
    bounds = np.linspace(0, N, min(N, n) + 1).astype(int)
    return [(int(a), int(e)) for a, e in zip(bounds[:-1], bounds[1:]) if e > a]


def _req_rows(b, a, e):
    """Requests [a, e) of batch b as views: target rows, draft rows, their
    CSR offsets, and the draft-row range."""
    d0, d1 = int(b.cu[a]), int(b.cu[e])
    t0, t1 = (d0 + a, d1 + e) if b.has_bonus else (d0, d1)
    cu = (b.cu[a:e + 1] - b.cu[a]).astype(np.int32)
    return b.target[t0:t1], b.draft[d0:d1], cu, d0, d1


def oracle_verify_all(b, T, tokens=None, alt_next=None):
    """oracle.spec_verify over every request of b (Philox request ids kept);
    with alt_next (another implementation's tokens) also "alt_dist"."""
    tok = b.tokens[float(T)] if tokens is None else tokens
    out = dict(accept_len=np.zeros(b.N, np.int32), next_token=np.zeros(b.N, np.int32),
               flags=np.zeros(b.N, np.int32))
    if alt_next is not None:
        out["alt_dist"] = np.zeros(b.N, np.float64)

    def work(g):
        a, e = g
        t, d, cu, d0, d1 = _req_rows(b, a, e)
        r = oracle.spec_verify(t, d, cu, tok[d0:d1], T, b.seed, req_ids=np.arange(a, e, dtype=np.int32),
                               alt_next=None if alt_next is None else alt_next[a:e])
        for k in out:
            out[k][a:e] = r[k]

    nt = host_threads()
    with ThreadPoolExecutor(nt) as pool:
        list(pool.map(work, _groups(b.N, 4 * nt)))
    return out


def compare_opd_all(b, loss, grad, rtol=1e-4, atol=1e-6, label="", **opd_kw):
    """compare_opd on every row of b, the oracle's rows computed group by group
    on host threads (so its fp64 gradients never all exist at once).
    Returns the number of rows skipped as near a clip boundary."""
    def work(g):
        a, e = g
        t, d, cu, d0, d1 = _req_rows(b, a, e)
        ref = oracle.opd_loss(t, d, cu_draft=cu if b.has_bonus else None, has_bonus=b.has_bonus,
                              want_grad=grad is not None, **opd_kw)
        return compare_opd(loss[d0:d1], None if grad is None else grad[d0:d1], ref, rtol=rtol, atol=atol,
                           label=f"{label} requests {a}..{e - 1}")

    nt = host_threads()
    with ThreadPoolExecutor(nt) as pool:
        return sum(pool.map(work, _groups(b.N, 4 * nt)))


def check_near_ties(ref, n_flagged_mismatch, label, max_share=0.01):
    """The oracle's near-tie excusals on a whole batch: flagged requests
    counted by kind and reported; the excusals actually used (flagged and
    differing; each one checked by compare_verify) bounded."""
    n = ref["flags"].shape[0]
    na, nc = near_tie_counts(ref["flags"])
    bound = int(np.ceil(max_share * n))
    print(f"{label}: of {n} requests {na} flagged near an accept threshold, {nc} near a CDF boundary "
          f"(band {BAND:g}); {n_flagged_mismatch} of them differ (bound {bound})")
    assert na <= bound, f"{label}: {na} of {n} requests flagged near an accept threshold"
    assert n_flagged_mismatch <= bound, f"{label}: {n_flagged_mismatch} excused mismatches"
