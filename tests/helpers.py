"""Shared test helpers: moving synthetic batches to the GPU and comparing the
CUDA path with the oracle."""
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


def compare_verify(acc, nxt, ref, label=""):
    """Bit-exact outside the oracle's flagged near-tie requests.
    Returns (n_flagged, n_flagged_mismatch)."""
    flags = ref["flags"]
    near = (flags & NEAR) != 0
    mism = (acc != ref["accept_len"]) | (nxt != ref["next_token"])
    bad_unflagged = np.nonzero(mism & ~near)[0]
    assert bad_unflagged.size == 0, (
        f"{label}: {bad_unflagged.size} unflagged mismatches, first requests "
        f"{bad_unflagged[:5]}: gpu acc {acc[bad_unflagged[:5]]} nxt {nxt[bad_unflagged[:5]]} "
        f"oracle acc {ref['accept_len'][bad_unflagged[:5]]} nxt {ref['next_token'][bad_unflagged[:5]]}")
    return int(near.sum()), int((mism & near).sum())


def compare_opd(loss, grad, ref, rtol=1e-4, label=""):
    """loss within rtol relative; each dlogits row within rtol * max|row|.
    Rows the oracle flags as near a clip boundary are skipped and counted."""
    skip = (ref["flags"] & oracle.FLAG_NEAR_CLIP) != 0
    ok = ~skip
    ol = ref["loss"]
    err = np.abs(loss.astype(np.float64) - ol)
    tol = rtol * np.abs(ol) + 1e-6
    assert np.all(err[ok] <= tol[ok]), f"{label}: loss err {err[ok].max()} (tol {tol[ok][np.argmax(err[ok])]})"
    if grad is not None and ref["dlogits"] is not None:
        og = ref["dlogits"]
        gerr = np.abs(grad.astype(np.float64) - og).max(axis=1)
        gscale = np.abs(og).max(axis=1)
        assert np.all(gerr[ok] <= rtol * gscale[ok] + 1e-12), \
            f"{label}: dlogits err {gerr[ok].max()} vs scale {gscale[ok].min()}"
    return int(skip.sum())
