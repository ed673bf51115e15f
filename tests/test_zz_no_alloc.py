"""The allocation-free verification entry point (spec_verify_noalloc).

It serves callers that cannot allocate device memory, by running the regular
verification kernels on a fixed scratch area the library keeps on each GPU.
Its results must equal those of spec_verify with a caller workspace.  The file
is named so that pytest collects it last; it passes on its own in a fresh
process as well as after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import to_torch_i32, to_torch_logits

pytestmark = pytest.mark.gpu


def _both(b, T):
    import torch
    import serving_vocab_wide_gb300 as svw
    t, d = to_torch_logits(b.target), to_torch_logits(b.draft)
    cu, tok = to_torch_i32(b.cu), to_torch_i32(b.tokens[float(T)])
    acc, nxt = svw.spec_verify(t, d, cu, tok, T, b.seed, total_draft_rows=b.total_rows)
    # the new entry point, called directly through the C ABI
    L = svw.lib()
    acc2 = torch.full((b.N,), -7, dtype=torch.int32, device="cuda")
    nxt2 = torch.full((b.N,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    rc = L.spec_verify_noalloc(P(t.data_ptr()), P(d.data_ptr()), svw._dtype_code(t), b.V, b.N,
                               P(cu.data_ptr()), b.total_rows, 32, P(tok.data_ptr()), float(T),
                               b.seed, P(acc2.data_ptr()), P(nxt2.data_ptr()),
                               P(status.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.svw_status_string(rc)
    return (acc.cpu().numpy(), nxt.cpu().numpy(), acc2.cpu().numpy(), nxt2.cpu().numpy(),
            int(status.item()))


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    import torch
    torch.cuda.set_device(0)
    b1 = synth.config(3, N=24, seed=31)
    b2 = synth.config(5, N=12, seed=32)
    b2.tokens[1.0] = synth.sample_tokens(b2.draft, 1.0, 32)
    for b, T in ((b1, 1.0), (b2, 0.0), (b2, 1.0)):
        acc, nxt, acc2, nxt2, st = _both(b, T)
        # same kernels on the same inputs: identical outputs, bit for bit
        assert np.array_equal(acc, acc2) and np.array_equal(nxt, nxt2), (T, acc, acc2)
        assert st == 0 and np.all(acc >= 0)


def test_noalloc_rejects_batches_beyond_its_scratch():
    import torch
    import serving_vocab_wide_gb300 as svw
    L = svw.lib()
    N, R, V = 4096, 65536, 151936
    assert svw.verify_workspace_size(N, R, V, svw.SVW_BF16) > (32 << 20)
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p(dummy.data_ptr())
    rc = L.spec_verify_noalloc(P, P, svw.SVW_BF16, V, N, P, R, 16, P, 1.0, 0, P, P, None, None)
    assert rc == 2  # SVW_ERR_UNSUPPORTED, nothing launched
